"""The seeded input recipe: determinism and the structure each workload promises."""
import torch

import workloads


def test_draws_are_deterministic():
    a = workloads.make_case(2, 3, 17, 8, dtype="bf16", seed=5, padded="uniform0")
    b = workloads.make_case(2, 3, 17, 8, dtype="bf16", seed=5, padded="uniform0")
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.kv_len, b.kv_len)):
        assert torch.equal(x, y)
    c = workloads.make_case(2, 3, 17, 8, dtype="bf16", seed=6, padded="uniform0")
    assert not torch.equal(a.q, c.q)


def test_bf16_rounding_is_exact_in_fp32():
    x = workloads.make_case(1, 2, 33, 16, dtype="bf16", seed=1)
    assert x.q.dtype == torch.bfloat16
    assert torch.equal(x.q.float().to(torch.bfloat16), x.q)


def test_padded_spiky_workload_structure():
    """5% of query rows x30 so raw logit rows span more than 1e3; key lengths
    uniform in [0, N] with batch 1 at 0."""
    x = workloads.make("bf16_b4h16n4096d128_causal_padded_spiky")
    w = x.workload
    assert x.kv_len.dtype == torch.int32 and x.kv_len.shape == (w.B,)
    assert int(x.kv_len[1]) == 0
    assert bool(((x.kv_len >= 0) & (x.kv_len <= w.N)).all())
    frac = x.spiky.float().mean().item()
    assert 0.04 < frac < 0.06
    # raw logit span of a few scaled rows against the first 1024 keys of their head
    idx = torch.nonzero(x.spiky[0, 0])[:8, 0]
    q = x.q[0, 0, idx].float()
    s = q @ x.k[0, 0, :1024].float().T
    assert float((s.max(1).values - s.min(1).values).max()) > 1e3


def test_ragged_workload_lengths():
    w = workloads.WORKLOADS["bf16_b8h16n8191d64_noncausal_padded"]
    assert w.N % 128 != 0
    x = workloads.make_case(8, 1, 64, 8, padded="uniform1", seed=3)
    assert bool(((x.kv_len >= 1) & (x.kv_len <= 64)).all())


def test_unmasked_pair_count():
    assert workloads.unmasked_pairs(4, True) == 10
    assert workloads.unmasked_pairs(4, False) == 16
    # causal, L=2 of N=4: rows 0,1 see 1,2 keys; rows 2,3 see 2 each
    assert workloads.unmasked_pairs(4, True, kv_len=[2]) == 1 + 2 + 2 + 2
    assert workloads.unmasked_pairs(4, False, kv_len=[0, 3], B=2, H=3) == 3 * (0 + 12)
    brute = 0
    N = 9
    for L in (0, 4, 9):
        for i in range(N):
            brute += sum(1 for j in range(N) if j < L and j <= i)
    assert workloads.unmasked_pairs(N, True, kv_len=[0, 4, 9], B=3) == brute
