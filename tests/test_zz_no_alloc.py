"""The allocation-free split-KV entry point, checked against the oracle.

fa_fwd_splitkv_noalloc serves callers that cannot allocate device memory:
code inside a framework's allocation-free region, a real-time loop where an
allocation could block, or a plugin that is handed only its input and output
buffers.  It
uses a fixed scratch array owned by the library instead of a caller
workspace.  These tests call it through the C ABI, on inputs and outputs
that the test allocates, and compare its results with the fp64 CPU oracle
on every element, within the bf16 tolerances of the parity tests
(max |dO| <= 2e-2, mean |dO| <= 2e-3, LSE within 1e-3 + 1e-5*|LSE|, rows
that see no key exact +0.0 with LSE = -inf).  They make two calls in a row,
a larger problem and then a smaller one, so that the second call runs over
scratch that still holds the first call's data, and check that the second
call leaves the device's free memory unchanged.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_23_gb300 as fa
import oracle
import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    fa.build()
    fa.load()
    oracle.library()


def _inputs(B, H, N, D, causal, seed, kv_len=None):
    inp = workloads.make_case(B, H, N, D, dtype="bf16", causal=causal, seed=seed, kv_len=kv_len)
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    kv = inp.kv_len.cuda() if inp.kv_len is not None else None
    return inp, (q, k, v, kv)


def _outputs(q):
    B, H, N, D = q.shape
    return torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=q.device)


def _noalloc(q, k, v, kv, causal, splits, o, lse):
    B, H, N, D = q.shape
    return fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     B, H, N, D, causal, float("nan"),
                                     kv.data_ptr() if kv is not None else None, splits,
                                     torch.cuda.current_stream().cuda_stream)


def _check_against_oracle(inp, o, lse):
    w = inp.workload
    B, H, N, D = w.B, w.H, w.N, w.D
    kv = None if inp.kv_len is None else inp.kv_len.numpy()
    o_ref, lse_ref = oracle.attention(inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(),
                                      causal=inp.causal, scale=w.scale, kv_len=kv)
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(og))
    dead = np.isneginf(lse_ref)
    assert np.all(og[dead] == 0.0) and not np.any(np.signbit(og[dead]))
    assert np.all(np.isneginf(lg[dead]))
    live = ~dead
    err = np.abs(og[live] - o_ref[live])
    assert err.max(initial=0) <= BF16_MAX
    assert (err.mean() if err.size else 0.0) <= BF16_MEAN
    lerr = np.abs(lg[live] - lse_ref[live])
    assert np.all(lerr <= 1e-3 + 1e-5 * np.abs(lse_ref[live]))


def test_two_calls_in_a_row_match_the_oracle():
    # call 1: D=128, causal, key padding with an empty batch, 3 key ranges
    inp, (q, k, v, kv) = _inputs(2, 4, 1024, 128, True, seed=71, kv_len=[1024, 0])
    o, lse = _outputs(q)
    assert _noalloc(q, k, v, kv, True, 3, o, lse) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == fa.FA_OK
    _check_against_oracle(inp, o, lse)
    assert bool((o[1] == 0).all()) and bool(torch.isneginf(lse[1]).all())

    # call 2: smaller, D=64, non-causal, ragged N, automatic split count; the
    # scratch still holds call 1's partials.  Outputs are allocated first, so
    # any change of free memory comes from the call itself.
    inp, (q, k, v, kv) = _inputs(1, 3, 777, 64, False, seed=72)
    o, lse = _outputs(q)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _noalloc(q, k, v, kv, False, 0, o, lse) == fa.FA_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, "the call changed the device's free memory"
    assert fa.fa_device_status(None) == fa.FA_OK
    _check_against_oracle(inp, o, lse)


def test_too_large_a_problem_is_rejected_before_launch():
    B, H, N, D, splits = 8, 16, 8192, 128, 4
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, N, D, splits) > fa.FA_NOALLOC_SCRATCH_BYTES
    p = 1 << 16
    st = fa.fa_fwd_splitkv_noalloc(p, p, p, p, None, B, H, N, D, True, float("nan"), None, splits, None)
    assert st == fa.FA_ERR_UNSUPPORTED
