"""The allocation-free split-KV entry point, checked against fa_fwd.

fa_fwd_splitkv_noalloc serves callers that cannot allocate device memory.
It uses a fixed scratch array owned by the library instead of a caller
workspace.  These tests call it through the C ABI, on inputs and outputs
that the test allocates, and compare its results with fa_fwd on the same
inputs within the bf16 tolerances used by the parity tests.  They make two
calls in a row, a larger problem and then a smaller one, so that the second
call runs over scratch that still holds the first call's data.

This file is named to be collected last.
"""
import pytest
import torch

import exact_tiled_attention_23_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    fa.build()
    fa.load()


def _inputs(B, H, N, D, causal, seed, kv_len=None):
    inp = workloads.make_case(B, H, N, D, dtype="bf16", causal=causal, seed=seed, kv_len=kv_len)
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    kv = inp.kv_len.cuda() if inp.kv_len is not None else None
    return q, k, v, kv


def _noalloc(q, k, v, kv, causal, splits):
    B, H, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, H, N, D, causal, float("nan"),
                                   kv.data_ptr() if kv is not None else None, splits,
                                   torch.cuda.current_stream().cuda_stream)
    return st, o, lse


def _check_against_fa_fwd(q, k, v, kv, causal, o, lse):
    ref_o, ref_lse = fa.forward(q, k, v, causal=causal, kv_len=kv)
    torch.cuda.synchronize()
    err = (o.float() - ref_o.float()).abs()
    assert err.max().item() <= BF16_MAX
    assert err.mean().item() <= BF16_MEAN
    assert torch.equal(torch.isneginf(lse), torch.isneginf(ref_lse))
    fin = torch.isfinite(ref_lse)
    if fin.any():
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= 1e-3


def test_two_calls_in_a_row_match_fa_fwd():
    # call 1: D=128, causal, key padding with an empty batch, 3 key ranges
    q, k, v, kv = _inputs(2, 4, 1024, 128, True, seed=71, kv_len=[1024, 0])
    st, o, lse = _noalloc(q, k, v, kv, True, 3)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == fa.FA_OK
    _check_against_fa_fwd(q, k, v, kv, True, o, lse)

    # call 2: smaller, D=64, non-causal, ragged N, automatic split count; the
    # scratch still holds call 1's partials
    q, k, v, kv = _inputs(1, 3, 777, 64, False, seed=72)
    st, o, lse = _noalloc(q, k, v, kv, False, 0)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == fa.FA_OK
    _check_against_fa_fwd(q, k, v, kv, False, o, lse)


def test_too_large_a_problem_is_rejected_before_launch():
    B, H, N, D, splits = 8, 16, 8192, 128, 4
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, N, D, splits) > fa.FA_NOALLOC_SCRATCH_BYTES
    p = 1 << 16
    st = fa.fa_fwd_splitkv_noalloc(p, p, p, p, None, B, H, N, D, True, float("nan"), None, splits, None)
    assert st == fa.FA_ERR_UNSUPPORTED
