"""Parity of the bf16 backward (fa_bwd) with the fp64 backward oracle.

Tolerance (bf16 inputs and outputs, fp32 accumulation; derived in the
design notes): for each of dQ, dK, dV, the largest error is at most 2e-2 of
the tensor's largest reference entry and the mean error at most 1e-2 of its
mean reference magnitude.  P and dS are rounded to bf16 for the tensor-core
products (relative 2^-9 each), O is the forward's bf16 output, and the
gradients are rounded once more to bf16 on output.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_23_gb300 as fa
import oracle
import workloads

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    fa.build()
    fa.load()
    oracle.library()


def run_case(B, H, N, D, causal, kv_len, seed, dtype="bf16"):
    inp = workloads.make_case(B, H, N, D, dtype=dtype, causal=causal, seed=seed, kv_len=kv_len)
    g = torch.Generator("cpu").manual_seed(seed + 77)
    do = torch.randn((B, H, N, D), generator=g).to(inp.q.dtype)
    q, k, v, dog = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), do.cuda()
    kv = inp.kv_len.cuda() if inp.kv_len is not None else None
    o, lse = fa.forward(q, k, v, causal=causal, kv_len=kv)
    dq, dk, dv = fa.backward(q, k, v, o, dog, lse, causal=causal, kv_len=kv)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == fa.FA_OK
    ref = oracle.attention_bwd(inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(),
                               do.float().numpy(), causal=causal,
                               kv_len=None if inp.kv_len is None else inp.kv_len.numpy())
    stats = {}
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        gn = got.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gn)), name
        err = np.abs(gn - r)
        scale_max = np.abs(r).max()
        scale_mean = np.abs(r).mean()
        stats[name] = (err.max() / max(scale_max, 1e-30), err.mean() / max(scale_mean, 1e-30))
        if scale_max == 0:
            assert np.all(gn == 0), name
            continue
        assert err.max() <= MAX_REL * scale_max, (name, stats[name])
        assert err.mean() <= MEAN_REL * scale_mean, (name, stats[name])
    if inp.kv_len is not None:
        for bi in range(B):
            L = int(inp.kv_len[bi])
            assert bool((dk[bi, :, L:] == 0).all()) and bool((dv[bi, :, L:] == 0).all())
    return stats


CASES = [
    # B, H, N, D, causal, kv_len
    (1, 1, 128, 64, True, None),
    (1, 2, 256, 128, False, None),
    (2, 2, 300, 64, True, [300, 0]),
    # head dims below 128 run zero-padded to 64 / 128
    (1, 2, 200, 32, True, None),
    (2, 1, 300, 96, False, [300, 77]),
    (1, 1, 257, 40, True, None),
    (1, 1, 130, 8, False, None),
    (1, 2, 640, 128, True, [500]),
    (2, 1, 777, 128, False, [777, 129]),
    (1, 2, 1024, 64, True, None),
]


@pytest.mark.parametrize("B,H,N,D,causal,kv_len", CASES)
def test_bwd_matches_oracle(B, H, N, D, causal, kv_len):
    stats = run_case(B, H, N, D, causal, kv_len, seed=N + D)
    print(stats)


@pytest.mark.parametrize("D", [40, 96])
def test_bwd_head_dim_writes_stay_in_bounds(D):
    """dQ, dK and dV go to views of larger buffers: nothing past the last
    row's D columns changes (the zero-padded columns are never stored)."""
    B, H, N = 1, 2, 300
    inp = workloads.make_case(B, H, N, D, dtype="bf16", causal=True, seed=D + 5)
    g = torch.Generator("cpu").manual_seed(D)
    do = torch.randn((B, H, N, D), generator=g).to(torch.bfloat16).cuda()
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    o, lse = fa.forward(q, k, v, causal=True)
    n = B * H * N * D
    bufs = [torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                   bufs[0].data_ptr(), bufs[1].data_ptr(), bufs[2].data_ptr(), B, H, N, D, True,
                   float("nan"), None, ws.data_ptr(), ws_bytes, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == fa.FA_OK
    for buf in bufs:
        assert torch.all(buf[n:] == 7.0)
    # the same gradients as the allocating entry point
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(bufs[1][:n].view(B, H, N, D), dk)
    assert torch.equal(bufs[2][:n].view(B, H, N, D), dv)
    assert (bufs[0][:n].view(B, H, N, D).float() - dq.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()


F16_CASES = [
    (1, 2, 256, 128, True, None),
    (2, 1, 300, 64, False, [300, 77]),
    (1, 1, 257, 96, True, None),
]


@pytest.mark.parametrize("B,H,N,D,causal,kv_len", F16_CASES)
def test_bwd_f16_matches_oracle(B, H, N, D, causal, kv_len):
    """fp16 tensors through fa_bwd_f16 (P and dS rounded to fp16)."""
    stats = run_case(B, H, N, D, causal, kv_len, seed=N + D + 1, dtype="fp16")
    print(stats)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_autograd_attention(dtype):
    """fa.attention is differentiable: torch autograd through it gives the
    gradients of fa.backward."""
    inp = workloads.make_case(2, 2, 300, 64, dtype="bf16" if dtype == torch.bfloat16 else "fp16",
                              causal=True, seed=31, kv_len=[300, 150])
    kv = inp.kv_len.cuda()
    q, k, v = (x.cuda().requires_grad_(True) for x in (inp.q, inp.k, inp.v))
    g = torch.Generator("cpu").manual_seed(5)
    do = torch.randn(q.shape, generator=g).to(dtype).cuda()
    o = fa.attention(q, k, v, causal=True, kv_len=kv)
    (o.float() * do.float()).sum().backward()
    o2, lse = fa.forward(q.detach(), k.detach(), v.detach(), causal=True, kv_len=kv)
    dq, dk, dv = fa.backward(q.detach(), k.detach(), v.detach(), o2, do, lse, causal=True, kv_len=kv)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o2)
    assert torch.equal(k.grad, dk) and torch.equal(v.grad, dv)
    assert (q.grad.float() - dq.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()
