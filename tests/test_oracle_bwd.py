"""Pins of the backward oracle (dQ, dK, dV of sum(O * dO)).

The backward is pinned to things other than itself: central finite
differences of the (separately pinned) forward oracle, torch autograd through
an fp64 softmax-attention, the identity rowsum(dP * P) = rowsum(dO * O) of the
"FlashAttention" module (Math), and planted mistakes.
"""
import math
import subprocess

import numpy as np
import pytest
import torch

import oracle

from test_oracle_pins import allowed_mask, rand


def _do(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def _torch_grads(q, k, v, do, causal, scale, kv_len):
    Q, K, V = (torch.from_numpy(np.asarray(x, np.float64)).requires_grad_(True) for x in (q, k, v))
    B, H, N, D = Q.shape
    ok = allowed_mask(B, N, causal, kv_len)
    S = (scale * Q @ K.transpose(-1, -2)).masked_fill(~ok, float("-inf"))
    P = torch.softmax(S, dim=-1)
    P = torch.nan_to_num(P, nan=0.0)          # fully masked rows: zero weights
    O = P @ V
    (O * torch.from_numpy(np.asarray(do, np.float64))).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


CASES = [
    (1, 1, 5, 4, True, None),
    (2, 2, 9, 6, False, [9, 4]),
    (1, 3, 17, 8, True, [12]),
    (2, 1, 33, 16, True, [0, 33]),
    (1, 2, 64, 32, False, None),
]


@pytest.mark.parametrize("B,H,N,D,causal,kv_len", CASES)
def test_matches_torch_autograd_fp64(oracle_lib, B, H, N, D, causal, kv_len):
    q, k, v = rand(B, H, N, D, 300 + N)
    do = _do(q.shape, 400 + N)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle_lib.attention_bwd(q, k, v, do, causal=causal, scale=scale, kv_len=kv_len)
    tq, tk, tv = _torch_grads(q, k, v, do, causal, scale, kv_len)
    np.testing.assert_allclose(dq, tq, atol=1e-12)
    np.testing.assert_allclose(dk, tk, atol=1e-12)
    np.testing.assert_allclose(dv, tv, atol=1e-12)


@pytest.mark.parametrize("causal,kv_len", [(True, None), (False, [4])])
def test_matches_central_finite_differences(oracle_lib, causal, kv_len):
    """d/dx sum(O * dO) by (f(x+h) - f(x-h)) / 2h on the forward oracle.

    The perturbed inputs are fp32 arrays, so h is a power of two and every
    perturbed value stays exactly representable."""
    B, H, N, D = 1, 1, 5, 3
    q, k, v = rand(B, H, N, D, 51)
    do = _do(q.shape, 52)
    scale = 0.7
    grads = oracle_lib.attention_bwd(q, k, v, do, causal=causal, scale=scale, kv_len=kv_len)
    h = 2.0 ** -10

    def f(qq, kk, vv):
        o, _ = oracle_lib.attention(qq, kk, vv, causal=causal, scale=scale, kv_len=kv_len)
        return float((o * do.astype(np.float64)).sum())

    for which, g in zip(range(3), grads):
        for idx in np.ndindex(q.shape):
            xs = [q.copy(), k.copy(), v.copy()]
            xs[which][idx] += h
            fp = f(*xs)
            xs[which][idx] -= 2 * h
            fm = f(*xs)
            fd = (fp - fm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (which, idx, fd, g[idx])


def test_delta_identity(oracle_lib):
    """The identity rowsum(dP * P) = rowsum(dO * O) = Delta makes every row
    of dS = P * (dP - Delta) sum to zero, so sum_j dK_j = scale * sum_i
    (sum_j dS_ij) q_i = 0; and since rows of P sum to one, sum_j dV_j =
    sum_i dO_i."""
    B, H, N, D = 1, 2, 20, 8
    q, k, v = rand(B, H, N, D, 61)
    do = _do(q.shape, 62)
    scale = 0.35
    dq, dk, dv = oracle_lib.attention_bwd(q, k, v, do, causal=True, scale=scale)
    # rows of P sum to 1, so sum_j dV_j = sum_i dO_i (every row has a key here)
    np.testing.assert_allclose(dv.sum(axis=2), do.astype(np.float64).sum(axis=2), atol=1e-12)
    # sum_j dS_ij = 0  =>  sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


def test_fully_masked_rows_have_no_gradient(oracle_lib):
    q, k, v = rand(2, 1, 6, 4, 71)
    do = _do(q.shape, 72)
    dq, dk, dv = oracle_lib.attention_bwd(q, k, v, do, causal=False, kv_len=[0, 6])
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)
    assert np.any(dq[1] != 0)


BWD_MUTANTS = {
    "Delta dropped": ("dp[j] = p[j] * (s - delta);", "dp[j] = p[j] * s;"),
    "dV from dS": ("dvj[d] += p[j] * (double)g[d];", "dvj[d] += dp[j] * (double)g[d];"),
    "dQ scale dropped": ("dqi[d] += scale * dp[j] * (double)k[d];", "dqi[d] += dp[j] * (double)k[d];"),
    "dK uses K": ("dkj[d] += scale * dp[j] * (double)q[d];", "dkj[d] += scale * dp[j] * (double)k[d];"),
    "P not normalised": ("for (int64_t j = 0; j < n_vis; ++j) p[j] /= l;", ""),
    "causal diagonal dropped": ("if (causal && i + 1 < n_vis) n_vis = i + 1;", "if (causal && i < n_vis) n_vis = i;"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_mutant_is_caught(tmp_path, name):
    old, new = BWD_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1
    (tmp_path / "m.c").write_text(src.replace(old, new))
    out = str(tmp_path / "libm.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", str(tmp_path / "m.c"),
                    "-o", out, "-lm"], check=True, capture_output=True)
    lib = oracle.OracleLibrary(out)
    q, k, v = rand(1, 2, 9, 5, 81)
    do = _do(q.shape, 82)
    scale = 1.0 / math.sqrt(5)
    got = lib.attention_bwd(q, k, v, do, causal=True, scale=scale, kv_len=None)
    ref = _torch_grads(q, k, v, do, True, scale, None)
    assert not all(np.allclose(a, b, atol=1e-10) for a, b in zip(got, ref)), f"mutant {name!r} survived"
