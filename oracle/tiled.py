"""The pages' block-tiled online-softmax forward, in fp64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This mirror is used to
pin the naive oracle: the pages claim the tiled loop reaches exactly the plain
result, for every block size ("vectorized-flash-attention-kernel",
Evidence & signatures: "Block size invariance (sizes 2,3,5,8,16,32)" and the
edge-case list "All block sizes from 2 to 64").  It is never compared with the
GPU path directly.

The loop follows "vectorized-flash-attention-kernel", Core algorithm:
for each batch and head, for each query block, start every row at
(m, l, acc) = (-inf, 0, 0); for each key/value block form the block's scores,
mask them, and apply the online-softmax update

    m_new = max(m_old, max_j S[i,j])
    corr  = exp(m_old - m_new)
    l     = corr * l_old   + sum_j exp(S[i,j] - m_new)
    acc   = corr * acc_old + sum_j exp(S[i,j] - m_new) V[j,:]

then normalise acc / l.  Key/value blocks that lie wholly in the future of
the query block are skipped (Key design decisions 3); padding is masked per
element only, so a block can hide every key of a row.  Rows whose running max
is still -inf take no update, and rows that end with l == 0 emit exact zeros
("js-flash-attention-tiled-online-softmax-exactness", Root causes 2).

The merge of two partial states follows "FlashAttention" (F08, Math & data
structures): partial softmax states form a monoid with identity
(-inf, 0, 0), combined by rescaling both to the larger running max.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass
class SoftmaxState:
    """Partial online-softmax state of a set of rows: running max m (scaled
    logits), running sum l and un-normalised numerator acc [rows, D]."""
    m: np.ndarray
    l: np.ndarray
    acc: np.ndarray

    @staticmethod
    def identity(rows: int, D: int) -> "SoftmaxState":
        return SoftmaxState(np.full(rows, -np.inf), np.zeros(rows), np.zeros((rows, D)))


def _exp_shift(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """exp(x - ref) with the convention that an empty side (x = -inf) weighs 0,
    also when ref is -inf (so -inf - -inf never produces NaN)."""
    out = np.zeros(np.broadcast(x, ref).shape)
    ok = np.broadcast_to(x > -np.inf, out.shape)
    xb = np.broadcast_to(x, out.shape)
    rb = np.broadcast_to(ref, out.shape)
    out[ok] = np.exp(xb[ok] - rb[ok])
    return out


def online_update(state: SoftmaxState, S: np.ndarray, Vb: np.ndarray) -> SoftmaxState:
    """One key/value block of the online-softmax recurrence.

    S: masked scaled scores [rows, cols] (masked entries are -inf),
    Vb: the block's values [cols, D].
    """
    m_blk = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    m_new = np.maximum(state.m, m_blk)
    alive = m_new > -np.inf                    # rows with at least one key so far
    corr = np.ones_like(m_new)
    corr[alive] = _exp_shift(state.m[alive], m_new[alive])
    p = np.zeros_like(S)
    p[alive] = _exp_shift(S[alive], m_new[alive][:, None])
    l = corr * state.l + p.sum(axis=1)
    acc = corr[:, None] * state.acc + p @ Vb
    return SoftmaxState(m_new, l, acc)


def merge(a: SoftmaxState, b: SoftmaxState) -> SoftmaxState:
    """Associative merge of two partial states over disjoint key sets."""
    m = np.maximum(a.m, b.m)
    fa = _exp_shift(a.m, m)
    fb = _exp_shift(b.m, m)
    return SoftmaxState(m, fa * a.l + fb * b.l, fa[:, None] * a.acc + fb[:, None] * b.acc)


def finalize(state: SoftmaxState):
    """O = acc / l (exact zeros where l == 0); LSE = m + ln l (-inf there)."""
    o = np.zeros_like(state.acc)
    lse = np.full(state.m.shape, -np.inf)
    nz = ~(state.l == 0)
    o[nz] = state.acc[nz] / state.l[nz][:, None]
    lse[nz] = state.m[nz] + np.log(state.l[nz])
    return o, lse


def partial_state(q_rows, K, V, key_idx, scale, allowed=None) -> SoftmaxState:
    """State of query rows q_rows [R, D] over the keys key_idx only.

    allowed: optional boolean [R, len(key_idx)] mask (False = masked).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    key_idx = np.asarray(key_idx, dtype=np.int64)
    Kb = np.asarray(K, dtype=np.float64)[key_idx]
    Vb = np.asarray(V, dtype=np.float64)[key_idx]
    S = scale * (q_rows @ Kb.T)
    if allowed is not None:
        S = np.where(allowed, S, -np.inf)
    return online_update(SoftmaxState.identity(q_rows.shape[0], q_rows.shape[1]), S, Vb)


def block_mask(rows, cols, L, causal):
    """True where key `cols[c]` is hidden from query `rows[r]`: keys at or past
    the key length L (padding), and, when causal, keys after the query
    ("kvRow > qRow -> -inf", Core algorithm step 2)."""
    masked = np.broadcast_to(cols[None, :] >= L, (rows.shape[0], cols.shape[0]))
    if causal:
        masked = masked | (cols[None, :] > rows[:, None])
    return masked


def forward(q, k, v, causal=True, scale=None, kv_len=None, block=64, block_kv=None,
            tracker=None):
    """Tiled forward over [B,H,N,D] inputs; returns (O, LSE) in fp64.

    block: query block size; block_kv: key/value block size (defaults to
    block, as in the pages' single blockSize option).  tracker, if given, is a
    callable that receives the element count of every working array the loop
    allocates (the pages' allocation tracker).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    bq = int(block)
    bk = int(block_kv if block_kv is not None else block)
    if bq <= 0 or bk <= 0:
        raise ValueError("block sizes must be positive")
    o = np.zeros((B, H, N, D))
    lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        L = N if kv_len is None else min(max(int(kv_len[b]), 0), N)
        for h in range(H):
            for q_start in range(0, N, bq):
                q_end = min(q_start + bq, N)           # rows q_start .. q_end-1
                rows = np.arange(q_start, q_end)
                st = SoftmaxState.identity(q_end - q_start, D)
                for kv_start in range(0, N, bk):
                    kv_end = min(kv_start + bk, N)
                    if causal and kv_start > q_end - 1:
                        break                           # block wholly in the future
                    cols = np.arange(kv_start, kv_end)
                    S = scale * (q[b, h, q_start:q_end] @ k[b, h, kv_start:kv_end].T)
                    if tracker is not None:
                        tracker(S.size)
                    S = np.where(block_mask(rows, cols, L, causal), -np.inf, S)
                    st = online_update(st, S, v[b, h, kv_start:kv_end])
                ob, lb = finalize(st)
                o[b, h, q_start:q_end] = ob
                lse[b, h, q_start:q_end] = lb
    return o, lse
