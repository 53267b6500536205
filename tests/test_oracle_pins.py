"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test names what fixes the expected value: a library routine that the
definition reduces to (torch softmax / scaled_dot_product_attention in fp64,
named by the "FlashAttention" module's sources), a closed form, an invariant
of softmax attention, a 40-digit brute force, or the pages' own tiled method
("vectorized-flash-attention-kernel", Core algorithm) run by the independent
fp64 mirror in ``oracle/tiled.py``.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import tiled

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def rand(B, H, N, D, seed, scale=1.0):
    r = np.random.default_rng(seed)
    q = (r.standard_normal((B, H, N, D)) * scale).astype(np.float32)
    k = (r.standard_normal((B, H, N, D)) * scale).astype(np.float32)
    v = r.standard_normal((B, H, N, D)).astype(np.float32)
    return q, k, v


def allowed_mask(B, N, causal, kv_len):
    """[B,1,N,N] bool: True where key j is visible to query i."""
    j = torch.arange(N)
    i = torch.arange(N)
    lens = [N] * B if kv_len is None else [min(max(int(x), 0), N) for x in kv_len]
    m = torch.stack([(j[None, :] < L).expand(N, N) for L in lens])[:, None]
    if causal:
        m = m & (j[None, :] <= i[:, None])[None, None]
    return m


def torch_reference(q, k, v, causal, scale, kv_len):
    """softmax(scale*Q K^T + mask) V and logsumexp in fp64 via torch (CPU)."""
    Q, K, V = (torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    B, H, N, D = Q.shape
    ok = allowed_mask(B, N, causal, kv_len)
    S = scale * (Q @ K.transpose(-1, -2))
    S = S.masked_fill(~ok, float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    O = torch.softmax(S, dim=-1) @ V
    return O.numpy(), lse.numpy(), ok.expand(B, H, N, N).any(-1).numpy()


def sdpa_reference(q, k, v, causal, scale, kv_len):
    Q, K, V = (torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    B, H, N, D = Q.shape
    ok = allowed_mask(B, N, causal, kv_len)
    return F.scaled_dot_product_attention(Q, K, V, attn_mask=ok, scale=scale).numpy()


CASES = [
    # B, H, N, D, causal, kv_len, seed
    (1, 1, 1, 8, True, None, 1),
    (1, 2, 7, 5, False, None, 2),
    (2, 3, 8, 16, True, None, 3),
    (2, 3, 8, 16, False, [8, 3], 4),
    (3, 2, 33, 12, True, [0, 17, 33], 5),
    (2, 1, 65, 64, False, [65, 1], 6),
    (1, 4, 130, 32, True, [99], 7),
]


@pytest.mark.parametrize("B,H,N,D,causal,kv_len,seed", CASES)
def test_matches_torch_softmax_fp64(oracle_lib, B, H, N, D, causal, kv_len, seed):
    q, k, v = rand(B, H, N, D, seed)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle_lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    ro, rlse, nonempty = torch_reference(q, k, v, causal, scale, kv_len)
    np.testing.assert_allclose(o[nonempty], ro[nonempty], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[nonempty], rlse[nonempty], rtol=1e-13, atol=1e-13)
    # fully masked rows: exact +0.0 and -inf (finite zeros, never NaN)
    assert np.all(o[~nonempty] == 0.0) and not np.any(np.signbit(o[~nonempty]))
    assert np.all(np.isneginf(lse[~nonempty]))


@pytest.mark.parametrize("B,H,N,D,causal,kv_len,seed", CASES)
def test_matches_sdpa_fp64(oracle_lib, B, H, N, D, causal, kv_len, seed):
    q, k, v = rand(B, H, N, D, seed + 100)
    scale = 0.37  # an explicit, non-default scale
    o, _ = oracle_lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    _, _, nonempty = torch_reference(q, k, v, causal, scale, kv_len)
    ref = sdpa_reference(q, k, v, causal, scale, kv_len)
    np.testing.assert_allclose(o[nonempty], ref[nonempty], rtol=0, atol=1e-12)


def _decimal_row(q, K, V, keys, scale):
    s = [Decimal(scale) * sum(Decimal(float(a)) * Decimal(float(b)) for a, b in zip(q, K[j])) for j in keys]
    m = max(s)
    w = [(x - m).exp() for x in s]
    l = sum(w)
    o = [sum(w[t] * Decimal(float(V[j][d])) for t, j in enumerate(keys)) / l for d in range(len(q))]
    return o, m + l.ln()


@pytest.mark.parametrize("B,H,N,D,causal,kv_len", [
    (2, 3, 8, 16, True, None),
    (2, 3, 8, 16, False, None),
    (1, 1, 1, 3, True, None),
    (1, 2, 2, 4, True, [2]),
    (2, 1, 3, 2, False, [3, 1]),
    (3, 1, 5, 3, True, [5, 0, 2]),
])
def test_decimal_brute_force(oracle_lib, B, H, N, D, causal, kv_len):
    """40-digit evaluation of the definition on tiny shapes, one row at a time."""
    getcontext().prec = 40
    q, k, v = rand(B, H, N, D, 11 + N + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle_lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    for b in range(B):
        L = N if kv_len is None else kv_len[b]
        for h in range(H):
            for i in range(N):
                keys = [j for j in range(min(L, N)) if (not causal or j <= i)]
                if not keys:
                    assert np.all(o[b, h, i] == 0) and np.isneginf(lse[b, h, i])
                    continue
                ro, rl = _decimal_row(q[b, h, i], k[b, h], v[b, h], keys, scale)
                np.testing.assert_allclose(o[b, h, i], [float(x) for x in ro], rtol=0, atol=1e-14)
                assert abs(lse[b, h, i] - float(rl)) <= 1e-14 * max(1.0, abs(float(rl)))


def test_hand_worked_two_keys(oracle_lib):
    """N=2, D=1 by hand: q=(1,2), k=(1,0), v=(1,3), scale 1.

    Row 0 (causal) sees key 0 only: O = 1, LSE = 1.
    Row 1 sees both: logits (2, 0), O = (e^2*1 + 3)/(e^2 + 1), LSE = ln(e^2 + 1).
    Non-causal row 0: logits (1, 0), O = (e + 3)/(e + 1), LSE = ln(e + 1).
    """
    q = np.array([1, 2], np.float32).reshape(1, 1, 2, 1)
    k = np.array([1, 0], np.float32).reshape(1, 1, 2, 1)
    v = np.array([1, 3], np.float32).reshape(1, 1, 2, 1)
    e = math.e
    o, lse = oracle_lib.attention(q, k, v, causal=True, scale=1.0)
    assert o[0, 0, 0, 0] == pytest.approx(1.0, abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(1.0, abs=1e-15)
    assert o[0, 0, 1, 0] == pytest.approx((e * e + 3) / (e * e + 1), abs=1e-15)
    assert lse[0, 0, 1] == pytest.approx(math.log(e * e + 1), abs=1e-15)
    o, lse = oracle_lib.attention(q, k, v, causal=False, scale=1.0)
    assert o[0, 0, 0, 0] == pytest.approx((e + 3) / (e + 1), abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(math.log(e + 1), abs=1e-15)


# ---------------------------------------------------------------- closed forms
def test_single_token_attends_to_itself(oracle_lib):
    """N=1: O = V[0] and LSE = scale * q.k ("vectorized-flash-attention-kernel",
    edge cases: N=1 attends only to itself)."""
    q, k, v = rand(2, 3, 1, 16, 21)
    for causal in (True, False):
        o, lse = oracle_lib.attention(q, k, v, causal=causal, scale=0.25)
        np.testing.assert_array_equal(o, v.astype(np.float64))
        ref = 0.25 * np.einsum("bhnd,bhnd->bhn", q.astype(np.float64), k.astype(np.float64))
        np.testing.assert_allclose(lse, ref, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal,kv_len", [(True, None), (False, None), (True, [5, 12]), (False, [9, 1])])
def test_all_zero_queries_give_uniform_weights(oracle_lib, causal, kv_len):
    """All-zero Q: every logit is 0, the weights are uniform over the visible
    keys: O_i = mean of those V rows, LSE_i = ln(count) (edge cases: all-zero
    tensors give a uniform distribution)."""
    B, H, N, D = 2, 2, 12, 8
    _, k, v = rand(B, H, N, D, 22)
    q = np.zeros_like(k)
    o, lse = oracle_lib.attention(q, k, v, causal=causal, kv_len=kv_len)
    for b in range(B):
        L = N if kv_len is None else kv_len[b]
        for i in range(N):
            keys = [j for j in range(L) if (not causal or j <= i)]
            np.testing.assert_allclose(o[b, :, i], v[b, :, keys].astype(np.float64).mean(axis=0)
                                       if len(keys) else 0.0, atol=1e-14)
            if keys:
                np.testing.assert_allclose(lse[b, :, i], math.log(len(keys)), atol=1e-14)


def test_identical_key_rows_give_uniform_weights(oracle_lib):
    """Identical K rows (edge cases: identical rows): every visible key has the
    same logit, so the weights are uniform."""
    B, H, N, D = 1, 2, 10, 6
    q, k, v = rand(B, H, N, D, 23)
    k[:] = k[:, :, :1, :]
    o, lse = oracle_lib.attention(q, k, v, causal=True, scale=0.5)
    for i in range(N):
        np.testing.assert_allclose(o[0, :, i], v[0, :, : i + 1].astype(np.float64).mean(axis=1), atol=1e-14)
        s = 0.5 * np.einsum("hd,hd->h", q[0, :, i].astype(np.float64), k[0, :, 0].astype(np.float64))
        np.testing.assert_allclose(lse[0, :, i], s + math.log(i + 1), atol=1e-13)


def test_constant_values_pass_through(oracle_lib):
    """V rows all equal to c: O is a convex combination of them, so O = c."""
    q, k, _ = rand(2, 2, 20, 8, 24, scale=3.0)
    c = np.linspace(-2, 2, 8).astype(np.float32)
    v = np.broadcast_to(c, q.shape).copy()
    o, _ = oracle_lib.attention(q, k, v, causal=True, kv_len=[20, 7])
    np.testing.assert_allclose(o, np.broadcast_to(c.astype(np.float64), o.shape), atol=1e-14)


def test_fully_masked_rows_are_finite_zeros(oracle_lib):
    """kv_len = 0 masks every key: O = +0.0 exactly and LSE = -inf
    ("js-flash-attention-tiled-online-softmax-exactness", Root causes 2 and
    Verification: fully masked rows give finite zeros, also from the
    reference)."""
    q, k, v = rand(3, 2, 9, 4, 25)
    o, lse = oracle_lib.attention(q, k, v, causal=False, kv_len=[0, 9, 0])
    for b in (0, 2):
        assert np.all(o[b] == 0.0) and not np.any(np.signbit(o[b]))
        assert np.all(np.isneginf(lse[b]))
    assert np.all(np.isfinite(o[1])) and np.all(np.isfinite(lse[1]))


def test_one_hot_limit(oracle_lib):
    """A scaled-logit gap of 100 puts all weight on one key (e^-100 is far
    below fp64 resolution): O = V[that key] and LSE = the top logit, with
    logits up to 100*N and no overflow (edge cases: very large logits)."""
    B, H, N, D = 1, 1, 16, 8
    q = np.zeros((B, H, N, D), np.float32)
    k = np.zeros_like(q)
    _, _, v = rand(B, H, N, D, 26)
    q[..., 0] = 100.0
    k[0, 0, :, 0] = np.arange(N, dtype=np.float32)  # logit of key j is 100*j
    o, lse = oracle_lib.attention(q, k, v, causal=True, scale=1.0)
    # causal row i sees keys 0..i; key i wins by a gap of 100
    np.testing.assert_allclose(o[0, 0], v[0, 0].astype(np.float64), rtol=0, atol=1e-30)
    np.testing.assert_allclose(lse[0, 0], 100.0 * np.arange(N), rtol=1e-15, atol=1e-12)


# ------------------------------------------------------------------ invariants
def test_joint_key_permutation_invariance(oracle_lib):
    """Non-causal, no padding: permuting K and V rows together leaves O and LSE
    unchanged (the softmax sum has no order)."""
    q, k, v = rand(2, 2, 24, 16, 27)
    perm = np.random.default_rng(0).permutation(24)
    o1, l1 = oracle_lib.attention(q, k, v, causal=False)
    o2, l2 = oracle_lib.attention(q, k[:, :, perm], v[:, :, perm], causal=False)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_logit_shift_invariance(oracle_lib):
    """Append a column c to Q and 1 to K: every logit of a row moves by scale*c.
    O is unchanged and LSE moves by scale*c."""
    B, H, N, D = 2, 2, 17, 7
    q, k, v = rand(B, H, N, D, 28)
    c = 40.0
    q2 = np.concatenate([q, np.full((B, H, N, 1), c, np.float32)], -1)
    k2 = np.concatenate([k, np.ones((B, H, N, 1), np.float32)], -1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1), np.float32)], -1)
    o1, l1 = oracle_lib.attention(q, k, v, causal=True, scale=0.3, kv_len=[17, 6])
    o2, l2 = oracle_lib.attention(q2, k2, v2, causal=True, scale=0.3, kv_len=[17, 6])
    np.testing.assert_allclose(o2[..., :D], o1, atol=1e-13)
    np.testing.assert_allclose(o2[..., D], 0.0, atol=0)
    np.testing.assert_allclose(l2, l1 + 0.3 * c, atol=1e-12)


def test_weights_sum_to_one(oracle_lib):
    q, k, _ = rand(2, 3, 31, 8, 29, scale=4.0)
    v = np.ones_like(q)
    o, _ = oracle_lib.attention(q, k, v, causal=True, kv_len=[31, 13])
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_large_values_stay_finite(oracle_lib, sign):
    """Values up to 100 (and large negative ones) with logits up to 100xD
    ("vectorized-flash-attention-kernel", numerical stability)."""
    fig = GOLDEN["large_logits"]
    B, H, N, D = 1, 2, 20, 16
    r = np.random.default_rng(30)
    q = (sign * r.uniform(0, fig["max_value"], (B, H, N, D))).astype(np.float32)
    k = r.uniform(0, fig["max_value"], (B, H, N, D)).astype(np.float32)
    v = r.standard_normal((B, H, N, D)).astype(np.float32)
    o, lse = oracle_lib.attention(q, k, v, causal=True, scale=1.0 / fig["max_value"])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    ro, rlse, _ = torch_reference(q, k, v, True, 1.0 / fig["max_value"], None)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=1e-14)


# ----------------------------------------------------- the pages' tiled method
@pytest.mark.parametrize("block", GOLDEN["block_sizes"]["value"])
@pytest.mark.parametrize("causal,kv_len", [(True, None), (False, None), (True, [70, 0]), (False, [33, 1])])
def test_tiled_mirror_equals_oracle_at_every_block_size(oracle_lib, block, causal, kv_len):
    """Block-size invariance: the tiled online-softmax loop at block sizes
    2..64 reaches the plain result ("vectorized-flash-attention-kernel",
    Evidence & signatures), within the pages' 1e-10."""
    tol = GOLDEN["small_exact_tolerance"]["value"]
    q, k, v = rand(2, 2, 70, 16, 31 + block)
    o, lse = oracle_lib.attention(q, k, v, causal=causal, kv_len=kv_len)
    mo, mlse = tiled.forward(q, k, v, causal=causal, kv_len=kv_len, block=block)
    np.testing.assert_allclose(mo, o, rtol=0, atol=tol)
    assert np.array_equal(np.isneginf(mlse), np.isneginf(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(mlse[fin], lse[fin], rtol=0, atol=tol)


def test_tiled_mirror_multihead_case(oracle_lib):
    fig = GOLDEN["multihead_case"]
    q, k, v = rand(fig["B"], fig["H"], fig["N"], fig["D"], 40)
    for causal in (True, False):
        o, lse = oracle_lib.attention(q, k, v, causal=causal)
        for block in (2, 3, 8):
            mo, mlse = tiled.forward(q, k, v, causal=causal, block=block)
            np.testing.assert_allclose(mo, o, rtol=0, atol=fig["tolerance"])
            np.testing.assert_allclose(mlse, lse, rtol=0, atol=fig["tolerance"])


def test_tiled_mirror_rectangular_blocks(oracle_lib):
    q, k, v = rand(1, 2, 50, 8, 41)
    o, lse = oracle_lib.attention(q, k, v, causal=True, kv_len=[45])
    for bq, bk in [(7, 3), (16, 5), (1, 64), (64, 1)]:
        mo, mlse = tiled.forward(q, k, v, causal=True, kv_len=[45], block=bq, block_kv=bk)
        np.testing.assert_allclose(mo, o, atol=1e-12)
        np.testing.assert_allclose(mlse, lse, atol=1e-12)


def test_exactness_with_span_of_a_million(oracle_lib):
    """Rows whose logits span >= 1e6: tiled vs plain relative error <= 1e-9
    ("js-flash-attention-tiled-online-softmax-exactness", problem statement)."""
    fig = GOLDEN["exactness_span"]
    B, H, N, D = 1, 2, 40, 8
    q, k, v = rand(B, H, N, D, 42)
    q[:, :, ::3] *= 1e5
    scale = 1.0
    S = scale * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    span = (S.max(-1) - S.min(-1)).max()
    assert span >= fig["min_span"]
    o, lse = oracle_lib.attention(q, k, v, causal=False, scale=scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for block in (3, 8, 16):
        mo, mlse = tiled.forward(q, k, v, causal=False, scale=scale, block=block)
        rel = np.abs(mo - o).max() / np.abs(o).max()
        assert rel <= fig["max_relative_error"]
        assert np.abs(mlse - lse).max() / np.abs(lse).max() <= fig["max_relative_error"]
    ro, rlse, _ = torch_reference(q, k, v, False, scale, None)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)


def test_tiled_scratch_independent_of_sequence_length():
    """The mirror's largest working array is one block of scores, whatever N
    ("js-flash-attention-tiled-online-softmax-exactness", Verification)."""
    fig = GOLDEN["scratch_independent_of_N"]
    peaks = []
    for N in (256, 2048):
        q, k, v = rand(1, 1, N, fig["d"], 43)
        peak = [0]
        tiled.forward(q, k, v, causal=True, block=fig["block"],
                      tracker=lambda n: peak.__setitem__(0, max(peak[0], n)))
        peaks.append(peak[0])
    assert peaks[0] == peaks[1] == fig["block"] ** 2


# --------------------------------------------------------------- merge monoid
def _row_states(q, K, V, keys_parts, scale):
    return [tiled.partial_state(q, K, V, part, scale) for part in keys_parts]


def test_merge_is_associative_and_matches_oracle(oracle_lib):
    """Partial states over disjoint key sets merge, in any grouping, to the
    plain result ("FlashAttention" module, Math: a monoid)."""
    rng = np.random.default_rng(44)
    q, k, v = rand(1, 1, 48, 16, 44)
    o, lse = oracle_lib.attention(q, k, v, causal=False)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    scale = 0.25
    for trial in range(6):
        nparts = 2 + trial % 3
        labels = rng.integers(0, nparts, 48)        # non-contiguous parts
        labels[:nparts] = np.arange(nparts)
        parts = [np.nonzero(labels == p)[0] for p in range(nparts)]
        st = _row_states(Q, K, V, parts, scale)
        left = st[0]
        for s in st[1:]:
            left = tiled.merge(left, s)                 # ((a.b).c).d
        right = st[-1]
        for s in reversed(st[:-1]):
            right = tiled.merge(s, right)               # a.(b.(c.d))
        for merged in (left, right):
            mo, mlse = tiled.finalize(merged)
            np.testing.assert_allclose(mo, o[0, 0], atol=1e-13)
            np.testing.assert_allclose(mlse, lse[0, 0], atol=1e-13)
        # commutativity
        mo, _ = tiled.finalize(tiled.merge(st[1], st[0]))
        mo2, _ = tiled.finalize(tiled.merge(st[0], st[1]))
        np.testing.assert_allclose(mo, mo2, atol=1e-14)


def test_merge_identity_and_empty_sides():
    rng = np.random.default_rng(45)
    q, k, v = rand(1, 1, 10, 4, 45)
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    st = tiled.partial_state(Q, K, V, np.arange(10), 0.5)
    ident = tiled.SoftmaxState.identity(10, 4)
    for merged in (tiled.merge(st, ident), tiled.merge(ident, st)):
        np.testing.assert_array_equal(merged.m, st.m)
        np.testing.assert_array_equal(merged.l, st.l)
        np.testing.assert_array_equal(merged.acc, st.acc)
    both_empty = tiled.merge(ident, ident)           # -inf - -inf must not give NaN
    assert np.all(np.isneginf(both_empty.m)) and np.all(both_empty.l == 0)
    o, lse = tiled.finalize(both_empty)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    # a side whose keys are all masked behaves as the identity
    masked = tiled.partial_state(Q, K, V, np.arange(5), 0.5, allowed=np.zeros((10, 5), bool))
    m2 = tiled.merge(masked, st)
    np.testing.assert_allclose(m2.acc, st.acc, atol=0)
    del rng


# ------------------------------------------------- the row-sampled oracle
# oracle_attention_rows computes chosen rows of the same definition, one flat
# row index r = (b*H + h)*N + i at a time.  It decodes (b, h, i) and picks the
# batch's key length on its own, so its pin checks exactly those steps: each
# chosen row against torch's fp64 softmax on the same (b, h, i) (a library
# routine, independent of the C code), and bit for bit against the same row
# of the all-rows oracle.  The shapes have B, H >= 3, N not a power of two and
# key lengths of 0, 1, N, a ragged value and values outside [0, N], so a row
# decoded to the wrong batch, head or position, or given another batch's key
# length, lands on different data.
ROWS_CASES = [
    # B, H, N, D, causal, kv_len, seed
    (3, 3, 37, 8, True, [0, 37, 20], 61),
    (4, 3, 45, 6, False, [1, 45, 0, 60], 62),
    (3, 2, 50, 5, True, [-3, 50, 17], 63),
    (3, 4, 29, 12, False, None, 64),
    (5, 3, 33, 16, True, [33, 1, 9, 0, 32], 65),
]


def boundary_rows(B, H, N):
    """Flat rows at the first and last position of every head, plus the rows
    next to each batch boundary."""
    rows = set()
    for b in range(B):
        for h in range(H):
            base = (b * H + h) * N
            rows.update({base, base + 1, base + N // 2, base + N - 2, base + N - 1})
    return sorted(r for r in rows if 0 <= r < B * H * N)


@pytest.mark.parametrize("B,H,N,D,causal,kv_len,seed", ROWS_CASES)
def test_attention_rows_match_torch_and_all_rows(oracle_lib, B, H, N, D, causal, kv_len, seed):
    q, k, v = rand(B, H, N, D, seed)
    scale = 1.0 / math.sqrt(D)
    rng = np.random.default_rng(seed)
    rows = np.array(boundary_rows(B, H, N) + rng.integers(0, B * H * N, 64).tolist(), dtype=np.int64)
    o_rows, lse_rows = oracle_lib.attention_rows(q, k, v, rows, causal=causal, scale=scale, kv_len=kv_len)
    assert o_rows.shape == (rows.size, D) and lse_rows.shape == (rows.size,)

    # independent: torch fp64 softmax at the (b, h, i) each row decodes to
    ro, rlse, nonempty = torch_reference(q, k, v, causal, scale, kv_len)
    b, h, i = rows // (H * N), (rows // N) % H, rows % N
    live = nonempty[b, h, i]
    np.testing.assert_allclose(o_rows[live], ro[b, h, i][live], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_rows[live], rlse[b, h, i][live], rtol=1e-13, atol=1e-13)
    assert np.all(o_rows[~live] == 0.0) and not np.any(np.signbit(o_rows[~live]))
    assert np.all(np.isneginf(lse_rows[~live]))

    # the same rows of the all-rows oracle, bit for bit
    o_all, lse_all = oracle_lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    np.testing.assert_array_equal(o_rows, o_all.reshape(-1, D)[rows])
    np.testing.assert_array_equal(lse_rows, lse_all.reshape(-1)[rows])


def test_attention_rows_every_row_in_order_and_shuffled(oracle_lib):
    """All rows requested, in order and shuffled with repeats: the result
    follows the request order exactly."""
    B, H, N, D = 3, 3, 19, 4
    q, k, v = rand(B, H, N, D, 66)
    kv = [19, 0, 7]
    o_all, lse_all = oracle_lib.attention(q, k, v, causal=True, kv_len=kv)
    rows = np.arange(B * H * N)
    o_rows, lse_rows = oracle_lib.attention_rows(q, k, v, rows, causal=True, kv_len=kv)
    np.testing.assert_array_equal(o_rows, o_all.reshape(-1, D))
    np.testing.assert_array_equal(lse_rows, lse_all.reshape(-1))
    perm = np.random.default_rng(1).permutation(np.concatenate([rows, rows[:10]]))
    o_p, lse_p = oracle_lib.attention_rows(q, k, v, perm, causal=True, kv_len=kv)
    np.testing.assert_array_equal(o_p, o_all.reshape(-1, D)[perm])
    np.testing.assert_array_equal(lse_p, lse_all.reshape(-1)[perm])


def test_attention_rows_rejects_out_of_range_rows(oracle_lib):
    q, k, v = rand(2, 2, 5, 4, 67)
    for bad in ([-1], [2 * 2 * 5]):
        with pytest.raises(RuntimeError):
            oracle_lib.attention_rows(q, k, v, bad, causal=True)
    o, lse = oracle_lib.attention_rows(q, k, v, [], causal=True)
    assert o.shape == (0, 4) and lse.shape == (0,)
