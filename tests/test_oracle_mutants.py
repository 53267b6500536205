"""Planted mistakes: the pins must catch every plausible slip in the oracle.

The "FlashAttention" module's break-it exercise asks which tests miss one-line
bugs in an online-softmax kernel; the bugs themselves are not on the pages, so
the ones below are chosen here.  Each mutant is planted on the CPU only: the C
oracle's source is copied, one line is changed textually, the copy is built
into a temporary directory, and a compact battery of the pins in
``test_oracle_pins.py`` (library special cases and closed forms) must fail on
it.  The tiled mirror's update step gets the same treatment.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import tiled

from test_oracle_pins import ROWS_CASES, boundary_rows, rand, torch_reference

C_MUTANTS = {
    "causal mask drops the diagonal": (
        "if (causal && i + 1 < nkeys) nkeys = i + 1;", "if (causal && i < nkeys) nkeys = i;"),
    "scale not applied": ("s[j] = scale * dot;", "s[j] = dot;"),
    "V used in place of K": ("const float *k = k0 + j * D;", "const float *k = v0 + j * D;"),
    "LSE drops the max": ("*lse = m + log(l);", "*lse = log(l);"),
    "exp of the wrong sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "no normalisation": ("for (int64_t d = 0; d < D; ++d) o[d] /= l;", ""),
    "head offset ignored for K": ("const float *k0 = K + head * N * D;", "const float *k0 = K;"),
    "padding ignored": ("int64_t nkeys = L;", "int64_t nkeys = N;"),
    "reversed feature index": ("dot += (double)q[d] * (double)k[d];",
                               "dot += (double)q[d] * (double)k[D - 1 - d];"),
    "wrong V column": ("o[d] += s[j] * (double)v[d];", "o[d] += s[j] * (double)v[0];"),
    "fully masked rows not zeroed": ("o[d] = 0.0;\n        *lse = -INFINITY;",
                                     "o[d] = 0.0 / 0.0;\n        *lse = -INFINITY;"),
}


def battery(lib) -> bool:
    """True when the library passes every pin of the compact battery."""
    try:
        for (B, H, N, D, causal, kv_len, seed) in [
            (2, 3, 9, 5, True, [9, 4], 1),
            (2, 2, 12, 6, False, [12, 0], 2),
            (1, 2, 1, 4, True, None, 3),
        ]:
            q, k, v = rand(B, H, N, D, 500 + seed)
            scale = 1.0 / math.sqrt(D)
            o, lse = lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
            ro, rlse, nonempty = torch_reference(q, k, v, causal, scale, kv_len)
            if not np.allclose(o[nonempty], ro[nonempty], rtol=0, atol=1e-12):
                return False
            if not np.allclose(lse[nonempty], rlse[nonempty], rtol=0, atol=1e-12):
                return False
            if not (np.all(o[~nonempty] == 0.0) and np.all(np.isneginf(lse[~nonempty]))):
                return False
        return True
    except Exception:
        return False


def test_battery_passes_on_the_real_oracle(oracle_lib):
    assert battery(oracle_lib)


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_mutant_is_caught(tmp_path, name):
    old, new = C_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    out = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", str(mutated),
                    "-o", out, "-lm"], check=True, capture_output=True)
    assert not battery(oracle.OracleLibrary(out)), f"mutant {name!r} survived the pins"


# ---- the row-sampled entry point's index decoding ------------------------------
# oracle_attention_rows shares the per-row step with oracle_attention but turns
# a flat row index into (batch, head, position) and picks the batch's key
# length by itself.  Each slip below is planted in that decoding only (the
# text matched includes names found only there), so the all-rows oracle stays
# correct and only the rows pins can catch it.  Every planted index stays
# inside the arrays for the shapes of ROWS_CASES (B*H <= N, H <= B where a
# key length is read).
_ROWS_SITE = ("int64_t flat = rows[r];\n"
              "            int64_t i = flat % N;\n"
              "            int64_t head = flat / N;\n"
              "            int64_t b = head / H;\n"
              "            oracle_row(Q, K, V, N, D, head, i, key_length(kv_len, b, N),\n"
              "                       causal, scale, s, O_rows + r * D, LSE_rows + r);")


def _rows_mutant(old, new):
    assert old in _ROWS_SITE
    return _ROWS_SITE, _ROWS_SITE.replace(old, new)


ROWS_MUTANTS = {
    "rows: position from division": _rows_mutant("int64_t i = flat % N;", "int64_t i = flat / N;"),
    "rows: head drops the batch offset": _rows_mutant("int64_t head = flat / N;",
                                                      "int64_t head = flat / N % H;"),
    "rows: batch from head modulo H": _rows_mutant("int64_t b = head / H;", "int64_t b = head % H;"),
    "rows: key length of batch 0": _rows_mutant("key_length(kv_len, b, N)", "key_length(kv_len, 0, N)"),
    "rows: key length indexed by head": _rows_mutant("key_length(kv_len, b, N)",
                                                     "key_length(kv_len, head % B, N)"),
    "rows: outputs in reversed slots": _rows_mutant("O_rows + r * D", "O_rows + (nrows - 1 - r) * D"),
}


def rows_battery(lib) -> bool:
    """True when the row-sampled entry point passes its pins: every chosen
    row equal to torch's fp64 softmax at the decoded (b, h, i) and, bit for
    bit, to the all-rows oracle."""
    try:
        for (B, H, N, D, causal, kv_len, seed) in ROWS_CASES:
            q, k, v = rand(B, H, N, D, seed)
            scale = 1.0 / math.sqrt(D)
            rows = np.array(boundary_rows(B, H, N), dtype=np.int64)
            o_rows, lse_rows = lib.attention_rows(q, k, v, rows, causal=causal, scale=scale, kv_len=kv_len)
            ro, rlse, nonempty = torch_reference(q, k, v, causal, scale, kv_len)
            b, h, i = rows // (H * N), (rows // N) % H, rows % N
            live = nonempty[b, h, i]
            if not np.allclose(o_rows[live], ro[b, h, i][live], rtol=0, atol=1e-12):
                return False
            if not np.allclose(lse_rows[live], rlse[b, h, i][live], rtol=0, atol=1e-12):
                return False
            if not (np.all(o_rows[~live] == 0.0) and np.all(np.isneginf(lse_rows[~live]))):
                return False
            o_all, lse_all = lib.attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
            if not (np.array_equal(o_rows, o_all.reshape(-1, D)[rows]) and
                    np.array_equal(lse_rows, lse_all.reshape(-1)[rows])):
                return False
        return True
    except Exception:
        return False


def test_rows_battery_passes_on_the_real_oracle(oracle_lib):
    assert rows_battery(oracle_lib)


@pytest.mark.parametrize("name", sorted(ROWS_MUTANTS))
def test_rows_mutant_is_caught(tmp_path, name):
    old, new = ROWS_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    out = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", str(mutated),
                    "-o", out, "-lm"], check=True, capture_output=True)
    lib = oracle.OracleLibrary(out)
    assert battery(lib), f"mutant {name!r} also broke the all-rows oracle"
    assert not rows_battery(lib), f"mutant {name!r} survived the rows pins"


# ---- the tiled mirror's update step --------------------------------------------
_real_update = tiled.online_update


def _no_l_rescale(state, S, Vb):
    st = _real_update(state, S, Vb)
    p_sum = st.l - _corr(state, st) * state.l
    return tiled.SoftmaxState(st.m, state.l + p_sum, st.acc)


def _no_acc_rescale(state, S, Vb):
    st = _real_update(state, S, Vb)
    pv = st.acc - _corr(state, st)[:, None] * state.acc
    return tiled.SoftmaxState(st.m, st.l, state.acc + pv)


def _inverted_correction(state, S, Vb):
    st = _real_update(state, S, Vb)
    c = _corr(state, st)
    inv = np.where(c > 0, 1.0 / np.where(c > 0, c, 1.0), 0.0)
    pv = st.acc - c[:, None] * state.acc
    ps = st.l - c * state.l
    return tiled.SoftmaxState(st.m, inv * state.l + ps, inv[:, None] * state.acc + pv)


def _unguarded(state, S, Vb):
    with np.errstate(invalid="ignore"):
        m_new = np.maximum(state.m, S.max(axis=1))
        corr = np.exp(state.m - m_new)
        p = np.exp(S - m_new[:, None])
    return tiled.SoftmaxState(m_new, corr * state.l + p.sum(1), corr[:, None] * state.acc + p @ Vb)


def _corr(old, new):
    c = np.zeros_like(new.m)
    ok = old.m > -np.inf
    c[ok] = np.exp(old.m[ok] - new.m[ok])
    return c


def _mask_ge(rows, cols, L, causal):
    masked = np.broadcast_to(cols[None, :] >= L, (rows.shape[0], cols.shape[0]))
    if causal:
        masked = masked | (cols[None, :] >= rows[:, None])
    return masked


MIRROR_MUTANTS = {
    "l not rescaled": ("online_update", _no_l_rescale),
    "acc not rescaled": ("online_update", _no_acc_rescale),
    "correction inverted": ("online_update", _inverted_correction),
    "no -inf guard": ("online_update", _unguarded),
    "causal mask uses >=": ("block_mask", _mask_ge),
}


def mirror_agrees(lib) -> bool:
    for (B, H, N, D, causal, kv_len, block) in [(2, 2, 20, 6, True, [20, 0], 4),
                                                 (1, 2, 17, 4, False, None, 5)]:
        q, k, v = rand(B, H, N, D, 600 + N)
        o, lse = lib.attention(q, k, v, causal=causal, kv_len=kv_len)
        with np.errstate(invalid="ignore"):
            mo, mlse = tiled.forward(q, k, v, causal=causal, kv_len=kv_len, block=block)
        if not (np.allclose(mo, o, atol=1e-10) and
                np.array_equal(np.isneginf(mlse), np.isneginf(lse)) and
                np.allclose(mlse[np.isfinite(lse)], lse[np.isfinite(lse)], atol=1e-10)):
            return False
    return True


def test_mirror_agrees_unmutated(oracle_lib):
    assert mirror_agrees(oracle_lib)


@pytest.mark.parametrize("name", sorted(MIRROR_MUTANTS))
def test_mirror_mutant_is_caught(oracle_lib, monkeypatch, name):
    attr, fn = MIRROR_MUTANTS[name]
    monkeypatch.setattr(tiled, attr, fn)
    assert not mirror_agrees(oracle_lib), f"mirror mutant {name!r} survived"
