"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so that the oracle and the CUDA path both read the same
inputs without sharing any of the method's code.

Every tensor is drawn on the CPU from ``torch.Generator('cpu')`` seeded with
``1234 + index`` (index = position of the workload below), in the order Q, K,
V (standard normal, fp32), then any row-selection mask, then the per-batch
key lengths.  Low-precision workloads round the fp32 draws to bf16 (or
fp16) with round-to-nearest-even; the oracle reads those same rounded values upcast to
fp32 (exact), so a measured error is the kernel's, not the input rounding's.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

SEED_BASE = 1234


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str            # "fp32", "bf16" or "fp16": the input / output element type
    B: int
    H: int
    N: int
    D: int
    causal: bool
    padded: str = "none"  # "none", "uniform0" (U{0..N}, batch 1 forced to 0), "uniform1" (U{1..N})
    spiky_rows: float = 0.0   # fraction of query rows multiplied by `spike`
    spike: float = 1.0
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


WORKLOADS = {
    w.name: w for w in [
        Workload("fp32_b1h2n128d64_causal", 0, "fp32", 1, 2, 128, 64, True,
                 note="fp32 path, tiny; the oracle runs it whole"),
        Workload("bf16_b2h8n1024d64_noncausal", 1, "bf16", 2, 8, 1024, 64, False,
                 note="short sequence, non-causal"),
        Workload("bf16_b2h8n1024d64_causal", 1, "bf16", 2, 8, 1024, 64, True,
                 note="short sequence, causal (same draws as the non-causal one)"),
        Workload("bf16_b4h16n4096d128_causal_padded_spiky", 2, "bf16", 4, 16, 4096, 128, True,
                 padded="uniform0", spiky_rows=0.05, spike=30.0,
                 note="5% of query rows x30 before rounding; key lengths U{0..N}, batch 1 at 0"),
        Workload("bf16_b1h32n16384d128_causal", 3, "bf16", 1, 32, 16384, 128, True,
                 note="long-context causal throughput workload"),
        Workload("bf16_b8h16n8191d64_noncausal_padded", 4, "bf16", 8, 16, 8191, 64, False,
                 padded="uniform1", note="ragged N; key lengths U{1..N}"),
    ]
}

# The workload whose throughput is the headline figure.
HEADLINE = "bf16_b1h32n16384d128_causal"


@dataclass
class Inputs:
    workload: Workload
    q: torch.Tensor          # [B,H,N,D] in the workload dtype (CPU)
    k: torch.Tensor
    v: torch.Tensor
    kv_len: Optional[torch.Tensor]   # int32 [B] (CPU) or None
    spiky: Optional[torch.Tensor] = field(default=None)   # bool [B,H,N] rows that were scaled

    @property
    def causal(self) -> bool:
        return self.workload.causal

    @property
    def scale(self) -> float:
        return self.workload.scale


def _torch_dtype(dtype: str):
    return {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[dtype]


def draw(B: int, H: int, N: int, D: int, dtype: str, seed: int, *, padded: str = "none",
         spiky_rows: float = 0.0, spike: float = 1.0, kv_len=None) -> tuple:
    """Draw (q, k, v, kv_len, spiky) with the recipe of the module docstring.

    kv_len, if given explicitly, overrides the `padded` rule (list or tensor).
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    spiky = None
    if spiky_rows > 0:
        spiky = torch.rand((B, H, N), generator=g) < spiky_rows
        q = torch.where(spiky[..., None], q * spike, q)
    lens = None
    if kv_len is not None:
        lens = torch.as_tensor(kv_len, dtype=torch.int32).reshape(B).clone()
    elif padded == "uniform0":
        lens = torch.randint(0, N + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
        if B > 1:
            lens[1] = 0
    elif padded == "uniform1":
        lens = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    elif padded != "none":
        raise ValueError(f"unknown padding rule {padded!r}")
    td = _torch_dtype(dtype)
    return q.to(td), k.to(td), v.to(td), lens, spiky


def make(name: str, heads: Optional[int] = None, dtype: Optional[str] = None,
         seq: Optional[int] = None, dim: Optional[int] = None) -> Inputs:
    """Inputs of a named workload (see WORKLOADS).  `heads`, `seq` and `dim`
    override H, N and D (a resized copy of the same workload, e.g. for
    profiler captures, the IO probe and other head dimensions) and `dtype` the
    element type of a 16-bit workload ("bf16" or "fp16")."""
    w = WORKLOADS[name]
    H = w.H if heads is None else int(heads)
    N = w.N if seq is None else int(seq)
    D = w.D if dim is None else int(dim)
    dt = w.dtype if dtype is None else dtype
    if (H, N, D, dt) != (w.H, w.N, w.D, w.dtype):
        suffix = (f"_h{H}" if H != w.H else "") + (f"_n{N}" if N != w.N else "") + \
                 (f"_d{D}" if D != w.D else "") + (f"_{dt}" if dt != w.dtype else "")
        w = Workload(f"{w.name}{suffix}", w.index, dt, w.B, H, N, D, w.causal,
                     padded=w.padded, spiky_rows=w.spiky_rows, spike=w.spike, note=w.note)
    q, k, v, lens, spiky = draw(w.B, w.H, w.N, w.D, w.dtype, w.seed, padded=w.padded,
                                spiky_rows=w.spiky_rows, spike=w.spike)
    return Inputs(w, q, k, v, lens, spiky)


def make_case(B: int, H: int, N: int, D: int, dtype: str = "bf16", causal: bool = True,
              seed: int = 0, kv_len=None, padded: str = "none") -> Inputs:
    """An ad-hoc small case for parity and edge-case tests."""
    w = Workload(f"case_b{B}h{H}n{N}d{D}", 0, dtype, B, H, N, D, causal, padded=padded)
    q, k, v, lens, spiky = draw(B, H, N, D, dtype, SEED_BASE + 1000 + seed, padded=padded,
                                kv_len=kv_len)
    return Inputs(w, q, k, v, lens, spiky)


def unmasked_pairs(N: int, causal: bool, kv_len=None, B: int = 1, H: int = 1) -> int:
    """Exact count of (query, key) pairs the mask allows, over all (b, h).

    Counting, not attention arithmetic: it sizes the FLOP figure of a run.
    """
    total = 0
    lens = [N] * B if kv_len is None else [min(max(int(x), 0), N) for x in kv_len]
    for L in lens:
        if causal:
            # rows i < L see i+1 keys; rows i >= L see L keys
            total += L * (L + 1) // 2 + (N - L) * L
        else:
            total += N * L
    return total * H
