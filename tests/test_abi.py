"""The C ABI library on the host: it builds, loads, exports every symbol that
include/fa.h declares, and rejects bad arguments before touching a GPU.

No call here reaches a CUDA API: every case returns from the host-side checks.
"""
import os
import re
import shutil

import pytest

import exact_tiled_attention_23_gb300 as fa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="CUDA toolkit not present")


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_fp32", "fa_status_string", "fa_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_status_strings(lib):
    for code, name in [(0, "FA_OK"), (1, "FA_ERR_INVALID_ARG"), (2, "FA_ERR_UNSUPPORTED"),
                       (3, "FA_ERR_CUDA"), (4, "FA_ERR_TIMEOUT")]:
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_UNKNOWN_STATUS"


NAN = float("nan")
P = 0x10000  # a 16-byte-aligned stand-in address; never dereferenced (checks fail first)


@pytest.mark.parametrize("fn", [fa.fa_fwd, fa.fa_fwd_fp32])
def test_empty_problem_is_a_no_op(lib, fn):
    for (B, H, N) in [(0, 4, 16), (2, 0, 16), (2, 4, 0)]:
        assert fn(None, None, None, None, None, B, H, N, 64, 1, NAN, None, None) == fa.FA_OK


@pytest.mark.parametrize("fn", [fa.fa_fwd, fa.fa_fwd_fp32])
def test_null_and_negative_arguments(lib, fn):
    assert fn(None, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fn(P, P, P, None, None, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fn(P, P, P, P, None, -1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fn(P, P, P, P, None, 1, 1, -5, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fn(P, P, P, P, None, 1, 1, 16, 0, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("fn", [fa.fa_fwd, fa.fa_fwd_f16])
def test_tensor_core_head_dims(lib, fn):
    # multiples of 8 up to 128 run; the rest is rejected before any CUDA call
    for D in (4, 12, 100, 129, 136, 192, 264):
        assert fn(P, P, P, P, None, 1, 1, 16, D, 1, NAN, None, None) == fa.FA_ERR_UNSUPPORTED


def test_fp32_head_dim_limit(lib):
    assert fa.fa_fwd_fp32(P, P, P, P, None, 1, 1, 16, 257, 1, NAN, None, None) == fa.FA_ERR_UNSUPPORTED


def test_misaligned_pointers(lib):
    assert fa.fa_fwd(P + 2, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd(P, P, P, P + 8, None, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd(P, P, P, P, P + 2, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, P + 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_fp32(P + 2, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG


def test_grid_overflow_is_rejected(lib):
    # B*H*ceil(N/256) above 2^31-1 work items
    assert fa.fa_fwd(P, P, P, P, None, 65536, 65536, 512, 64, 1, NAN, None, None) == fa.FA_ERR_INVALID_ARG


def test_forward_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)


def test_splitkv_workspace_size(lib):
    # num_splits * B*H*N * (D + 1) floats
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 1024, 64, 3) == 3 * 2 * 8 * 1024 * 65 * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 128, 1) == 129 * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 16, 64, fa.FA_MAX_SPLITS + 1) == 0
    assert fa.fa_fwd_splitkv_workspace_bytes(-1, 1, 16, 64, 2) == 0


def test_splitkv_argument_checks(lib):
    big = 1 << 40
    # missing / misaligned workspace, split count out of range, too small a workspace
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, 2, None, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, 2, P + 4, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, -1, P, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, fa.FA_MAX_SPLITS + 1, P, big, None) == fa.FA_ERR_INVALID_ARG
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 1, 16, 64, 2)
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 64, 1, NAN, None, 2, P, need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 100, 1, NAN, None, 2, P, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv(P, P, P, P, None, 1, 1, 16, 256, 1, NAN, None, 2, P, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv(None, None, None, None, None, 1, 1, 0, 64, 1, NAN, None, 2, None, 0, None) == fa.FA_OK


def test_bwd_workspace_and_argument_checks(lib):
    assert fa.fa_bwd_workspace_bytes(2, 3, 100, 64) == 2 * 3 * 100 * 65 * 4
    assert fa.fa_bwd_workspace_bytes(1, 1, -1, 64) == 0
    big = 1 << 40
    assert fa.fa_bwd(P, P, P, P, P, P, P, P, P, 1, 1, 16, 100, 1, NAN, None, P, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_f16(P, P, P, P, P, P, P, P, P, 1, 1, 16, 100, 1, NAN, None, P, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_f16(P, P, P, None, P, P, P, P, P, 1, 1, 16, 64, 1, NAN, None, P, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(P, P, P, P, P, P, P, P, P, 1, 1, 16, 256, 1, NAN, None, P, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd(P, P, P, None, P, P, P, P, P, 1, 1, 16, 64, 1, NAN, None, P, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(P, P, P, P, P, P, P, P, P, 1, 1, 16, 64, 1, NAN, None, None, big, None) == fa.FA_ERR_INVALID_ARG
    need = fa.fa_bwd_workspace_bytes(1, 1, 16, 64)
    assert fa.fa_bwd(P, P, P, P, P, P, P, P, P, 1, 1, 16, 64, 1, NAN, None, P, need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(P, P, P, P, P + 8, P, P, P, P, 1, 1, 16, 64, 1, NAN, None, P, big, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(None, None, None, None, None, None, None, None, None, 1, 1, 0, 64, 1, NAN, None, None, 0, None) == fa.FA_OK


def test_from_host_argument_checks(lib):
    """fa_fwd_from_host rejects bad arguments before creating streams or
    copying anything."""
    H_ = P + (1 << 20)      # stands in for a host array (never dereferenced here)
    args = lambda **kw: dict(dict(Qh=H_, Kh=H_, Vh=H_, Oh=H_, Lh=None, Qd=P, Kd=P, Vd=P, Od=P, Ld=None,
                                  B=1, H=2, N=16, D=64, groups=0), **kw)

    def call(a):
        return fa.fa_fwd_from_host(a["Qh"], a["Kh"], a["Vh"], a["Oh"], a["Lh"], a["Qd"], a["Kd"], a["Vd"],
                                   a["Od"], a["Ld"], a["B"], a["H"], a["N"], a["D"], 1, NAN, None, 0,
                                   a["groups"], None)
    assert call(args(Qh=None)) == fa.FA_ERR_INVALID_ARG
    assert call(args(Od=None)) == fa.FA_ERR_INVALID_ARG
    assert call(args(Lh=H_, Ld=None)) == fa.FA_ERR_INVALID_ARG          # LSE wanted, no device buffer
    assert call(args(groups=-1)) == fa.FA_ERR_INVALID_ARG
    assert call(args(groups=fa.FA_MAX_HOST_GROUPS + 1)) == fa.FA_ERR_INVALID_ARG
    assert call(args(D=100)) == fa.FA_ERR_UNSUPPORTED
    assert call(args(Qd=P + 8)) == fa.FA_ERR_INVALID_ARG
    assert call(args(B=-1)) == fa.FA_ERR_INVALID_ARG
    assert call(args(N=0, Qh=None, Qd=None)) == fa.FA_OK                 # empty problem: nothing to do


def test_kernel_choice(lib, monkeypatch):
    """fa_fwd_kernel_choice answers without device work: D = 256 runs the
    one-tile kernel, unsupported head dims give 0, long rows at D = 128 the
    split-row kernel, many short items the two-tile kernel, and FA_FWD_TILES
    forces a kernel except at D = 256."""
    monkeypatch.delenv("FA_FWD_TILES", raising=False)
    assert fa.fa_fwd_kernel_choice(1, 2, 100, 256) == 1
    assert fa.fa_fwd_kernel_choice(1, 2, 100, 7) == 0
    assert fa.fa_fwd_kernel_choice(1, 2, 100, 136) == 0
    assert fa.fa_fwd_kernel_choice(1, 32, 16384, 128) == 3
    assert fa.fa_fwd_kernel_choice(8, 16, 8191, 64) == 2
    assert fa.fa_fwd_kernel_choice(4, 16, 4096, 128) == 2
    for forced in ("1", "2", "3"):
        monkeypatch.setenv("FA_FWD_TILES", forced)
        assert fa.fa_fwd_kernel_choice(4, 16, 4096, 128) == int(forced)
        assert fa.fa_fwd_kernel_choice(4, 16, 4096, 256) == 1


def test_auto_split_count(lib):
    """fa_fwd_splitkv_auto_splits splits only at D <= 64 with N >= 4096 and a
    single-pass grid that leaves SMs idle (148 or 152 SMs here give the same
    counts); otherwise 1, which runs the single-pass kernel."""
    assert fa.fa_fwd_splitkv_auto_splits(2, 8, 1024, 64) == 1
    assert fa.fa_fwd_splitkv_auto_splits(1, 1, 16384, 128) == 1
    assert fa.fa_fwd_splitkv_auto_splits(1, 2, 16384, 64) == 1
    assert fa.fa_fwd_splitkv_auto_splits(1, 1, 4096, 64) == 9
    assert fa.fa_fwd_splitkv_auto_splits(1, 1, 16384, 64) == 2
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 1024, 64, 0) == 2 * 8 * 1024 * 65 * 4
