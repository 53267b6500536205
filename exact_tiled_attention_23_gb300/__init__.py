"""Exact tiled attention for GB300 -- Python binding of libfa.so.

The functions named like the C ABI (``fa_fwd``, ``fa_fwd_f16``,
``fa_fwd_fp32``, ``fa_fwd_splitkv``, ``fa_fwd_splitkv_noalloc``,
``fa_fwd_from_host``, ``fa_bwd``, ``fa_bwd_f16``, the workspace and status
helpers) take raw pointers and sizes exactly as declared in ``include/fa.h``
and only marshal arguments through ctypes.  The torch conveniences on top:

* ``forward()`` -- O, LSE for CUDA tensors (allocates O and LSE with torch);
* ``forward_from_host()`` -- the same for CPU tensors, copies overlapped with
  the computation;
* ``backward()`` -- dQ, dK, dV by recomputation;
* ``attention()`` -- a differentiable torch operation (forward + backward).

Every step of the computation runs in the library's CUDA kernels; there is no
other code path, and calling without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
           "FAError", "load", "library_path", "fa_fwd", "fa_fwd_fp32", "fa_status_string",
           "fa_device_status", "fa_last_error_detail", "fa_fwd_splitkv",
           "fa_fwd_splitkv_workspace_bytes", "fa_fwd_splitkv_auto_splits", "fa_fwd_kernel_choice", "FA_MAX_SPLITS",
           "fa_fwd_splitkv_noalloc", "FA_NOALLOC_SCRATCH_BYTES", "fa_fwd_f16",
           "fa_bwd", "fa_bwd_f16", "fa_bwd_workspace_bytes", "backward", "attention",
           "fa_fwd_from_host", "fa_fwd_from_host_auto_groups", "FA_MAX_HOST_GROUPS", "forward_from_host",
           "forward", "build"]

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_MAX_SPLITS = 64
FA_NOALLOC_SCRATCH_BYTES = 32 << 20
FA_MAX_HOST_GROUPS = 1024

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {fa_status_string(status)}")


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force, verbose=verbose)


def load():
    """The loaded ctypes library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA attention library is not built ({path}); "
                               "run exact_tiled_attention_23_gb300.build() first")
        lib = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp]
        lib.fa_fwd.argtypes = fwd_args
        lib.fa_fwd.restype = i32
        lib.fa_fwd_fp32.argtypes = fwd_args
        lib.fa_fwd_fp32.restype = i32
        lib.fa_fwd_f16.argtypes = fwd_args
        lib.fa_fwd_f16.restype = i32
        lib.fa_status_string.argtypes = [i32]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_status.argtypes = [vp]
        lib.fa_device_status.restype = i32
        lib.fa_last_error_detail.argtypes = []
        lib.fa_last_error_detail.restype = ctypes.c_uint32
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, i32, vp,
                                       ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = i32
        lib.fa_fwd_splitkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv_auto_splits.argtypes = [i32, i32, i32, i32]
        lib.fa_fwd_splitkv_auto_splits.restype = i32
        lib.fa_fwd_kernel_choice.argtypes = [i32, i32, i32, i32]
        lib.fa_fwd_kernel_choice.restype = i32
        lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp,
                                               i32, vp]
        lib.fa_fwd_splitkv_noalloc.restype = i32
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp,
                               ctypes.c_size_t, vp]
        lib.fa_bwd.restype = i32
        lib.fa_bwd_f16.argtypes = lib.fa_bwd.argtypes
        lib.fa_bwd_f16.restype = i32
        lib.fa_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_from_host.argtypes = [vp] * 10 + [i32, i32, i32, i32, i32, f32, vp, i32, i32, vp]
        lib.fa_fwd_from_host.restype = i32
        lib.fa_fwd_from_host_auto_groups.argtypes = [i32, i32, i32, i32]
        lib.fa_fwd_from_host_auto_groups.restype = i32
        _lib = lib
        return lib


# ---------------------------------------------------------------- raw C ABI
def fa_fwd(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream) -> int:
    """bf16 forward; pointers are integers (device addresses) or None."""
    return int(load().fa_fwd(Q, K, V, O, LSE, B, H, N, D, int(bool(causal)), float(scale),
                             kv_len, stream))


def fa_fwd_f16(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream) -> int:
    """fp16 forward on the tensor cores; pointers are integers (device addresses) or None."""
    return int(load().fa_fwd_f16(Q, K, V, O, LSE, B, H, N, D, int(bool(causal)), float(scale),
                                 kv_len, stream))


def fa_fwd_fp32(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream) -> int:
    """fp32 forward; pointers are integers (device addresses) or None."""
    return int(load().fa_fwd_fp32(Q, K, V, O, LSE, B, H, N, D, int(bool(causal)), float(scale),
                                  kv_len, stream))


def fa_fwd_splitkv(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, num_splits, workspace,
                   workspace_bytes, stream) -> int:
    """Split-KV bf16 forward with a caller-provided device workspace."""
    return int(load().fa_fwd_splitkv(Q, K, V, O, LSE, B, H, N, D, int(bool(causal)), float(scale),
                                     kv_len, int(num_splits), workspace, int(workspace_bytes), stream))


def fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, num_splits,
                           stream) -> int:
    """Split-KV forward on the library's fixed device scratch, for callers
    that cannot allocate device memory (no workspace argument; the call
    allocates nothing).  Problems needing more than FA_NOALLOC_SCRATCH_BYTES
    of scratch return FA_ERR_UNSUPPORTED.  Calls that overlap on the GPU
    share the scratch and race."""
    return int(load().fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, B, H, N, D, int(bool(causal)),
                                             float(scale), kv_len, int(num_splits), stream))


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, causal, scale, kv_len, workspace,
           workspace_bytes, stream) -> int:
    """bf16 backward by recomputation; pointers are device addresses or None."""
    return int(load().fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, int(bool(causal)),
                             float(scale), kv_len, workspace, int(workspace_bytes), stream))


def fa_fwd_from_host(Q_host, K_host, V_host, O_host, LSE_host, Q_dev, K_dev, V_dev, O_dev, LSE_dev,
                     B, H, N, D, causal, scale, kv_len, f16, groups, stream) -> int:
    """Forward over host arrays, copies overlapped with the computation in
    `groups` (batch, head) groups; the device buffers are the caller's."""
    return int(load().fa_fwd_from_host(Q_host, K_host, V_host, O_host, LSE_host, Q_dev, K_dev, V_dev,
                                       O_dev, LSE_dev, B, H, N, D, int(bool(causal)), float(scale),
                                       kv_len, int(bool(f16)), int(groups), stream))


def fa_fwd_from_host_auto_groups(B, H, N, D) -> int:
    return int(load().fa_fwd_from_host_auto_groups(B, H, N, D))


def fa_bwd_f16(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, causal, scale, kv_len, workspace,
               workspace_bytes, stream) -> int:
    """fp16 backward by recomputation; pointers are device addresses or None."""
    return int(load().fa_bwd_f16(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, int(bool(causal)),
                                 float(scale), kv_len, workspace, int(workspace_bytes), stream))


def fa_bwd_workspace_bytes(B, H, N, D) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, D))


def fa_fwd_splitkv_workspace_bytes(B, H, N, D, num_splits) -> int:
    return int(load().fa_fwd_splitkv_workspace_bytes(B, H, N, D, num_splits))


def fa_fwd_splitkv_auto_splits(B, H, N, D) -> int:
    return int(load().fa_fwd_splitkv_auto_splits(B, H, N, D))


def fa_fwd_kernel_choice(B, H, N, D) -> int:
    return int(load().fa_fwd_kernel_choice(B, H, N, D))


def fa_status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except RuntimeError:
        return {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
                4: "FA_ERR_TIMEOUT"}.get(int(status), "FA_UNKNOWN_STATUS")


def fa_device_status(stream) -> int:
    return int(load().fa_device_status(stream))


def fa_last_error_detail() -> int:
    return int(load().fa_last_error_detail())


# ---------------------------------------------------------------- torch call
def forward(q, k, v, causal: bool = True, scale=None, kv_len=None, out=None, lse=None,
            return_lse: bool = True, stream=None, splits=None, workspace=None):
    """O, LSE = attention(q, k, v) for CUDA tensors of shape [B, H, N, D].

    bf16 and fp16 inputs use the tensor-core path (D a multiple of 8 up to
    128, or 256); fp32 inputs use the fp32 path (D <= 256).  scale=None
    selects 1/sqrt(D).  kv_len: optional int32 CUDA tensor [B] of key
    lengths.  Runs asynchronously on `stream` (default: torch's current
    stream).

    splits: None for fa_fwd; an integer (0 = automatic) selects the split-KV
    path (bf16 only), whose workspace is `workspace` (a CUDA tensor of at
    least fa_fwd_splitkv_workspace_bytes bytes) or, if None, a torch
    allocation made here.
    """
    import torch

    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all have shape [B, H, N, D]")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float16,
                                                              torch.float32):
        raise ValueError("q, k, v must share dtype bfloat16, float16 or float32")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    kv_ptr = None
    if kv_len is not None:
        if kv_len.dtype != torch.int32 or not kv_len.is_cuda or kv_len.numel() != B:
            raise ValueError("kv_len must be an int32 CUDA tensor with B entries")
        kv_len = kv_len.contiguous()
        kv_ptr = kv_len.data_ptr()
    sc = float("nan") if scale is None else float(scale)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    if splits is not None:
        if q.dtype != torch.bfloat16:
            raise ValueError("the split-KV path takes bf16 inputs")
        need = fa_fwd_splitkv_workspace_bytes(B, H, N, D, int(splits))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, H, N, D, causal, sc,
                            kv_ptr, int(splits), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), sp)
        if st != FA_OK:
            raise FAError(st, "fa_fwd_splitkv")
        return (out, lse) if return_lse else out
    fn = {torch.bfloat16: fa_fwd, torch.float16: fa_fwd_f16, torch.float32: fa_fwd_fp32}[q.dtype]
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
            lse.data_ptr() if lse is not None else None, B, H, N, D, causal, sc, kv_ptr, sp)
    if st != FA_OK:
        raise FAError(st, fn.__name__)
    return (out, lse) if return_lse else out


def forward_from_host(q, k, v, causal: bool = True, scale=None, kv_len=None, out=None, lse=None,
                      device_buffers=None, groups: int = 0, stream=None):
    """O, LSE = attention(q, k, v) for bf16 / fp16 CPU tensors [B, H, N, D]
    (page-locked for asynchronous copies), through fa_fwd_from_host.  out
    and lse are CPU tensors to write (allocated page-locked when None);
    device_buffers = (q, k, v, o, lse) CUDA tensors of the same shapes
    (allocated with torch when None).  kv_len: optional int32 CUDA tensor
    [B].  Returns (out, lse) after the stream has finished."""
    import torch

    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all have shape [B, H, N, D]")
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise ValueError("q, k, v must be CPU tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must share dtype bfloat16 or float16")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    if device_buffers is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        device_buffers = (torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty((B, H, N), dtype=torch.float32, device=dev))
    qd, kd, vd, od, ld = device_buffers
    kv_ptr = None
    if kv_len is not None:
        if kv_len.dtype != torch.int32 or not kv_len.is_cuda or kv_len.numel() != B:
            raise ValueError("kv_len must be an int32 CUDA tensor with B entries")
        kv_ptr = kv_len.contiguous().data_ptr()
    if stream is None:
        stream = torch.cuda.current_stream()
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    st = fa_fwd_from_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                          qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(),
                          B, H, N, D, causal, float("nan") if scale is None else float(scale), kv_ptr,
                          q.dtype == torch.float16, groups, sp)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_from_host")
    if hasattr(stream, "synchronize"):
        stream.synchronize()
    else:
        torch.cuda.synchronize()
    return out, lse


def backward(q, k, v, o, do, lse, causal: bool = True, scale=None, kv_len=None, workspace=None,
             stream=None):
    """(dQ, dK, dV) of sum(O * dO) for O, LSE = forward(q, k, v, ...), bf16
    or fp16 CUDA tensors [B, H, N, D] with D a multiple of 8 up to 128 (LSE
    fp32 [B, H, N]).  The workspace (a CUDA
    tensor of at least fa_bwd_workspace_bytes bytes) is allocated here with
    torch when not given."""
    import torch

    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, o, do must be bf16 or fp16")
    for x in (q, k, v, o, do):
        if x.shape != q.shape or x.dtype != q.dtype or not x.is_cuda:
            raise ValueError("q, k, v, o, do must be CUDA tensors of one dtype and shape [B, H, N, D]")
    q, k, v, o, do = (x.contiguous() for x in (q, k, v, o, do))
    B, H, N, D = q.shape
    lse = lse.contiguous()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    need = fa_bwd_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    kv_ptr = None
    if kv_len is not None:
        if kv_len.dtype != torch.int32 or not kv_len.is_cuda or kv_len.numel() != B:
            raise ValueError("kv_len must be an int32 CUDA tensor with B entries")
        kv_len = kv_len.contiguous()
        kv_ptr = kv_len.data_ptr()
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    bwd = fa_bwd_f16 if q.dtype == torch.float16 else fa_bwd
    st = bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D, causal,
             float("nan") if scale is None else float(scale), kv_ptr, workspace.data_ptr(),
             workspace.numel() * workspace.element_size(), sp)
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


# ------------------------------------------------------------- autograd
def _attention_function():
    import torch

    class _Attention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, scale, kv_len):
            o, lse = forward(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
            ctx.save_for_backward(q, k, v, o, lse, kv_len)
            ctx.causal, ctx.scale = causal, scale
            return o

        @staticmethod
        def backward(ctx, d_o):
            q, k, v, o, lse, kv_len = ctx.saved_tensors
            dq, dk, dv = backward(q, k, v, o, d_o.contiguous(), lse, causal=ctx.causal, scale=ctx.scale,
                                  kv_len=kv_len)
            return dq, dk, dv, None, None, None

    return _Attention


_ATTENTION = None


def attention(q, k, v, causal: bool = True, scale=None, kv_len=None):
    """softmax(scale * q k^T + mask) v as a differentiable torch operation:
    the forward is fa_fwd / fa_fwd_f16 and the backward fa_bwd / fa_bwd_f16
    (bf16 or fp16 CUDA tensors [B, H, N, D], D a multiple of 8 up to 128)."""
    global _ATTENTION
    if _ATTENTION is None:
        _ATTENTION = _attention_function()
    return _ATTENTION.apply(q, k, v, bool(causal), scale, kv_len)
