"""Python binding of the C ABI in include/fa.h (libfa.so), via ctypes.

Argument marshalling only: every step of the attention forward and backward
passes runs in the library's CUDA kernels. PyTorch supplies device memory and streams. There
is no fallback: if the library is missing or the device is unsupported, the
calls raise.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

from .build import INCLUDE, LIB

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_BOUNDS = range(6)
FA_DEBUG_SERIALIZE_FLAG, FA_DEBUG_BOUNDS_FLAG = 1, 2
FA_MASK_NONE, FA_MASK_CAUSAL, FA_MASK_WINDOW = range(3)
FA_DTYPE_FP16, FA_DTYPE_BF16 = range(2)

_MASKS = {"none": FA_MASK_NONE, "causal": FA_MASK_CAUSAL, "window": FA_MASK_WINDOW,
          FA_MASK_NONE: FA_MASK_NONE, FA_MASK_CAUSAL: FA_MASK_CAUSAL, FA_MASK_WINDOW: FA_MASK_WINDOW}
_DTYPES = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16}


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = "fa_forward"):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)}")


_lib = None


def load_library(path: str = LIB) -> ctypes.CDLL:
    """Load libfa.so (build it first with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = load_library_at(path)
    return _lib


def load_library_at(path: str) -> ctypes.CDLL:
    """Load a build of the library at `path` (for example a debug build) with its
    argument types declared, without replacing the one the binding uses."""
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    lib.fa_forward.restype = ctypes.c_int
    lib.fa_forward.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
        ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.fa_forward_gqa.restype = ctypes.c_int
    lib.fa_forward_gqa.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.fa_forward_splitkv.restype = ctypes.c_int
    lib.fa_forward_splitkv.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.fa_forward_splitkv_static.restype = ctypes.c_int
    lib.fa_forward_splitkv_static.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_void_p]
    lib.fa_forward_host.restype = ctypes.c_int
    lib.fa_forward_host.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 6 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.fa_forward_host_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_forward_host_workspace_bytes.argtypes = [ctypes.c_int64] * 8
    lib.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_splitkv_workspace_bytes.argtypes = [ctypes.c_int64] * 5
    lib.fa_splitkv_default_splits.restype = ctypes.c_int64
    lib.fa_splitkv_default_splits.argtypes = [ctypes.c_int64] * 5
    lib.fa_forward_varlen.restype = ctypes.c_int
    lib.fa_forward_varlen.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 7 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.fa_backward_varlen.restype = ctypes.c_int
    lib.fa_backward_varlen.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int64] * 8 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.fa_backward_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_backward_varlen_workspace_bytes.argtypes = [ctypes.c_int64] * 3
    lib.fa_backward.restype = ctypes.c_int
    lib.fa_backward.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int64] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.fa_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_backward_workspace_bytes.argtypes = [ctypes.c_int64] * 4
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_sync_status.restype = ctypes.c_int
    lib.fa_sync_status.argtypes = [ctypes.c_void_p]
    lib.fa_set_wait_budget_ns.restype = None
    lib.fa_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    lib.fa_launch_count.restype = ctypes.c_int64
    lib.fa_launch_count.argtypes = []
    lib.fa_test_arm_fault.restype = None
    lib.fa_test_arm_fault.argtypes = [ctypes.c_int32]
    lib.fa_test_arm_row_shift.restype = None
    lib.fa_test_arm_row_shift.argtypes = [ctypes.c_int64]
    lib.fa_debug_flags.restype = ctypes.c_int32
    lib.fa_debug_flags.argtypes = []
    return lib


def declared_functions() -> list[str]:
    """Names of the functions include/*.h declares (for export checks)."""
    names = []
    for fn in sorted(os.listdir(INCLUDE)):
        if fn.endswith(".h"):
            with open(os.path.join(INCLUDE, fn)) as f:
                src = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names += re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_sync_status(stream=None) -> int:
    return load_library().fa_sync_status(_stream_handle(stream))


def fa_set_wait_budget_ns(ns: int) -> None:
    load_library().fa_set_wait_budget_ns(int(ns))


def fa_launch_count() -> int:
    return load_library().fa_launch_count()


def fa_test_arm_fault(kv_position: int) -> None:
    """Test hook: the next launch skips one K load in every CTA (see include/fa.h)."""
    load_library().fa_test_arm_fault(int(kv_position))


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(q, k, v, o, lse, same_n=True):
    for t in (q, k, v, o, lse):
        if not t.is_cuda or not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype or o.dtype != q.dtype \
            or lse.dtype != torch.float32:
        raise FaError(FA_ERR_INVALID_ARG)
    if q.dim() != 4 or k.dim() != 4:
        raise FaError(FA_ERR_INVALID_ARG)
    B, H, N, d = q.shape
    if k.shape[0] != B or k.shape[3] != d or (same_n and k.shape[2] != N) or \
            v.shape != k.shape or o.shape != q.shape or lse.shape != (B, H, N):
        raise FaError(FA_ERR_INVALID_ARG)


def fa_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
               lse: torch.Tensor, scale: float, mask_mode=FA_MASK_NONE, window_left: int = 0,
               window_right: int = 0, stream=None) -> None:
    """Enqueue fa_forward on device tensors (B, H, N, d) -> o, lse (B, H, N)."""
    lib = load_library()
    _check(q, k, v, o, lse)
    if k.shape != q.shape:
        raise FaError(FA_ERR_INVALID_ARG)
    B, H, N, d = q.shape
    rc = lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, N, d, float(scale), _MASKS[mask_mode], int(window_left),
                        int(window_right), _DTYPES[q.dtype], _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc)


def fa_forward_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                   lse: torch.Tensor, scale: float, mask_mode=FA_MASK_NONE, window_left: int = 0,
                   window_right: int = 0, stream=None) -> None:
    """Enqueue fa_forward_gqa: q, o (B, H, N, d); k, v (B, H_kv, N, d); lse (B, H, N)."""
    lib = load_library()
    _check(q, k, v, o, lse)
    B, H, N, d = q.shape
    rc = lib.fa_forward_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, k.shape[1], N, d, float(scale),
                            _MASKS[mask_mode], int(window_left), int(window_right),
                            _DTYPES[q.dtype], _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc)


# Input bytes per chunk of forward()'s host pipeline.
HOST_CHUNK_BYTES = 64 << 20


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
            mask="none", window=(0, 0), stream=None, num_splits: int | None = None,
            out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None):
    """Attention forward: returns (O, LSE). K and V may have fewer heads than Q
    (grouped-query attention: H_kv must divide H) and more positions than Q (the
    queries are then the last positions; this runs the split-KV entry point, as
    does any num_splits, with 0 meaning its default).

    Device tensors run in place on the device. Host tensors go through
    fa_forward_host: the library copies them to the current CUDA device, processes
    and copies the results back in chunks of about HOST_CHUNK_BYTES (a batch entry
    and a range of K/V heads with their query heads), with the copy in of chunk
    c+1, the kernel on chunk c and the copy out of chunk c-1 overlapped, and this
    call returns once O and LSE are in host memory. Pinned host tensors make the
    copies asynchronous; `out` / `lse_out` (host, pinned) receive the results and
    avoid allocating them per call. For host tensors, num_splits None or 0 means
    no key split when Nq == Nk and the default split count otherwise.
    """
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if q.is_cuda:
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o = torch.empty_like(q) if out is None else out
        lse = (torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
               if lse_out is None else lse_out)
        _forward_device(q, k, v, o, lse, scale, mask, window, stream, num_splits)
        return o, lse
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse_out is None:
        lse_out = torch.empty(q.shape[:-1], dtype=torch.float32, pin_memory=True)
    fa_forward_host(q, k, v, out, lse_out, scale, mask, window[0], window[1],
                    num_splits or 0, HOST_CHUNK_BYTES, None, stream)
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    return out, lse_out


def fa_forward_host_workspace_bytes(B: int, H: int, H_kv: int, Nq: int, Nk: int, d: int,
                                    num_splits: int = 0, chunk_bytes: int = 0) -> int:
    return load_library().fa_forward_host_workspace_bytes(B, H, H_kv, Nq, Nk, d, num_splits,
                                                          chunk_bytes)


def fa_forward_host(q, k, v, o, lse, scale: float, mask_mode=FA_MASK_NONE, window_left: int = 0,
                    window_right: int = 0, num_splits: int = 0, chunk_bytes: int = 0,
                    workspace: torch.Tensor | None = None, stream=None) -> None:
    """Enqueue fa_forward_host on host tensors q, o (B, H, Nq, d), k, v (B, H_kv, Nk,
    d) and lse (B, H, Nq) float32. Without a workspace tensor one is taken from
    PyTorch's caching allocator on the current device (released to it once this
    call's work on `stream` is done)."""
    lib = load_library()
    for t in (q, k, v, o, lse):
        if t.is_cuda or not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype or o.dtype != q.dtype:
        raise FaError(FA_ERR_INVALID_ARG)
    if lse.dtype != torch.float32:
        raise FaError(FA_ERR_INVALID_ARG)
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    need = fa_forward_host_workspace_bytes(B, H, H_kv, Nq, Nk, d, num_splits, chunk_bytes)
    if need == 0:
        raise FaError(FA_ERR_INVALID_ARG)
    dev = torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        workspace.record_stream(torch.cuda.current_stream(dev) if stream is None else stream)
    rc = lib.fa_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), B, H, H_kv, Nq, Nk, d, float(scale),
                             _MASKS[mask_mode], int(window_left), int(window_right),
                             _DTYPES[q.dtype], int(num_splits), int(chunk_bytes),
                             workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc)


def _forward_device(q, k, v, o, lse, scale, mask, window, stream, num_splits):
    if num_splits is not None or q.shape[2] != k.shape[2]:
        fa_forward_splitkv(q, k, v, o, lse, scale, mask, window[0], window[1],
                           num_splits or 0, None, stream)
    else:
        fa_forward_gqa(q, k, v, o, lse, scale, mask, window[0], window[1], stream)


def fa_splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return load_library().fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits)


def fa_splitkv_default_splits(B: int, H: int, H_kv: int, Nq: int, Nk: int) -> int:
    return load_library().fa_splitkv_default_splits(B, H, H_kv, Nq, Nk)


def fa_forward_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                       lse: torch.Tensor, scale: float, mask_mode=FA_MASK_NONE,
                       window_left: int = 0, window_right: int = 0, num_splits: int = 0,
                       workspace: torch.Tensor | None = None, stream=None) -> None:
    """Enqueue fa_forward_splitkv: q, o (B, H, Nq, d); k, v (B, H_kv, Nk, d);
    lse (B, H, Nq). num_splits = 0 takes fa_splitkv_default_splits. Without a
    workspace tensor one is taken from PyTorch's caching allocator."""
    lib = load_library()
    _check(q, k, v, o, lse, same_n=False)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if num_splits <= 0:
        num_splits = fa_splitkv_default_splits(B, H, k.shape[1], Nq, Nk)
    need = fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise FaError(FA_ERR_INVALID_ARG)
    rc = lib.fa_forward_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, H, k.shape[1], Nq, Nk, d, float(scale),
                                _MASKS[mask_mode], int(window_left), int(window_right),
                                _DTYPES[q.dtype], int(num_splits), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc)


FA_SPLITKV_STATIC_SCRATCH_BYTES = 16 << 20


def fa_forward_splitkv_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                              lse: torch.Tensor, scale: float, mask_mode=FA_MASK_NONE,
                              window_left: int = 0, window_right: int = 0, num_splits: int = 1,
                              stream=None) -> None:
    """Enqueue fa_forward_splitkv_static: split-KV attention whose scratch is the
    library's fixed device array (no allocation; see include/fa.h)."""
    lib = load_library()
    _check(q, k, v, o, lse, same_n=False)
    B, H, Nq, d = q.shape
    rc = lib.fa_forward_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, H, k.shape[1], Nq, k.shape[2], d,
                                       float(scale), _MASKS[mask_mode], int(window_left),
                                       int(window_right), _DTYPES[q.dtype], int(num_splits),
                                       _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc)


def fa_backward_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return load_library().fa_backward_workspace_bytes(B, H, N, d)


def fa_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                do: torch.Tensor, lse: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
                dv: torch.Tensor, scale: float, mask_mode=FA_MASK_NONE, window_left: int = 0,
                window_right: int = 0, workspace: torch.Tensor | None = None,
                stream=None) -> None:
    """Enqueue fa_backward: q, o, do, dq (B, H, N, d); k, v, dk, dv (B, H_kv, N, d);
    lse (B, H, N) float32 from the forward. Without a workspace tensor one is
    taken from PyTorch's caching allocator."""
    lib = load_library()
    _check(q, k, v, o, lse)
    for t, like in ((do, q), (dq, q), (dk, k), (dv, k)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.shape != like.shape:
            raise FaError(FA_ERR_INVALID_ARG, "fa_backward")
    B, H, N, d = q.shape
    need = fa_backward_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise FaError(FA_ERR_INVALID_ARG, "fa_backward")
    rc = lib.fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         B, H, k.shape[1], N, d, float(scale), _MASKS[mask_mode],
                         int(window_left), int(window_right), _DTYPES[q.dtype],
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                         _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_backward")


def backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, do: torch.Tensor, scale: float | None = None, mask="none",
             window=(0, 0), stream=None):
    """Attention backward on device tensors: returns (dQ, dK, dV) for the forward
    that produced (o, lse) from (q, k, v) and the upstream gradient do."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    q, k, v, o, lse, do = (t.contiguous() for t in (q, k, v, o, lse, do))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_backward(q, k, v, o, do, lse, dq, dk, dv, scale, mask, window[0], window[1], None, stream)
    return dq, dk, dv


def fa_forward_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                      lse: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                      max_seqlen_q: int, scale: float, mask_mode=FA_MASK_NONE,
                      window_left: int = 0, window_right: int = 0, stream=None) -> None:
    """Enqueue fa_forward_varlen: q, o (total_q, H, d); k, v (total_k, H_kv, d);
    lse (total_q, H) float32; cu_seqlens_q / _k int32 (B + 1,) on the device."""
    lib = load_library()
    for t in (q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k):
        if not t.is_cuda or not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG, "fa_forward_varlen")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype or o.dtype != q.dtype \
            or lse.dtype != torch.float32 or cu_seqlens_q.dtype != torch.int32 \
            or cu_seqlens_k.dtype != torch.int32 or q.dim() != 3 or k.dim() != 3:
        raise FaError(FA_ERR_INVALID_ARG, "fa_forward_varlen")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if k.shape[2] != d or v.shape != k.shape or o.shape != q.shape or lse.shape != (total_q, H) \
            or cu_seqlens_k.numel() != B + 1 or B < 1:
        raise FaError(FA_ERR_INVALID_ARG, "fa_forward_varlen")
    rc = lib.fa_forward_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                               B, H, H_kv, total_q, total_k, int(max_seqlen_q), d, float(scale),
                               _MASKS[mask_mode], int(window_left), int(window_right),
                               _DTYPES[q.dtype], _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_forward_varlen")


def fa_backward_varlen_workspace_bytes(B: int, H: int, total_q: int) -> int:
    return load_library().fa_backward_varlen_workspace_bytes(B, H, total_q)


def fa_backward_varlen(q, k, v, o, do, lse, cu_seqlens_q, cu_seqlens_k, dq, dk, dv,
                       max_seqlen_q: int, max_seqlen_k: int, scale: float, mask_mode=FA_MASK_NONE,
                       window_left: int = 0, window_right: int = 0, workspace=None,
                       stream=None) -> None:
    """Enqueue fa_backward_varlen: q, o, do, dq (total_q, H, d); k, v, dk, dv
    (total_k, H_kv, d); lse (total_q, H) float32; cu_seqlens_* int32 (B + 1,)."""
    lib = load_library()
    ts = (q, k, v, o, do, lse, cu_seqlens_q, cu_seqlens_k, dq, dk, dv)
    if any(not t.is_cuda or not t.is_contiguous() for t in ts) or q.dim() != 3 or k.dim() != 3:
        raise FaError(FA_ERR_INVALID_ARG, "fa_backward_varlen")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    need = fa_backward_varlen_workspace_bytes(B, H, total_q)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = lib.fa_backward_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                do.data_ptr(), lse.data_ptr(), cu_seqlens_q.data_ptr(),
                                cu_seqlens_k.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, H_kv, total_q, total_k, int(max_seqlen_q),
                                int(max_seqlen_k), d, float(scale), _MASKS[mask_mode],
                                int(window_left), int(window_right), _DTYPES[q.dtype],
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_backward_varlen")
