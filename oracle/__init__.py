"""fp64 CPU oracle for the attention forward pass -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product (the CUDA library and its
Python binding) never calls it and shares no code with it.

The arithmetic lives in ``attention_oracle.c`` (forward) and
``attention_bwd_oracle.c`` (gradients), plain loops in double precision; see
their headers for the definitions they follow and the passages of the pages
they cite. This module compiles them with gcc and marshals arguments.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attention_oracle.c"), os.path.join(_HERE, "attention_bwd_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")

FP16, BF16 = 0, 1
MASKS = {"none": 0, "causal": 1, "window": 2, 0: 0, 1: 1, 2: 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (plain gcc, no fast-math) next to its source."""
    if (force or not os.path.exists(_LIB)
            or os.path.getmtime(_LIB) < max(os.path.getmtime(s) for s in _SRCS)):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_attention_ex.restype = ctypes.c_int
        lib.oracle_attention_ex.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64,
            ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        _lib = lib
    return _lib


def decode16(bits: int, dtype: torch.dtype) -> float:
    lib = _load()
    if dtype == torch.float16:
        return lib.oracle_fp16_to_double(bits)
    return lib.oracle_bf16_to_double(bits)


def _bits(t: torch.Tensor) -> np.ndarray:
    assert t.device.type == "cpu" and t.dtype in (torch.float16, torch.bfloat16)
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy()).view(np.uint16)


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
              mask="none", window=(0, 0), units=None, nthreads: int | None = None,
              return_p: bool = False, online_bc: int = 0):
    """fp64 attention over 16-bit CPU tensors: Q (B, H, Nq, d), K and V
    (B, Hk, Nk, d) with Hk dividing H (grouped-query attention when Hk < H).
    Query i stands at key position i + Nk - Nq (the masks refer to that).

    ``units`` is a list of (b*H + h, row0, row1); by default every row of
    every head. Returns (O, LSE[, P]) as float64 numpy arrays with rows packed
    in unit order: O (rows, d), LSE (rows,), P (rows, N).
    ``online_bc > 0`` evaluates the online-softmax recurrence with key blocks
    of that size instead of the direct definition.
    """
    lib = _load()
    B, H, Nq, d = q.shape
    Hk, N = k.shape[1], k.shape[2]
    assert k.shape == (B, Hk, N, d) and v.shape == k.shape
    assert q.dtype == k.dtype == v.dtype
    dt = FP16 if q.dtype == torch.float16 else BF16
    if units is None:
        units = [(bh, 0, Nq) for bh in range(B * H)]
    u = np.ascontiguousarray(np.array(units, dtype=np.int64).reshape(-1, 3))
    rows = int((u[:, 2] - u[:, 1]).sum()) if len(u) else 0
    O = np.zeros((rows, d), dtype=np.float64)
    LSE = np.zeros((rows,), dtype=np.float64)
    P = np.zeros((rows, N), dtype=np.float64) if return_p else None
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_attention_ex(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, dt, B, H, Hk, Nq, N, d,
        float(scale), MASKS[mask], int(window[0]), int(window[1]),
        u.ctypes.data, len(u), O.ctypes.data, LSE.ctypes.data,
        P.ctypes.data if P is not None else None, int(online_bc), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    if return_p:
        return O, LSE, P
    return O, LSE


def attention_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, do: torch.Tensor,
                  scale: float, mask="none", window=(0, 0), kv_heads=None,
                  nthreads: int | None = None):
    """fp64 gradients of the attention forward over 16-bit CPU tensors, for an
    upstream gradient ``do`` of O: Q and dO (B, H, Nq, d), K and V (B, Hk, Nk, d).

    ``kv_heads`` lists K/V heads b*Hk + hk (default: all). Returns float64 numpy
    arrays dQ (n, H/Hk, Nq, d) -- the query heads reading each listed K/V head, in
    order -- and dK, dV (n, Nk, d).
    """
    lib = _load()
    B, H, Nq, d = q.shape
    Hk, N = k.shape[1], k.shape[2]
    assert k.shape == (B, Hk, N, d) and v.shape == k.shape and do.shape == q.shape
    assert q.dtype == k.dtype == v.dtype == do.dtype
    dt = FP16 if q.dtype == torch.float16 else BF16
    if kv_heads is None:
        kv_heads = list(range(B * Hk))
    kv = np.ascontiguousarray(np.array(kv_heads, dtype=np.int64).reshape(-1))
    n, group = len(kv), H // Hk
    dQ = np.zeros((n, group, Nq, d), dtype=np.float64)
    dK = np.zeros((n, N, d), dtype=np.float64)
    dV = np.zeros((n, N, d), dtype=np.float64)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(do)
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_attention_bwd(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, db.ctypes.data, dt, B, H, Hk, Nq, N, d,
        float(scale), MASKS[mask], int(window[0]), int(window[1]), kv.ctypes.data, n,
        dQ.ctypes.data, dK.ctypes.data, dV.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    return dQ, dK, dV
