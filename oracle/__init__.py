"""fp64 CPU oracle for single-token MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The library under test
(``mla_decode_stage1_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``mla_oracle.cpp`` (plain C++, fp64); this module only
compiles it with the host compiler and marshals numpy arrays through ctypes.
What it computes, and which page and section each step follows, is written at
the top of ``mla_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.cpp")
_LIB = os.path.join(_HERE, "libmla_oracle.so")

DT_BF16, DT_FP8_E4M3, DT_MXFP4 = 0, 1, 2
HEADS, QK_DIM, V_DIM = 16, 576, 512

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmla_oracle.so`` (host C++ only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", _SRC,
                               "-o", tmp, "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        for name in ("oracle_decode_bf16", "oracle_decode_e4m3", "oracle_decode_e2m1",
                     "oracle_decode_e8m0"):
            getattr(lib, name).argtypes = [P, i64, P]
            getattr(lib, name).restype = None
        lib.oracle_dequant_kv.argtypes = [i32, P, dbl, P, i64, i64, i64, P]
        lib.oracle_dequant_kv.restype = i32
        lib.oracle_mla_decode.argtypes = [i32, i32, i32, i32, P, dbl, P, dbl, P, i64,
                                          P, P, P, i32, P, i32, i32, P, P]
        lib.oracle_mla_decode.restype = i32
        lib.oracle_mla_decode_q.argtypes = [i32, i32, i32, i32, i32, P, dbl, P, dbl, P, i64,
                                            P, P, P, i32, P, i32, i32, P, P]
        lib.oracle_mla_decode_q.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def decode(fmt: str, codes) -> np.ndarray:
    """Decode raw codes with the oracle's own format decoder.

    fmt: 'bf16' (uint16 bit patterns), 'e4m3', 'e2m1' (low nibble), 'e8m0'.
    """
    lib = _load()
    dt = np.uint16 if fmt == "bf16" else np.uint8
    c = _c(codes, dt).ravel()
    out = np.empty(c.size, dtype=np.float64)
    fn = {"bf16": lib.oracle_decode_bf16, "e4m3": lib.oracle_decode_e4m3,
          "e2m1": lib.oracle_decode_e2m1, "e8m0": lib.oracle_decode_e8m0}[fmt]
    fn(_ptr(c), c.size, _ptr(out))
    return out


def dequant_kv(kv_dtype: int, kv, kv_scale: float = 1.0, e8m0=None, e8m0_stride: int = 0,
               row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Dequantise KV rows to fp64 [nrows, 576] with the oracle's decoders."""
    lib = _load()
    if kv_dtype == DT_BF16:
        k = _c(kv, np.uint16)
        total = k.size // QK_DIM
    elif kv_dtype == DT_FP8_E4M3:
        k = _c(kv, np.uint8)
        total = k.size // QK_DIM
    else:
        k = _c(kv, np.uint8)
        total = k.size // (QK_DIM // 2)
    e = _c(e8m0, np.uint8)
    if nrows is None:
        nrows = total - row0
    assert 0 <= row0 and row0 + nrows <= total
    out = np.empty((nrows, QK_DIM), dtype=np.float64)
    rc = lib.oracle_dequant_kv(kv_dtype, _ptr(k), float(kv_scale), _ptr(e), int(e8m0_stride),
                               row0, nrows, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dequant_kv rejected its arguments")
    return out


def mla_decode(*, bs: int, page_size: int, q_dtype: int, kv_dtype: int, q, kv,
               kv_indptr, kv_indices=None, kv_last_page_len=None, q_scale: float = 1.0,
               kv_scale: float = 1.0, e8m0=None, e8m0_stride: int = 0,
               num_splits: int = 0, select=None, nthreads: int | None = None, q_len: int = 1):
    """Reference decode.  Returns (o [n*q_len,16,512] fp64, lse [n*q_len,16]
    fp64) for the selected requests (all of them when ``select`` is None), row
    i*q_len + t holding query token t of the i-th selected request.

    q: raw bf16 bit patterns (uint16) or e4m3 bytes (uint8), shape
    [bs*q_len,16,576] (row b*q_len + t = query token t of request b).  Query
    token t of a request with n tokens attends to its first n - q_len + 1 + t
    tokens (causal over the last q_len positions).
    kv: raw rows (bf16 bits / e4m3 bytes / 288 packed MXFP4 bytes per row).
    kv_indptr is in pages; kv_indices None means the identity page table.
    """
    lib = _load()
    qa = _c(q, np.uint16 if q_dtype == DT_BF16 else np.uint8)
    ka = _c(kv, np.uint16 if kv_dtype == DT_BF16 else np.uint8)
    ea = _c(e8m0, np.uint8)
    ip = _c(kv_indptr, np.int32)
    ix = _c(kv_indices, np.int32)
    ll = _c(kv_last_page_len, np.int32)
    sel = _c(select, np.int32)
    n = (bs if sel is None else sel.size) * int(q_len)
    o = np.empty((n, HEADS, V_DIM), dtype=np.float64)
    lse = np.empty((n, HEADS), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    assert qa.size == bs * int(q_len) * HEADS * QK_DIM, "q must hold bs * q_len rows"
    rc = lib.oracle_mla_decode_q(bs, int(q_len), page_size, q_dtype, kv_dtype, _ptr(qa),
                               float(q_scale),
                               _ptr(ka), float(kv_scale), _ptr(ea), int(e8m0_stride),
                               _ptr(ip), _ptr(ix), _ptr(ll), int(num_splits), _ptr(sel),
                               0 if sel is None else sel.size, int(nthreads), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_mla_decode rejected its arguments")
    return o, lse
