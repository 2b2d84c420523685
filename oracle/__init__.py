"""CPU oracle for exact softmax attention — test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU product path (the package
``exact_tiled_attention_04_gb300``) never imports it, and it never imports
that package: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain three-pass softmax attention
in fp64, one query row at a time) and ``attn_bwd_oracle.c`` (its exact
gradients, row by row); this module only compiles them with gcc and marshals
numpy arrays through ctypes.

    O = softmax(scale * Q K^T) V,   lse_i = log sum_j exp(scale * q_i . k_j)

("CUDA Flash Attention: Online Softmax with Shared Memory Tiling", Problem
Statement; "FlashAttention dissected", softmax formula in "The mathematical
breakthrough: Tiling and Online Softmax".)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attn_bwd_oracle.c")]
_LIB_NAME = "liboracle_attn.so"
_lock = threading.Lock()
_lib = None


def build(out_dir: str | None = None, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc and return the shared library's path.

    ``mutant`` > 0 builds a copy with a deliberately planted mistake (see the
    ORACLE_MUTANT cases in attn_oracle.c); only the pin tests ask for one.
    """
    out_dir = out_dir or _HERE
    name = _LIB_NAME if mutant == 0 else f"liboracle_attn_mutant{mutant}.so"
    path = os.path.join(out_dir, name)
    if (not force and os.path.exists(path)
            and all(os.path.getmtime(path) >= os.path.getmtime(src) for src in _SRCS)):
        return path
    tmp = f"{path}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_attention_f64.restype = ctypes.c_int
    lib.oracle_attention_f64.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    lib.oracle_attention_f64_ex.restype = ctypes.c_int
    lib.oracle_attention_f64_ex.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    shape = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 6 + [ctypes.c_double, ctypes.c_int]
    lib.oracle_attention_bwd_f64.restype = ctypes.c_int
    lib.oracle_attention_bwd_f64.argtypes = shape + [ctypes.c_void_p] * 3 + [ctypes.c_int]
    lib.oracle_attention_bwd_dq_rows_f64.restype = ctypes.c_int
    lib.oracle_attention_bwd_dq_rows_f64.argtypes = shape + [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_attention_bwd_dkv_cols_f64.restype = ctypes.c_int
    lib.oracle_attention_bwd_dkv_cols_f64.argtypes = shape + [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    return lib


def load(mutant: int = 0):
    """Return the ctypes handle of the oracle library (building it if needed)."""
    global _lib
    if mutant:
        return _bind(build(mutant=mutant))
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def default_threads() -> int:
    return int(load().oracle_default_threads())


def attention_f64(q, k, v, scale: float, rows=None, threads: int = 0, lib=None):
    """Exact attention in fp64.

    q, k, v : float32 arrays [B, H, N, d] (values already rounded to the input
              dtype; they are widened to float64 inside the oracle).
    scale   : the score scale (the fp32 value the kernel receives, widened).
    rows    : None for every row, else an int array [R, 3] of (b, h, i).
    Returns (o, lse): float64 [B, H, N, d] and [B, H, N] for rows=None,
    else [R, d] and [R].
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"q, k, v must share one [B,H,N,d] shape: {q.shape} {k.shape} {v.shape}")
    B, H, N, d = (int(x) for x in q.shape)
    if rows is None:
        nrows = B * H * N
        rows_ptr = None
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        nrows = rows_arr.shape[0]
        rows_ptr = rows_arr.ctypes.data
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_attention_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                  B, H, N, d, float(scale), rows_ptr, nrows,
                                  o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_f64 failed with status {rc}")
    if rows is None:
        return o.reshape(B, H, N, d), lse.reshape(B, H, N)
    return o, lse


def attention_f64_ex(q, k, v, scale: float, rows=None, threads: int = 0, lib=None,
                     causal: bool = False):
    """Exact attention in fp64, general shapes: q [B, H, Nq, d], k and v
    [B, H_kv, Nkv, d] with H_kv dividing H (query head h uses key/value head
    h // (H // H_kv)).  causal: query i sees keys j <= i + (Nkv - Nq) only
    (no visible key: O = 0, lse = -inf).  Returns (o, lse): [B, H, Nq, d] and
    [B, H, Nq] for rows=None, else [R, d] and [R] for the (b, h, i) triples in
    `rows`."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] \
            or q.shape[3] != k.shape[3]:
        raise ValueError(f"incompatible shapes: q {q.shape}, k {k.shape}, v {v.shape}")
    B, H, Nq, d = (int(x) for x in q.shape)
    H_kv, Nkv = int(k.shape[1]), int(k.shape[2])
    if rows is None:
        nrows, rows_ptr = B * H * Nq, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        nrows, rows_ptr = rows_arr.shape[0], rows_arr.ctypes.data
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_attention_f64_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, H_kv, Nq,
                                     Nkv, d, float(scale), int(bool(causal)), rows_ptr, nrows,
                                     o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_f64_ex failed with status {rc}")
    if rows is None:
        return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)
    return o, lse


def flops(B: int, H: int, N: int, d: int, rows: int | None = None) -> float:
    """Algorithmic flops counted by the throughput metric: 4*N*d per query row
    (2*N*d for the scores, 2*N*d for the weighted sum of V)."""
    r = B * H * N if rows is None else rows
    return 4.0 * r * N * d


def _bwd_operands(q, k, v, dout):
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or dout.shape != q.shape \
            or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3] or q.shape[1] % k.shape[1]:
        raise ValueError(f"incompatible shapes: q {q.shape}, k {k.shape}, v {v.shape}, "
                         f"dout {dout.shape}")
    B, H, Nq, d = (int(x) for x in q.shape)
    H_kv, Nkv = int(k.shape[1]), int(k.shape[2])
    return (q, k, v, dout), (B, H, H_kv, Nq, Nkv, d)


def attention_bwd_f64(q, k, v, dout, scale: float, causal: bool = False, threads: int = 0,
                      lib=None):
    """Exact gradients of O = softmax(scale * Q K^T) V for the upstream
    gradient dout, in fp64.  q, dout: [B, H, Nq, d]; k, v: [B, H_kv, Nkv, d]
    (H_kv divides H).  Returns (dq, dk, dv) with the shapes of q, k, v.  The
    softmax weights are recomputed from their definition (no saved lse)."""
    lib = lib or load()
    ops, dims = _bwd_operands(q, k, v, dout)
    q, k, v, dout = ops
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    rc = lib.oracle_attention_bwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                      *dims, float(scale), int(bool(causal)), dq.ctypes.data,
                                      dk.ctypes.data, dv.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_f64 failed with status {rc}")
    return dq, dk, dv


def attention_bwd_dq_rows_f64(q, k, v, dout, scale: float, rows, causal: bool = False,
                              threads: int = 0, lib=None):
    """dQ of the query rows (b, h, i) in `rows` ([R, 3]); returns fp64 [R, d].
    Each row needs only its own scores, so this is cheap at any size."""
    lib = lib or load()
    ops, dims = _bwd_operands(q, k, v, dout)
    q, k, v, dout = ops
    rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    dq = np.empty((rows_arr.shape[0], dims[5]), dtype=np.float64)
    rc = lib.oracle_attention_bwd_dq_rows_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                              dout.ctypes.data, *dims, float(scale),
                                              int(bool(causal)), rows_arr.ctypes.data,
                                              rows_arr.shape[0], dq.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dq_rows_f64 failed with status {rc}")
    return dq


def attention_bwd_dkv_cols_f64(q, k, v, dout, scale: float, cols, causal: bool = False,
                               threads: int = 0, lib=None):
    """dK and dV of the keys (b, kv_head, j) in `cols` ([C, 3]); returns two
    fp64 [C, d] arrays.  Every query row of each requested key/value head is
    evaluated once (cost ~ 4 * group * Nq * Nkv * d per head)."""
    lib = lib or load()
    ops, dims = _bwd_operands(q, k, v, dout)
    q, k, v, dout = ops
    cols_arr = np.ascontiguousarray(cols, dtype=np.int64).reshape(-1, 3)
    dk = np.empty((cols_arr.shape[0], dims[5]), dtype=np.float64)
    dv = np.empty((cols_arr.shape[0], dims[5]), dtype=np.float64)
    rc = lib.oracle_attention_bwd_dkv_cols_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                               dout.ctypes.data, *dims, float(scale),
                                               int(bool(causal)), cols_arr.ctypes.data,
                                               cols_arr.shape[0], dk.ctypes.data, dv.ctypes.data,
                                               int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dkv_cols_f64 failed with status {rc}")
    return dk, dv
