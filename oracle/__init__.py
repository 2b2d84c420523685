"""CPU oracle for exact softmax attention — test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU product path (the package
``exact_tiled_attention_04_gb300``) never imports it, and it never imports
that package: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain three-pass softmax attention
in fp64, one query row at a time); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

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
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = f"{path}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
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
