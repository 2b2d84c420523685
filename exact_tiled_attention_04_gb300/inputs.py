"""Seeded synthetic inputs for the attention forward pass.

This module is the only code shared by the GPU path's tests/benchmark and the
CPU oracle's tests.  It holds no attention arithmetic: it draws numbers,
rounds them to the input dtype and names the workloads.

Generator (counter based, so any element can be drawn on its own):
  * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): output i of a stream with key K is
    mix64(K + (i+1)*0x9E3779B97F4A7C15) with the published mix64 finaliser.
  * Standard normals by the Box-Muller transform (Box & Muller, 1958) on
    pairs of 53-bit uniforms: u1 in (0, 1], u2 in [0, 1),
    z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = sqrt(-2 ln u1) sin(2 pi u2).
  * Values are drawn in float64, multiplied by the workload's factor, rounded
    to float32 (round to nearest even), then to bfloat16 (round to nearest
    even) for bf16 workloads.  The float32 arrays returned hold exactly the
    values the kernel reads.

The workloads follow the sizes the pages discuss: a single 512-row head like
the Tesla T4 runs of "CUDA Flash Attention: Online Softmax with Shared Memory
Tiling" (Performance Results), sequence lengths of 2048 and 8192, and the
N = 16,384 case that "How Did I Write My First FlashAttention Kernel in
CUDA?" uses to show that the N x N matrix exceeds 1 GB per head.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20  # pairs per chunk: bounds temporary memory

TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_ROWS, TENSOR_DO = 0, 1, 2, 3, 4


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (modifies a copy)."""
    z = np.array(z, dtype=np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    """Key of the SplitMix64 stream for (seed, tensor): output tensor_id of
    the stream keyed by the seed itself."""
    with np.errstate(over="ignore"):
        base = np.array([np.uint64(seed) + np.uint64(tensor_id + 1) * _GAMMA], dtype=np.uint64)
    return mix64(base)[0]


def uint64_stream(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the stream with the given key."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + idx * _GAMMA)


def _normal_pairs(key: np.uint64, p0: int, n: int, factor: float, out: np.ndarray) -> None:
    u = uint64_stream(key, 2 * p0, 2 * n)
    a = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    b = (u[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(a)) * factor
    t = (2.0 * np.pi) * b
    out[2 * p0:2 * (p0 + n):2] = r * np.cos(t)
    out[2 * p0 + 1:2 * (p0 + n):2] = r * np.sin(t)


def normals(seed: int, tensor_id: int, count: int, factor: float = 1.0) -> np.ndarray:
    """`count` float64 standard normals times `factor` (Box-Muller pairs).
    Chunks are independent (counter based), so they are drawn on a thread
    pool; the result does not depend on the thread count."""
    key = stream_key(seed, tensor_id)
    out = np.empty(count + (count & 1), dtype=np.float64)
    npairs = out.size // 2
    starts = list(range(0, npairs, _CHUNK))
    workers = max(1, min(len(starts), os.cpu_count() or 1, 32))
    if workers == 1:
        for p0 in starts:
            _normal_pairs(key, p0, min(_CHUNK, npairs - p0), factor, out)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(lambda p0: _normal_pairs(key, p0, min(_CHUNK, npairs - p0), factor, out), starts))
    return out[:count]


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 values that are exactly representable in bfloat16.  NaN stays
    NaN (quietened); +-inf stay infinite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    out = np.empty_like(bits)
    with np.errstate(over="ignore"):
        np.right_shift(bits, np.uint32(16), out=out)
        np.bitwise_and(out, np.uint32(1), out=out)
        out += np.uint32(0x7FFF)
        out += bits
        np.bitwise_and(out, np.uint32(0xFFFF0000), out=out)
    out = out.view(np.float32)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.float32(np.nan)
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def default_scale(d: int) -> np.float32:
    """1/sqrt(d) evaluated in float32, as 1.0f / sqrtf((float)d)."""
    return np.float32(1.0) / np.sqrt(np.float32(d))


@dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16", "f16" or "f32": the kernel's input/output dtype
    seed: int
    factor: float = 1.0   # multiplier applied to every drawn value
    identical_k_heads: tuple = ()      # (b, h): every K row equals that head's K row 0
    q_scaled_heads: tuple = ()         # (b, h, factor): that head's Q drawn times factor
    oracle_rows: int | None = None     # compare on this many seeded rows (None = all)
    note: str = ""
    H_kv: int = 0          # key/value heads (0: H, plain multi-head attention)
    Nkv: int = 0           # key/value rows per head (0: N; N is the query rows)
    causal: bool = False   # query i sees keys j <= i + Nkv - N only
    splits: int = 0        # key-range partitions (0: the library's plan for the device)
    backward: bool = False  # the step is the backward pass (dQ, dK, dV) for a fixed dO
    scale: np.float32 = field(init=False)

    def __post_init__(self):
        self.scale = default_scale(self.d)
        self.H_kv = self.H_kv or self.H
        self.Nkv = self.Nkv or self.N

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)

    @property
    def kv_shape(self):
        return (self.B, self.H_kv, self.Nkv, self.d)

    @property
    def general(self) -> bool:
        return self.H_kv != self.H or self.Nkv != self.N

    def visible_pairs(self) -> float:
        """(query, key) pairs that carry weight, per (b, h)."""
        if not self.causal:
            return float(self.N) * float(self.Nkv)
        off = self.Nkv - self.N
        i = np.arange(self.N, dtype=np.float64)
        return float(np.clip(i + off + 1, 0, self.Nkv).sum())

    def flops(self) -> float:
        """Forward: 4 d flops per visible (query, key) pair (Q K^T and P V),
        4*B*H*N^2*d unmasked.  Backward: 10 d per pair, the five products
        K Q^T, V dO^T, P^T dO, dS^T Q and dS K (2.5x the forward)."""
        per_pair = 10.0 if self.backward else 4.0
        return per_pair * self.B * self.H * self.visible_pairs() * self.d

    def bytes(self) -> float:
        """Algorithmic bytes.  Forward: read q, k, v once, write o and lse.
        Backward: read q, k, v, o, dO and lse once, write dq, dk, dv."""
        elem = 4 if self.dtype == "f32" else 2
        q_rows, kv_rows = self.B * self.H * self.N, self.B * self.H_kv * self.Nkv
        if self.backward:
            return elem * self.d * (4 * q_rows + 4 * kv_rows) + 4 * q_rows
        return elem * self.d * (2 * q_rows + 2 * kv_rows) + 4 * q_rows

    def describe(self) -> str:
        return f"{self.name}: B={self.B} H={self.H} N={self.N} d={self.d} {self.dtype}"


WORKLOADS = {
    "single_head_n512": Workload(
        "single_head_n512", 1, 1, 512, 64, "f32", seed=1,
        note="single head, fp32 inputs and output"),
    "tail_n1000": Workload(
        "tail_n1000", 2, 4, 1000, 64, "bf16", seed=2,
        identical_k_heads=((0, 1),), q_scaled_heads=((1, 2, 30.0),),
        note="N not a multiple of the tile; one head with identical keys, one with Q x30"),
    "b4h16_n2048": Workload("b4h16_n2048", 4, 16, 2048, 64, "bf16", seed=3),
    "b2h32_n8192_d128": Workload(
        "b2h32_n8192_d128", 2, 32, 8192, 128, "bf16", seed=4, factor=0.5,
        oracle_rows=512, note="compute-bound headline shape, values x0.5"),
    "long_n16384": Workload(
        "long_n16384", 1, 8, 16384, 64, "bf16", seed=5, oracle_rows=256,
        note="N x N scores would be 1 GB per head; never materialised"),
}
# Half of the headline shape (134 MB of q, k, v, o: still larger than the
# 129 MB L2); the case multi-pass profiler captures run on.
WORKLOADS["b1h32_n8192_d128"] = Workload(
    "b1h32_n8192_d128", 1, 32, 8192, 128, "bf16", seed=6, factor=0.5, oracle_rows=256,
    note="profiling case: half the headline shape")
# Shapes of the next rows: a decode step of a grouped-query model against a
# 16k-key cache (FlashDecoding: the keys split across the GPU), the headline
# shape with 4:1 grouped key/value heads, with the causal mask, and in fp16.
WORKLOADS["decode_b8h32kv8_n16384_d128"] = Workload(
    "decode_b8h32kv8_n16384_d128", 8, 32, 1, 128, "bf16", seed=7, H_kv=8, Nkv=16384,
    note="one query per head against a 16k-key cache, grouped heads, split-KV")
WORKLOADS["gqa_b2h32kv8_n8192_d128"] = Workload(
    "gqa_b2h32kv8_n8192_d128", 2, 32, 8192, 128, "bf16", seed=8, factor=0.5, H_kv=8,
    oracle_rows=256, note="headline shape, 4 query heads per key/value head")
WORKLOADS["causal_b2h32_n8192_d128"] = Workload(
    "causal_b2h32_n8192_d128", 2, 32, 8192, 128, "bf16", seed=9, factor=0.5, causal=True,
    oracle_rows=256, note="headline shape, causal mask")
WORKLOADS["f16_b2h32_n8192_d128"] = Workload(
    "f16_b2h32_n8192_d128", 2, 32, 8192, 128, "f16", seed=10, factor=0.5, oracle_rows=256,
    note="headline shape in fp16")
# The backward pass (gradients for a seeded dO) on the headline shape, with
# the causal mask, at d = 64, and on the half-size profiling case.
WORKLOADS["bwd_b2h32_n8192_d128"] = Workload(
    "bwd_b2h32_n8192_d128", 2, 32, 8192, 128, "bf16", seed=4, factor=0.5, backward=True,
    note="backward pass on the headline shape, values x0.5")
WORKLOADS["bwd_causal_b2h32_n8192_d128"] = Workload(
    "bwd_causal_b2h32_n8192_d128", 2, 32, 8192, 128, "bf16", seed=9, factor=0.5, causal=True,
    backward=True, note="backward pass, causal mask")
WORKLOADS["bwd_b4h16_n2048"] = Workload(
    "bwd_b4h16_n2048", 4, 16, 2048, 64, "bf16", seed=3, backward=True, note="backward pass, d = 64")
WORKLOADS["bwd_b1h32_n8192_d128"] = Workload(
    "bwd_b1h32_n8192_d128", 1, 32, 8192, 128, "bf16", seed=6, factor=0.5, backward=True,
    note="backward profiling case: half the headline shape")
HEADLINE = "b2h32_n8192_d128"
SMALL = "single_head_n512"


def custom(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 11,
           factor: float = 1.0) -> Workload:
    return Workload(f"custom_b{B}h{H}n{N}d{d}_{dtype}", B, H, N, d, dtype, seed, factor)


def _finish(values: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 or float16 (RNE) for bf16 / f16
    workloads, in independent chunks on a thread pool."""
    flat = values.reshape(-1)
    out = np.empty(flat.shape, dtype=np.float32)
    step = 1 << 22

    def one(i0):
        x = flat[i0:i0 + step].astype(np.float32)
        if dtype == "bf16":
            x = round_to_bf16(x)
        elif dtype == "f16":
            x = x.astype(np.float16).astype(np.float32)  # round to nearest even
        out[i0:i0 + step] = x

    starts = list(range(0, flat.size, step))
    workers = max(1, min(len(starts), os.cpu_count() or 1, 32))
    if workers == 1:
        for i0 in starts:
            one(i0)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, starts))
    return out.reshape(values.shape)


def make(w: Workload):
    """Return (q, k, v) float32 arrays holding the rounded inputs: q
    [B, H, N, d], k and v [B, H_kv, Nkv, d]."""
    if w.general:
        return make_general(w.B, w.H, w.H_kv, w.N, w.Nkv, w.d, w.dtype, w.seed, w.factor)
    n = w.B * w.H * w.N * w.d
    out = []
    for t in (TENSOR_Q, TENSOR_K, TENSOR_V):
        x = normals(w.seed, t, n, w.factor).reshape(w.shape)
        if t == TENSOR_Q:
            for (b, h, f) in w.q_scaled_heads:
                x[b, h] *= f
        if t == TENSOR_K:
            for (b, h) in w.identical_k_heads:
                x[b, h, :, :] = x[b, h, 0, :]
        out.append(_finish(x, w.dtype))
    return tuple(out)


def sample_rows(w: Workload, count: int, seed_offset: int = 0) -> np.ndarray:
    """`count` seeded (b, h, i) query rows, uniform over the workload."""
    key = stream_key(w.seed + seed_offset, TENSOR_ROWS)
    u = uint64_stream(key, 0, 3 * count).reshape(count, 3)
    rows = np.empty((count, 3), dtype=np.int64)
    rows[:, 0] = (u[:, 0] % np.uint64(w.B)).astype(np.int64)
    rows[:, 1] = (u[:, 1] % np.uint64(w.H)).astype(np.int64)
    rows[:, 2] = (u[:, 2] % np.uint64(w.N)).astype(np.int64)
    return rows


def make_general(B: int, H: int, H_kv: int, Nq: int, Nkv: int, d: int, dtype: str = "bf16",
                 seed: int = 13, factor: float = 1.0):
    """Seeded q [B, H, Nq, d] and k, v [B, H_kv, Nkv, d] (grouped key/value
    heads, separate query and key lengths), rounded like make()."""
    out = []
    for t, shape in ((TENSOR_Q, (B, H, Nq, d)), (TENSOR_K, (B, H_kv, Nkv, d)),
                     (TENSOR_V, (B, H_kv, Nkv, d))):
        n = shape[0] * shape[1] * shape[2] * shape[3]
        out.append(_finish(normals(seed, t, n, factor).reshape(shape), dtype))
    return tuple(out)


def make_dout(B: int, H: int, Nq: int, d: int, dtype: str = "bf16", seed: int = 13,
              factor: float = 1.0) -> np.ndarray:
    """Seeded upstream gradient dO [B, H, Nq, d] for the backward pass, drawn
    like the inputs (its own counter stream) and rounded to the dtype."""
    n = B * H * Nq * d
    return _finish(normals(seed, TENSOR_DO, n, factor).reshape(B, H, Nq, d), dtype)
