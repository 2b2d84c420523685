"""Pins of the CPU oracle to facts it does not compute itself.

The oracle (oracle/attn_oracle.c) is the plain three-pass definition of
softmax attention.  Each pin below checks it against something independent:
a closed form, an invariant of softmax, a library routine (PyTorch's
scaled_dot_product_attention and SciPy's softmax/logsumexp on a materialised
score matrix), or a brute-force online-softmax sweep over random tile splits.
`test_pins_catch_planted_mistakes` rebuilds the oracle with deliberate
mistakes (dropped scale, transposed K, flipped exponent sign, wrong log base,
dropped last key, transposed V) and requires every one to fail some pin.

Page references: "CUDA Flash Attention: Online Softmax with Shared Memory
Tiling" (Problem Statement: softmax(QK^T/sqrt(d))V); "How Did I Write My First
FlashAttention Kernel in CUDA?" (online softmax, pseudo-algorithm steps 1-5);
"FlashAttention dissected" (softmax formula, the correction factor
e^{m_1 - m_new}, pseudocode with one final division by l).
"""
import math

import numpy as np
import pytest

import oracle
from exact_tiled_attention_04_gb300 import inputs as I

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0, rng=RNG):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


# --------------------------------------------------------------------------
# pins, written as functions of the oracle library so that the mutation test
# can run them against planted mistakes
# --------------------------------------------------------------------------

def pin_weights_sum_to_one(lib):
    """V = all ones: every output is the sum of the softmax weights, so 1."""
    for (B, H, N, d, scale) in [(1, 2, 37, 8, 0.3), (2, 1, 129, 16, 1.7), (1, 1, 5, 3, -0.9)]:
        q, k = rand(B, H, N, d), rand(B, H, N, d)
        v = np.ones((B, H, N, d), np.float32)
        o, _ = oracle.attention_f64(q, k, v, scale, lib=lib)
        assert np.max(np.abs(o - 1.0)) <= 1e-13


def pin_identical_keys(lib):
    """Every key equal: all scores in a row equal, so O is the plain mean of
    the V rows and lse = s + ln N."""
    N, d, scale = 1000, 64, 0.125
    q = rand(1, 1, N, d)
    k = np.broadcast_to(rand(1, 1, 1, d), (1, 1, N, d)).copy()
    v = rand(1, 1, N, d)
    o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
    mean_v = v[0, 0].astype(np.float64).mean(axis=0)
    assert np.max(np.abs(o[0, 0] - mean_v)) <= 1e-12
    s = scale * (q[0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))
    assert np.max(np.abs(lse[0, 0] - (s + math.log(N)))) <= 1e-12


def pin_single_key(lib):
    """N = 1: the only weight is 1, O = v_0 and lse = s_00."""
    d, scale = 16, 0.7
    q, k, v = rand(2, 3, 1, d), rand(2, 3, 1, d), rand(2, 3, 1, d)
    o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
    assert np.array_equal(o, v.astype(np.float64))
    s = scale * np.einsum("bhnd,bhnd->bhn", q.astype(np.float64), k.astype(np.float64))
    assert np.max(np.abs(lse - s)) <= 1e-13


def pin_zero_scale(lib):
    """scale = 0: all scores 0, O = mean of V, lse = ln N."""
    N, d = 77, 8
    q, k, v = rand(1, 2, N, d), rand(1, 2, N, d), rand(1, 2, N, d)
    o, lse = oracle.attention_f64(q, k, v, 0.0, lib=lib)
    assert np.max(np.abs(o - v.astype(np.float64).mean(axis=2, keepdims=True))) <= 1e-13
    assert np.max(np.abs(lse - math.log(N))) <= 1e-13


def pin_dominant_score(lib):
    """One score exceeds every other by at least Delta: O is within
    2(N-1)e^{-Delta} max|v| of that key's V row (the other weights sum to at
    most (N-1)e^{-Delta}).  The dominant key is placed first, in the middle
    and last."""
    N, d, scale = 50, 4, 1.0
    for kstar in (0, N // 2, N - 1):
        q = np.zeros((1, 1, N, d), np.float32)
        q[..., 0] = 1.0
        k = rand(1, 1, N, d, scale=0.1)
        k[0, 0, :, 0] = np.float32(0.0)
        k[0, 0, kstar, 0] = np.float32(12.0)
        v = rand(1, 1, N, d)
        o, _ = oracle.attention_f64(q, k, v, scale, lib=lib)
        delta = 12.0
        bound = 2 * (N - 1) * math.exp(-delta) * np.abs(v).max()
        err = np.abs(o[0, 0] - v[0, 0, kstar].astype(np.float64)).max()
        assert err <= bound, (kstar, err, bound)


def pin_bounds(lib):
    """max_j s_j <= lse <= max_j s_j + ln N, and each output column lies in
    [min_j v_j, max_j v_j] (a convex combination)."""
    N, d, scale = 300, 32, 0.2
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
    s = scale * (q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T)
    smax = s.max(axis=1)
    assert np.all(lse[0, 0] >= smax - 1e-12)
    assert np.all(lse[0, 0] <= smax + math.log(N) + 1e-12)
    vmin, vmax = v[0, 0].min(axis=0), v[0, 0].max(axis=0)
    assert np.all(o[0, 0] >= vmin - 1e-12) and np.all(o[0, 0] <= vmax + 1e-12)


def pin_torch_sdpa(lib):
    """PyTorch's scaled_dot_product_attention (CPU, float64) on non-square
    shapes with a scale that is not 1/sqrt(d); lse against torch.logsumexp."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    for (B, H, N, d, scale) in [(2, 3, 45, 24, 0.37), (1, 2, 130, 64, 0.125)]:
        q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
        o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
        tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=float(scale)).numpy()
        assert np.max(np.abs(o - ref)) <= 1e-12
        ref_lse = torch.logsumexp(float(scale) * tq @ tk.transpose(-1, -2), dim=-1).numpy()
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12


def pin_materialised_scipy(lib):
    """Standard (materialised) attention with SciPy: S = scale Q K^T as a
    full matrix, P = softmax(S), O = P V, lse = logsumexp(S)."""
    from scipy.special import logsumexp, softmax
    B, H, N, d, scale = 1, 2, 96, 40, 0.61
    q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    S = scale * np.matmul(q64, np.swapaxes(k64, -1, -2))
    assert np.max(np.abs(o - np.matmul(softmax(S, axis=-1), v64))) <= 1e-12
    assert np.max(np.abs(lse - logsumexp(S, axis=-1))) <= 1e-12


def online_attention(q, k, v, scale, splits, deferred, masked_prefix=0):
    """Brute-force online softmax over a given split of the keys into
    consecutive tiles, in float64.  `deferred=False` normalises after every
    tile (the per-step form of the first page's step 5); `deferred=True`
    keeps an unnormalised accumulator and divides once at the end (the
    dissected pseudocode).  The first `masked_prefix` keys get score -inf."""
    q, k, v = (x.astype(np.float64) for x in (q, k, v))
    n_rows, d = q.shape
    m = np.full(n_rows, -np.inf)
    l = np.zeros(n_rows)
    o = np.zeros((n_rows, d))
    start = 0
    for size in splits:
        kj, vj = k[start:start + size], v[start:start + size]
        s = scale * (q @ kj.T)
        s[:, :max(0, masked_prefix - start)] = -np.inf
        m_tile = s.max(axis=1)
        m_new = np.maximum(m, m_tile)
        shift = np.where(m_new == -np.inf, 0.0, m_new)   # -inf guard
        alpha = np.exp(np.where(m == -np.inf, -np.inf, m - shift))
        if deferred:
            p = np.exp(s - shift[:, None])
            l_new = alpha * l + p.sum(axis=1)
            o = alpha[:, None] * o + p @ vj
        else:
            m_tile_s = np.where(m_tile == -np.inf, 0.0, m_tile)
            p_t = np.exp(s - m_tile_s[:, None])
            l_t = p_t.sum(axis=1)
            beta = np.exp(np.where(m_tile == -np.inf, -np.inf, m_tile_s - shift))
            l_new = alpha * l + beta * l_t
            safe = np.where(l_new == 0, 1.0, l_new)
            o = ((l * alpha)[:, None] * o + beta[:, None] * (p_t @ vj)) / safe[:, None]
        m, l = m_new, l_new
        start += size
    if deferred:
        o = o / l[:, None]
    return o, m + np.log(l)


def pin_online_tile_splits(lib):
    """Online softmax over random consecutive tile splits (sizes 1..N), in both
    normalisation forms, equals the three-pass result within 1e-12."""
    rng = np.random.default_rng(99)
    for trial in range(12):
        N = int(rng.integers(1, 65))
        d = int(rng.integers(1, 9))
        scale = float(rng.uniform(0.1, 2.0))
        q, k, v = (rand(1, 1, N, d, rng=rng) for _ in range(3))
        o, lse = oracle.attention_f64(q, k, v, scale, lib=lib)
        splits, left = [], N
        while left:
            t = int(rng.integers(1, left + 1))
            splits.append(t)
            left -= t
        for deferred in (False, True):
            oo, ll = online_attention(q[0, 0], k[0, 0], v[0, 0], scale, splits, deferred)
            assert np.max(np.abs(oo - o[0, 0])) <= 1e-12, (trial, deferred)
            assert np.max(np.abs(ll - lse[0, 0])) <= 1e-12, (trial, deferred)


def pin_general_shapes_sdpa(lib):
    """Grouped key/value heads and different query / key lengths against
    PyTorch SDPA with the key/value heads repeated explicitly (query head h
    uses key/value head h // group)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    for (B, H, H_kv, Nq, Nkv, d, scale) in [(2, 6, 3, 37, 53, 24, 0.4), (1, 4, 1, 1, 130, 16, 0.25),
                                             (1, 2, 2, 70, 9, 8, 1.1)]:
        q, k, v = rand(B, H, Nq, d), rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
        o, lse = oracle.attention_f64_ex(q, k, v, scale, lib=lib)
        tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
        g = H // H_kv
        tk, tv = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=float(scale)).numpy()
        assert np.max(np.abs(o - ref)) <= 1e-12
        ref_lse = torch.logsumexp(float(scale) * tq @ tk.transpose(-1, -2), dim=-1).numpy()
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12


def pin_decode_row_materialised(lib):
    """One query against many keys (a decode step) equals the materialised
    softmax of its score row (SciPy), for every query head of a grouped layout."""
    from scipy.special import logsumexp, softmax
    B, H, H_kv, Nkv, d, scale = 2, 8, 2, 300, 32, 0.17
    q, k, v = rand(B, H, 1, d), rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
    o, lse = oracle.attention_f64_ex(q, k, v, scale, lib=lib)
    for b in range(B):
        for h in range(H):
            kk = k[b, h // (H // H_kv)].astype(np.float64)
            vv = v[b, h // (H // H_kv)].astype(np.float64)
            srow = scale * (kk @ q[b, h, 0].astype(np.float64))
            assert np.max(np.abs(o[b, h, 0] - softmax(srow) @ vv)) <= 1e-12
            assert abs(lse[b, h, 0] - logsumexp(srow)) <= 1e-12


def pin_causal_sdpa(lib):
    """Causal attention against PyTorch SDPA with an explicit boolean mask
    built independently (key j visible to query i iff j <= i + Nkv - Nq),
    with query and key lengths equal and different, and grouped heads."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    for (B, H, H_kv, Nq, Nkv, d, scale) in [(1, 2, 2, 40, 40, 16, 0.3), (2, 4, 2, 17, 60, 8, 0.7),
                                             (1, 2, 1, 1, 33, 8, 0.5)]:
        q, k, v = rand(B, H, Nq, d), rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
        o, lse = oracle.attention_f64_ex(q, k, v, scale, lib=lib, causal=True)
        tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
        g = H // H_kv
        tk, tv = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
        mask = torch.ones(Nq, Nkv, dtype=torch.bool).tril(diagonal=Nkv - Nq)
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=float(scale)).numpy()
        assert np.max(np.abs(o - ref)) <= 1e-12
        sc = (float(scale) * tq @ tk.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
        assert np.max(np.abs(lse - torch.logsumexp(sc, dim=-1).numpy())) <= 1e-12


def pin_causal_first_row_and_full_row(lib):
    """Square causal attention: the first query sees only key 0 (O = v_0,
    lse = s_00); the last query sees every key (equals the unmasked row)."""
    N, d, scale = 50, 8, 0.6
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    oc, lc = oracle.attention_f64_ex(q, k, v, scale, lib=lib, causal=True)
    of, lf = oracle.attention_f64_ex(q, k, v, scale, lib=lib, causal=False)
    assert np.array_equal(oc[0, 0, 0], v[0, 0, 0].astype(np.float64))
    assert abs(lc[0, 0, 0] - scale * float(q[0, 0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))) <= 1e-13
    assert np.max(np.abs(oc[0, 0, -1] - of[0, 0, -1])) == 0.0 and lc[0, 0, -1] == lf[0, 0, -1]


ALL_PINS = [pin_weights_sum_to_one, pin_identical_keys, pin_single_key, pin_zero_scale,
            pin_dominant_score, pin_bounds, pin_torch_sdpa, pin_materialised_scipy,
            pin_online_tile_splits, pin_general_shapes_sdpa, pin_decode_row_materialised,
            pin_causal_sdpa, pin_causal_first_row_and_full_row]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_masked_prefix_is_excluded(oracle_lib):
    """A fully masked leading tile (scores -inf) contributes nothing: the
    online sweep with the guard equals the oracle on the unmasked keys."""
    N, d, scale, masked = 40, 6, 0.5, 16
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    kk = np.ascontiguousarray(k[:, :, masked:])
    vv = np.ascontiguousarray(v[:, :, masked:])
    # the oracle takes equal query and key counts: evaluate one query row at
    # a time against the N - masked unmasked keys
    ref_o, ref_l = [], []
    for i in range(N):
        qi = np.broadcast_to(q[:, :, i:i + 1], (1, 1, N - masked, d)).copy()
        oi, li = oracle.attention_f64(qi, kk, vv, scale, rows=[(0, 0, 0)])
        ref_o.append(oi[0])
        ref_l.append(li[0])
    for deferred in (False, True):
        oo, ll = online_attention(q[0, 0], k[0, 0], v[0, 0], scale, [16, 10, 14], deferred, masked)
        assert np.max(np.abs(oo - np.array(ref_o))) <= 1e-12
        assert np.max(np.abs(ll - np.array(ref_l))) <= 1e-12


def test_row_subset_matches_full(oracle_lib):
    B, H, N, d = 2, 3, 33, 8
    q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    o, lse = oracle.attention_f64(q, k, v, 0.4)
    rows = [(1, 2, 32), (0, 0, 0), (1, 0, 5)]
    o2, l2 = oracle.attention_f64(q, k, v, 0.4, rows=rows)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(o2[r], o[b, h, i]) and l2[r] == lse[b, h, i]


def test_thread_count_does_not_change_bits(oracle_lib):
    q, k, v = rand(1, 4, 64, 16), rand(1, 4, 64, 16), rand(1, 4, 64, 16)
    a = oracle.attention_f64(q, k, v, 0.25, threads=1)
    b = oracle.attention_f64(q, k, v, 0.25, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_arguments_rejected(oracle_lib):
    q = rand(1, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.attention_f64(q, q, q, 1.0, rows=[(0, 0, 4)])
    with pytest.raises(ValueError):
        oracle.attention_f64(q, q, q[:, :, :3], 1.0)
    with pytest.raises(ValueError):  # 3 query heads cannot share 2 key/value heads
        oracle.attention_f64_ex(rand(1, 3, 4, 4), rand(1, 2, 5, 4), rand(1, 2, 5, 4), 1.0)


def test_nan_input_propagates(oracle_lib):
    q, k, v = rand(1, 1, 8, 4), rand(1, 1, 8, 4), rand(1, 1, 8, 4)
    k[0, 0, 3, 1] = np.nan
    o, lse = oracle.attention_f64(q, k, v, 0.5)
    assert np.isnan(o).all() and np.isnan(lse).all()


def test_tail_workload_special_heads(oracle_lib):
    """The 1000-row workload's special heads: identical keys give the plain
    mean of V over exactly 1000 rows; the Q x30 head is nearly one-hot and
    within the dominant-score bound row by row."""
    w = I.WORKLOADS["tail_n1000"]
    q, k, v = I.make(w)
    o, lse = oracle.attention_f64(q[0:1, 1:2], k[0:1, 1:2], v[0:1, 1:2], float(w.scale))
    assert np.max(np.abs(o[0, 0] - v[0, 1].astype(np.float64).mean(axis=0))) <= 1e-12
    o, _ = oracle.attention_f64(q[1:2, 2:3], k[1:2, 2:3], v[1:2, 2:3], float(w.scale))
    q64, k64, v64 = (x[1, 2].astype(np.float64) for x in (q, k, v))
    s = float(w.scale) * (q64 @ k64.T)
    top2 = np.sort(s, axis=1)[:, -2:]
    delta = top2[:, 1] - top2[:, 0]
    kstar = s.argmax(axis=1)
    bound = 2 * (w.N - 1) * np.exp(-delta) * np.abs(v64).max()
    err = np.abs(o[0, 0] - v64[kstar]).max(axis=1)
    assert np.all(err <= bound + 1e-12)
    assert np.median(delta) > 3.0  # top-2 score gap: the head really is peaked


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_pins_catch_planted_mistakes(mutant, tmp_path):
    """Rebuild the oracle with one planted mistake; some pin must fail."""
    path = oracle.build(out_dir=str(tmp_path), mutant=mutant)
    lib = oracle._bind(path)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


def test_causal_query_without_visible_key(oracle_lib):
    """More queries than keys: the first Nq - Nkv queries see no key."""
    q, k, v = rand(1, 1, 10, 4), rand(1, 1, 6, 4), rand(1, 1, 6, 4)
    o, lse = oracle.attention_f64_ex(q, k, v, 0.5, causal=True)
    assert np.all(o[0, 0, :4] == 0.0) and np.all(np.isneginf(lse[0, 0, :4]))
    assert np.all(np.isfinite(lse[0, 0, 4:]))
