"""Pins of the backward-pass oracle (oracle/attn_bwd_oracle.c) to facts it
does not compute itself.

The pages say the backward pass recomputes the attention blocks from Q, K, V
and the saved softmax statistics ("FlashAttention dissected", section
"Memory complexity: from O(N^2) to O(N)"); what it must produce is the exact
gradient of the forward definition.  So the pins are:

- central finite differences of the FORWARD oracle (an independent program:
  it never forms dS, D or any gradient), on tiny grouped-head and causal
  problems, every input coordinate;
- automatic differentiation by PyTorch in float64 on a materialised score
  matrix (a different derivation of the same gradient);
- closed forms (zero scale, a single key, constant value rows) and the
  softmax-gradient invariants: each row of dS sums to zero, so the dK rows of
  a head sum to zero, and each row of P sums to one, so the dV rows of a
  key/value head sum to the dO rows that see any key.

`test_pins_catch_planted_mistakes` rebuilds the oracle with each planted
mistake (the -D term dropped, dK or dQ without the scale, dV weighted by dP,
K transposed in dQ, the causal mask forgotten) and requires a pin to fail.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(4321)


def rand(*shape, scale=1.0, rng=RNG):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def loss(lib, q, k, v, dout, scale, causal):
    """L = sum(O * dO), evaluated by the forward oracle in fp64."""
    o, _ = oracle.attention_f64_ex(q, k, v, scale, lib=lib, causal=causal)
    return float(np.sum(o * dout.astype(np.float64)))


def finite_difference(lib, arrays, which, scale, causal, eps=2.0 ** -10):
    """dL/dx for every coordinate of arrays[which] by central differences of
    the forward oracle.  The perturbed values are fp32 numbers; the quotient
    divides by their exact difference."""
    base = arrays[which]
    grad = np.zeros(base.shape, dtype=np.float64)
    for idx in np.ndindex(base.shape):
        x = base[idx]
        hi, lo = np.float32(x + eps), np.float32(x - eps)
        vals = []
        for val in (hi, lo):
            pert = [a.copy() for a in arrays]
            pert[which][idx] = val
            vals.append(loss(lib, pert[0], pert[1], pert[2], pert[3], scale, causal))
        grad[idx] = (vals[0] - vals[1]) / (float(hi) - float(lo))
    return grad


def pin_finite_differences(lib):
    """Every coordinate of dQ, dK, dV against central differences of the
    forward oracle: grouped heads (4 query heads on 2 key/value heads),
    Nq != Nkv, with and without the causal mask."""
    for causal in (False, True):
        q, dout = rand(1, 4, 4, 3), rand(1, 4, 4, 3)
        k, v = rand(1, 2, 6, 3), rand(1, 2, 6, 3)
        scale = 0.7
        dq, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, scale, causal=causal, lib=lib)
        arrays = [q, k, v, dout]
        for which, g in ((0, dq), (1, dk), (2, dv)):
            fd = finite_difference(lib, arrays, which, scale, causal)
            assert np.max(np.abs(fd - g)) <= 1e-5 * max(1.0, np.max(np.abs(g))), (causal, which)


def pin_torch_autograd(lib):
    """dQ, dK, dV against torch.autograd through a materialised fp64
    softmax(scale Q K^T) V with grouped heads and the causal mask."""
    torch = pytest.importorskip("torch")
    B, H, H_kv, Nq, Nkv, d, scale = 2, 4, 2, 9, 13, 8, 0.45
    for causal in (False, True):
        q, dout = rand(B, H, Nq, d), rand(B, H, Nq, d)
        k, v = rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        kk = tk.repeat_interleave(H // H_kv, dim=1)
        vv = tv.repeat_interleave(H // H_kv, dim=1)
        s = scale * tq @ kk.transpose(-1, -2)
        if causal:
            i = torch.arange(Nq).view(-1, 1)
            j = torch.arange(Nkv).view(1, -1)
            s = s.masked_fill(j > i + (Nkv - Nq), float("-inf"))
        o = torch.softmax(s, dim=-1) @ vv
        o.backward(torch.tensor(dout, dtype=torch.float64))
        dq, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, scale, causal=causal, lib=lib)
        for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-12 * max(1.0, float(ref.abs().max()))


def pin_zero_scale(lib):
    """scale = 0: every weight is 1/Nkv, so dQ = dK = 0 and every dV row is
    sum_i dO_i / Nkv over all query rows of the key/value head."""
    q, dout = rand(1, 2, 5, 4), rand(1, 2, 5, 4)
    k, v = rand(1, 1, 7, 4), rand(1, 1, 7, 4)
    dq, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, 0.0, lib=lib)
    assert np.max(np.abs(dq)) == 0.0 and np.max(np.abs(dk)) == 0.0
    want = dout.astype(np.float64).sum(axis=(1, 2)) / 7.0  # both query heads share the kv head
    assert np.max(np.abs(dv[0, 0] - want[0])) <= 1e-14


def pin_single_key(lib):
    """One key: P = 1 for every query, so dS = 0 (dQ = dK = 0) and dV_0 is
    the sum of all dO rows of its query heads."""
    q, dout = rand(1, 3, 6, 5), rand(1, 3, 6, 5)
    k, v = rand(1, 1, 1, 5), rand(1, 1, 1, 5)
    dq, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, 1.3, lib=lib)
    assert np.max(np.abs(dq)) <= 1e-15 and np.max(np.abs(dk)) <= 1e-15
    assert np.max(np.abs(dv[0, 0, 0] - dout.astype(np.float64).sum(axis=(0, 1, 2)))) <= 1e-13


def pin_constant_values(lib):
    """Equal value rows: O = v for any Q and K, so dQ = dK = 0."""
    q, dout = rand(2, 2, 8, 4), rand(2, 2, 8, 4)
    k = rand(2, 2, 11, 4)
    v = np.broadcast_to(rand(1, 1, 1, 4), (2, 2, 11, 4)).copy()
    for causal in (False, True):
        dq, dk, _ = oracle.attention_bwd_f64(q, k, v, dout, 0.9, causal=causal, lib=lib)
        assert np.max(np.abs(dq)) <= 1e-12 and np.max(np.abs(dk)) <= 1e-12


def pin_gradient_sums(lib):
    """Rows of dS sum to zero (sum_j P_ij (dP_ij - D_i) = D_i - D_i), so the
    dK rows of every key/value head sum to zero; rows of P sum to one, so
    the dV rows sum to the dO rows of the queries that see a key."""
    B, H, H_kv, Nq, Nkv, d = 2, 6, 3, 10, 7, 5
    for causal in (False, True):
        q, dout = rand(B, H, Nq, d), rand(B, H, Nq, d)
        k, v = rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
        _, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, 0.8, causal=causal, lib=lib)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
        sees = np.arange(Nq) + (Nkv - Nq) >= 0 if causal else np.ones(Nq, bool)
        want = dout.astype(np.float64)[:, :, sees].reshape(B, H_kv, -1, d).sum(axis=2)
        assert np.max(np.abs(dv.sum(axis=2) - want)) <= 1e-12


ALL_PINS = [pin_finite_differences, pin_torch_autograd, pin_zero_scale, pin_single_key,
            pin_constant_values, pin_gradient_sums]


@pytest.fixture(scope="module")
def oracle_lib():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("mutant", [11, 12, 13, 14, 15, 16])
def test_pins_catch_planted_mistakes(mutant, tmp_path):
    """Rebuild the oracle with one planted mistake; some pin must fail."""
    lib = oracle._bind(oracle.build(out_dir=str(tmp_path), mutant=mutant))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


def test_samplers_match_full_backward(oracle_lib):
    """The row (dQ) and key (dK, dV) samplers give the full backward's
    values, grouped heads and causal included."""
    B, H, H_kv, Nq, Nkv, d, scale = 2, 4, 2, 12, 17, 6, 0.5
    q, dout = rand(B, H, Nq, d), rand(B, H, Nq, d)
    k, v = rand(B, H_kv, Nkv, d), rand(B, H_kv, Nkv, d)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd_f64(q, k, v, dout, scale, causal=causal)
        rows = np.array([(1, 3, 0), (0, 0, 11), (1, 2, 5)])
        got = oracle.attention_bwd_dq_rows_f64(q, k, v, dout, scale, rows, causal=causal)
        assert np.max(np.abs(got - dq[rows[:, 0], rows[:, 1], rows[:, 2]])) <= 1e-14
        cols = np.array([(1, 1, 16), (0, 0, 0), (1, 1, 3), (0, 1, 9)])
        gk, gv = oracle.attention_bwd_dkv_cols_f64(q, k, v, dout, scale, cols, causal=causal, threads=3)
        assert np.max(np.abs(gk - dk[cols[:, 0], cols[:, 1], cols[:, 2]])) <= 1e-13
        assert np.max(np.abs(gv - dv[cols[:, 0], cols[:, 1], cols[:, 2]])) <= 1e-13


def test_thread_count_does_not_change_bits(oracle_lib):
    q, dout = rand(2, 4, 9, 4), rand(2, 4, 9, 4)
    k, v = rand(2, 2, 9, 4), rand(2, 2, 9, 4)
    a = oracle.attention_bwd_f64(q, k, v, dout, 0.5, threads=1)
    b = oracle.attention_bwd_f64(q, k, v, dout, 0.5, threads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bad_arguments_rejected(oracle_lib):
    q, k = rand(1, 3, 4, 4), rand(1, 2, 4, 4)  # 3 query heads on 2 kv heads
    with pytest.raises(ValueError):
        oracle.attention_bwd_f64(q, k, k, q, 0.5)
    q, k = rand(1, 2, 4, 4), rand(1, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.attention_bwd_dq_rows_f64(q, k, k, q, 0.5, [(0, 2, 0)])
    with pytest.raises(ValueError):
        oracle.attention_bwd_dkv_cols_f64(q, k, k, q, 0.5, [(0, 0, 4)])
