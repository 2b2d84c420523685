"""Extreme sizes against the oracle on sampled outputs: very long sequences
(forward N = 131072, backward N = 16384), tensors past 2 GiB (the forward's
query and output, the backward's dQ accumulator), very many short heads
(4096 heads of 64 rows: one ragged tile each), and a decode step against a
262144-key cache with one key/value head for eight query heads (MQA)."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import (TOL_LSE, compare_ex, ensure_library, grad_errors, run_bwd, run_fa_ex, tol_grad,
                       tol_o_dtype)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def sample_rows(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, B, n), rng.integers(0, H, n), rng.integers(0, N, n)], axis=1)
    rows[:3] = [(0, 0, 0), (B - 1, H - 1, N - 1), (0, H - 1, N // 2)]
    return rows


@pytest.mark.parametrize("N,d", [(131072, 64), (65536, 128)])
def test_forward_long_sequence(N, d):
    q, k, v = I.make_general(1, 1, 1, N, N, d, "bf16", seed=800 + d)
    for causal in (False, True):
        o, lse = run_fa_ex(q, k, v, "bf16", 1, causal=causal)
        rows = sample_rows(1, 1, N, 12, 801)
        err_o, err_l = compare_ex("bf16", o, lse, q, k, v, rows=rows, causal=causal)
        assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (causal, err_o, err_l)


def test_forward_query_tensor_over_2_gib():
    """q and o of 264 x 32768 x 128 bf16 elements (2.2 GB each, byte offsets
    past 2^31) against one key/value head, in the automatic plan (which
    splits the last 48 of 33792 query blocks): rows at the far end of the
    tensors match the oracle."""
    B, H, H_kv, N, d = 1, 264, 1, 32768, 128
    q, k, v = I.make_general(B, H, H_kv, N, N, d, "bf16", seed=850, factor=0.5)
    o, lse = run_fa_ex(q, k, v, "bf16", 0)
    rows = sample_rows(B, H, N, 12, 851)
    rows = np.concatenate([rows, np.array([(0, H - 1, N - 2), (0, H - 2, N - 1), (0, H - 9, 0)])])
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v, rows=rows)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (err_o, err_l)
    assert np.isfinite(o[0, -48:]).all() and np.isfinite(lse[0, -48:]).all()


def test_forward_many_short_heads():
    q, k, v = I.make_general(64, 64, 64, 64, 64, 64, "bf16", seed=810)
    o, lse = run_fa_ex(q, k, v, "bf16", 1)
    rows = sample_rows(64, 64, 64, 64, 811)
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v, rows=rows)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE


def test_decode_long_cache_mqa():
    B, H, H_kv, Nkv, d = 2, 8, 1, 262144, 128
    q, k, v = I.make_general(B, H, H_kv, 1, Nkv, d, "bf16", seed=820)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits = fab.fa_fwd_ex_splits(B, H, H_kv, 1, Nkv, sms)
    o, lse = run_fa_ex(q, k, v, "bf16", splits)
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (splits, err_o, err_l)


def test_backward_long_sequence():
    B, H, N, d = 1, 1, 16384, 128
    q, k, v = I.make_general(B, H, H, N, N, d, "bf16", seed=830, factor=0.5)
    dout = I.make_dout(B, H, N, d, "bf16", seed=830)
    (dq, dk, dv), sc = run_bwd(q, k, v, dout, "bf16")
    rows = sample_rows(B, H, N, 8, 831)
    ref_dq = oracle.attention_bwd_dq_rows_f64(q, k, v, dout, sc, rows)
    e_dq = np.max(np.abs(dq[rows[:, 0], rows[:, 1], rows[:, 2]] - ref_dq)) / np.max(np.abs(ref_dq))
    cols = np.array([(0, 0, 0), (0, 0, 8191), (0, 0, N - 1)])
    ref_dk, ref_dv = oracle.attention_bwd_dkv_cols_f64(q, k, v, dout, sc, cols)
    got = [g[cols[:, 0], cols[:, 1], cols[:, 2]] for g in (dk, dv)]
    e_dk = np.max(np.abs(got[0] - ref_dk)) / np.max(np.abs(ref_dk))
    e_dv = np.max(np.abs(got[1] - ref_dv)) / np.max(np.abs(ref_dv))
    assert max(e_dq, e_dk, e_dv) <= tol_grad("bf16"), (e_dq, e_dk, e_dv)


def test_backward_accumulator_over_2_gib():
    """136 heads x 32768 rows x d = 128: q, dO and the gradients are 1.1 GB
    each and dQ's fp32 accumulator 2.3 GB (byte offsets past 2^31); dq rows
    at the far end and dK, dV of two keys of the last head match the oracle."""
    B, H, N, d = 1, 136, 32768, 128
    q, k, v = I.make_general(B, H, H, N, N, d, "bf16", seed=860, factor=0.5)
    dout = I.make_dout(B, H, N, d, "bf16", seed=860)
    (dq, dk, dv), sc = run_bwd(q, k, v, dout, "bf16")
    rows = np.concatenate([sample_rows(B, H, N, 6, 861),
                           np.array([(0, H - 1, N - 1), (0, H - 1, N - 2), (0, H - 2, 0)])])
    ref_dq = oracle.attention_bwd_dq_rows_f64(q, k, v, dout, sc, rows)
    e_dq = np.max(np.abs(dq[rows[:, 0], rows[:, 1], rows[:, 2]] - ref_dq)) / np.max(np.abs(ref_dq))
    cols = np.array([(0, H - 1, N - 1), (0, H - 1, 5)])
    ref_dk, ref_dv = oracle.attention_bwd_dkv_cols_f64(q, k, v, dout, sc, cols)
    got = [g[cols[:, 0], cols[:, 1], cols[:, 2]] for g in (dk, dv)]
    e_dk = np.max(np.abs(got[0] - ref_dk)) / np.max(np.abs(ref_dk))
    e_dv = np.max(np.abs(got[1] - ref_dv)) / np.max(np.abs(ref_dv))
    assert max(e_dq, e_dk, e_dv) <= tol_grad("bf16"), (e_dq, e_dk, e_dv)
    assert np.isfinite(dq[0, -2:]).all() and np.isfinite(dk[0, -2:]).all() and np.isfinite(dv[0, -2:]).all()


def test_backward_many_short_heads():
    q, k, v = I.make_general(16, 64, 16, 64, 100, 64, "bf16", seed=840)
    dout = I.make_dout(16, 64, 64, 64, "bf16", seed=840)
    got, sc = run_bwd(q, k, v, dout, "bf16", causal=True)
    errs = grad_errors(got, oracle.attention_bwd_f64(q, k, v, dout, sc, causal=True))
    assert max(errs) <= tol_grad("bf16"), errs


def test_causal_forward_item_order_groups():
    """Causal forward blocks are launched heaviest first within groups of
    heads (8 heads of 16 blocks each here, then a partial group of 3): every
    output row is written (the outputs start as NaN) and sampled rows of
    every head match the oracle."""
    B, H, N, d = 1, 11, 4096, 64
    q, k, v = I.make_general(B, H, H, N, N, d, "bf16", seed=850)
    o, lse = run_fa_ex(q, k, v, "bf16", 1, causal=True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(851)
    rows = np.array([(0, h, i) for h in range(H) for i in (0, 255, 256, N - 1, int(rng.integers(0, N)))])
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v, rows=rows, causal=True)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (err_o, err_l)


def test_causal_backward_item_order_groups():
    """Causal backward key blocks are launched heaviest first within groups
    of key/value heads (8 heads of 32 blocks, then 3; two query heads per
    key/value head): every gradient is written (they start as NaN) and
    sampled dQ rows and dK, dV columns of every head match the oracle."""
    B, H, H_kv, N, d = 1, 22, 11, 4096, 64
    q, k, v = I.make_general(B, H, H_kv, N, N, d, "bf16", seed=860, factor=0.5)
    dout = I.make_dout(B, H, N, d, "bf16", seed=860)
    (dq, dk, dv), sc = run_bwd(q, k, v, dout, "bf16", causal=True)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    rows = np.array([(0, h, i) for h in range(0, H, 3) for i in (5, 2100, N - 1)])
    ref_dq = oracle.attention_bwd_dq_rows_f64(q, k, v, dout, sc, rows, causal=True)
    e_dq = np.max(np.abs(dq[rows[:, 0], rows[:, 1], rows[:, 2]] - ref_dq)) / np.max(np.abs(ref_dq))
    cols = np.array([(0, h, j) for h in range(H_kv) for j in (0, 3000)])
    ref_dk, ref_dv = oracle.attention_bwd_dkv_cols_f64(q, k, v, dout, sc, cols, causal=True)
    got = [gr[cols[:, 0], cols[:, 1], cols[:, 2]] for gr in (dk, dv)]
    e_dk = np.max(np.abs(got[0] - ref_dk)) / np.max(np.abs(ref_dk))
    e_dv = np.max(np.abs(got[1] - ref_dv)) / np.max(np.abs(ref_dv))
    assert max(e_dq, e_dk, e_dv) <= tol_grad("bf16"), (e_dq, e_dk, e_dv)
