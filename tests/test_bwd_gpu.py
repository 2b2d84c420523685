"""fa_bwd on the GPU against the fp64 backward oracle.

Small problems are compared element by element with the full oracle
gradients (several query tiles and key blocks with ragged tails, both input
dtypes, both head dimensions, causal masks, grouped key/value heads, more
queries than keys).  The full-size case (B=2, H=32, N=8192, d=128 bf16, the
forward headline shapes) is checked on sampled dQ rows and sampled dK / dV
keys the oracle evaluates one by one, and on the gradient-sum invariants of
every head.  The forward outputs o and lse the backward consumes come from
the GPU forward pass; every expected value comes from the oracle alone.
"""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import ensure_library, grad_errors, run_bwd, tol_grad

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def check(B, H, H_kv, Nq, Nkv, d, dtype, causal, seed, factor=1.0):
    q, k, v = I.make_general(B, H, H_kv, Nq, Nkv, d, dtype, seed=seed, factor=factor)
    dout = I.make_dout(B, H, Nq, d, dtype, seed=seed)
    got, sc = run_bwd(q, k, v, dout, dtype, causal=causal)
    ref = oracle.attention_bwd_f64(q, k, v, dout, sc, causal=causal)
    errs = grad_errors(got, ref)
    print(f"B{B} H{H}/{H_kv} Nq{Nq} Nkv{Nkv} d{d} {dtype} causal={causal}: "
          f"dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    for name, e in zip(("dq", "dk", "dv"), errs):
        assert e <= tol_grad(dtype), (name, e)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_tiles(d, dtype, causal):
    check(1, 2, 2, 300, 333, d, dtype, causal, seed=600 + d)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads(causal):
    check(2, 8, 2, 200, 260, 64, "bf16", causal, seed=610)
    check(1, 6, 1, 130, 129, 128, "bf16", causal, seed=611)


def test_exact_tiles():
    check(2, 2, 2, 256, 256, 128, "bf16", False, seed=620, factor=0.5)
    check(1, 3, 3, 128, 128, 64, "f16", True, seed=621)


def test_more_queries_than_keys_causal():
    """Queries i < Nq - Nkv see no key: their dQ is 0 and they add nothing."""
    check(1, 2, 2, 260, 100, 64, "bf16", True, seed=630)


def test_short_queries():
    check(2, 4, 2, 1, 500, 128, "bf16", False, seed=640)
    check(1, 4, 4, 7, 900, 64, "f16", True, seed=641)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_multi_head_sweep_d128(dtype):
    """d = 128 without the causal mask (the kernel with the dQ read-out
    warpgroup): two query heads per key/value head, four query tiles each
    with a ragged last one, so one CTA sweeps eight tiles through its
    two-stage ring, changes query head half way, and stages and reduces dQ
    of partial tiles."""
    check(1, 4, 2, 390, 256, 128, dtype, False, seed=660)


def test_long_keys_one_head():
    check(1, 1, 1, 64, 2000, 128, "bf16", False, seed=650)


def test_full_size_sampled():
    """B=2, H=32, N=8192, d=128 bf16 (inputs x0.5): sampled dQ rows and
    dK / dV keys against the oracle, invariants over every head."""
    B, H, N, d = 2, 32, 8192, 128
    q, k, v = I.make_general(B, H, H, N, N, d, "bf16", seed=4, factor=0.5)
    dout = I.make_dout(B, H, N, d, "bf16", seed=4)
    (dq, dk, dv), sc = run_bwd(q, k, v, dout, "bf16")
    rng = np.random.default_rng(7)
    rows = np.stack([rng.integers(0, B, 24), rng.integers(0, H, 24), rng.integers(0, N, 24)], axis=1)
    rows[:4] = [(0, 0, 0), (1, 31, N - 1), (0, 5, 127), (1, 17, 128)]
    ref_dq = oracle.attention_bwd_dq_rows_f64(q, k, v, dout, sc, rows)
    got_dq = dq[rows[:, 0], rows[:, 1], rows[:, 2]]
    e_dq = np.max(np.abs(got_dq - ref_dq)) / np.max(np.abs(ref_dq))
    cols = np.array([(1, 9, j) for j in (0, 1, 127, 128, 4095, 8190, 8191)] + [(0, 0, 77), (0, 0, 5000)])
    ref_dk, ref_dv = oracle.attention_bwd_dkv_cols_f64(q, k, v, dout, sc, cols)
    got_dk = dk[cols[:, 0], cols[:, 1], cols[:, 2]]
    got_dv = dv[cols[:, 0], cols[:, 1], cols[:, 2]]
    e_dk = np.max(np.abs(got_dk - ref_dk)) / np.max(np.abs(ref_dk))
    e_dv = np.max(np.abs(got_dv - ref_dv)) / np.max(np.abs(ref_dv))
    print(f"full size sampled: dq {e_dq:.2e} dk {e_dk:.2e} dv {e_dv:.2e}")
    assert e_dq <= tol_grad("bf16") and e_dk <= tol_grad("bf16") and e_dv <= tol_grad("bf16")
    # invariants of every head: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    dk_sum = dk.astype(np.float64).sum(axis=2)
    dv_sum = dv.astype(np.float64).sum(axis=2)
    do_sum = dout.astype(np.float64).sum(axis=2)
    # each sum adds N outputs with relative rounding 2^-9: bound by the sum
    # of magnitudes, not by the (near-zero) result
    dk_mag = np.abs(dk.astype(np.float64)).sum(axis=2)
    dv_mag = np.abs(dv.astype(np.float64)).sum(axis=2)
    assert np.all(np.abs(dk_sum) <= 4e-3 * dk_mag + 1e-6)
    assert np.all(np.abs(dv_sum - do_sum) <= 4e-3 * dv_mag + 1e-6)
