"""The decode kernel (at most 32 query rows per key/value head: N_q x group
<= 32, 16-bit inputs) against the fp64 oracle on every output row: 16- and
32-row variants, head dimensions 64 and 128, bf16 and fp16, causal masks
(including rows that see no key), partitions that hold no visible key,
scores that keep growing along the sequence (a rescale in a late tile), and
key counts that are not a multiple of the 128-key tile."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_LSE, compare_ex, ensure_library, run_fa_ex, tol_o_dtype

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def check(dtype, q, k, v, splits, causal=False):
    o, lse = run_fa_ex(q, k, v, dtype, splits, causal=causal)
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v, causal=causal)
    assert err_o <= tol_o_dtype(dtype), (q.shape, k.shape, splits, causal, err_o)
    assert err_l <= TOL_LSE, (q.shape, k.shape, splits, causal, err_l)
    return o, lse


# (Nq, group): rows per key/value head 1, 4, 15, 16 (16-row variant) and
# 17, 24, 32 (32-row variant)
ROWS = [(1, 1), (1, 4), (3, 5), (2, 8), (17, 1), (3, 8), (4, 8)]


@pytest.mark.parametrize("Nq,G", ROWS)
@pytest.mark.parametrize("d", [64, 128])
def test_rows_and_head_dims(Nq, G, d):
    q, k, v = I.make_general(2, 2 * G, 2, Nq, 1000, d, "bf16", seed=900 + 10 * Nq + G + d)
    check("bf16", q, k, v, 1)
    check("bf16", q, k, v, 3)


@pytest.mark.parametrize("Nkv", [1, 100, 128, 129, 4096])
def test_key_counts(Nkv):
    q, k, v = I.make_general(1, 8, 2, 1, Nkv, 128, "bf16", seed=920 + Nkv)
    check("bf16", q, k, v, 1)
    check("bf16", q, k, v, 4)


@pytest.mark.parametrize("d", [64, 128])
def test_fp16(d):
    q, k, v = I.make_general(2, 16, 4, 2, 777, d, "f16", seed=930 + d)
    check("f16", q, k, v, 1)
    check("f16", q, k, v, 2)


@pytest.mark.parametrize("Nq,G,Nkv", [(4, 4, 700), (1, 8, 300), (8, 4, 5), (32, 1, 20), (16, 2, 1000)])
@pytest.mark.parametrize("splits", [1, 3])
def test_causal(Nq, G, Nkv, splits):
    """Causal rows see keys up to i + N_kv - N_q; with N_q > N_kv the first
    rows see none (O = 0, lse = -inf), and with splits some partitions hold
    no visible key."""
    q, k, v = I.make_general(1, 2 * G, 2, Nq, Nkv, 64, "bf16", seed=940 + Nq + G + Nkv)
    check("bf16", q, k, v, splits, causal=True)


@pytest.mark.parametrize("splits", [1, 2])
def test_late_rescale(splits):
    """Keys whose scale grows along the sequence: the tile maxima keep
    rising, so the shared reference maxima move in late tiles and O^T, l
    and lq are rescaled there."""
    q, k, v = I.make_general(2, 8, 2, 1, 3000, 128, "bf16", seed=950)
    ramp = np.linspace(0.2, 3.0, k.shape[2], dtype=np.float32)[None, None, :, None]
    k = I.round_to_bf16((k * ramp).astype(np.float32))  # both sides see the same bf16 keys
    check("bf16", q, k, v, splits)


def test_matches_grouped_tile_path_closely():
    """33 rows per key/value head take the general packed kernel, 32 the
    decode kernel: on the same inputs the shared rows agree to within the
    rounding of the output."""
    q, k, v = I.make_general(1, 33, 1, 1, 2000, 128, "bf16", seed=960)
    o33, l33 = run_fa_ex(q, k, v, "bf16", 1)
    o32, l32 = run_fa_ex(q[:, :32], k, v, "bf16", 1)
    assert np.max(np.abs(o33[:, :32] - o32)) <= 2 ** -7
    assert np.max(np.abs(l33[:, :32] - l32)) <= 1e-4


@pytest.mark.parametrize("splits", [1, 2])
def test_fp16_causal_32_rows(splits):
    """fp16, causal, the 32-row variant at d = 128 (four queries of eight
    query heads per key/value head)."""
    q, k, v = I.make_general(1, 16, 2, 4, 500, 128, "f16", seed=970 + splits)
    check("f16", q, k, v, splits, causal=True)
