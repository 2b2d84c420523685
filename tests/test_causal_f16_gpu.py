"""fp16 inputs and causal masking on the GPU against the fp64 oracle.

Causal: query i sees keys j <= i + (N_kv - N_q); a query with no visible key
gets O = 0 and lse = -inf (both sides).  Tolerances as the other parity
tests; fp16 O: 4e-3 (derivation in tests/gpu_util.py)."""
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


def check(dtype, q, k, v, splits=1, causal=False):
    o, lse = run_fa_ex(q, k, v, dtype, splits, causal=causal)
    assert np.isfinite(o).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v, causal=causal)
    assert err_o <= tol_o_dtype(dtype), (q.shape, k.shape, splits, causal, err_o)
    assert err_l <= TOL_LSE, (q.shape, k.shape, splits, causal, err_l)
    return o, lse


@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_f16_square(N, d):
    q, k, v = I.make_general(1, 2, 2, N, N, d, "f16", seed=400 + N)
    check("f16", q, k, v)


def test_f16_split_gqa_decode():
    q, k, v = I.make_general(2, 8, 2, 1, 5000, 128, "f16", seed=410)
    check("f16", q, k, v, splits=8)
    q, k, v = I.make_general(1, 4, 2, 600, 900, 64, "f16", seed=411)
    check("f16", q, k, v, splits=3)


@pytest.mark.parametrize("N", [1, 127, 129, 300, 1000, 2048])
@pytest.mark.parametrize("d", [64, 128])
def test_causal_square_bf16(N, d):
    q, k, v = I.make_general(1, 2, 2, N, N, d, "bf16", seed=420 + N)
    o, _ = check("bf16", q, k, v, causal=True)
    # the first query sees only key 0: O = v_0 exactly representable
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) <= 1e-6


@pytest.mark.parametrize("Nq,Nkv", [(300, 1000), (1, 777), (129, 4096)])
def test_causal_fewer_queries_than_keys(Nq, Nkv):
    q, k, v = I.make_general(2, 4, 2, Nq, Nkv, 128, "bf16", seed=430 + Nq)
    check("bf16", q, k, v, causal=True)
    check("bf16", q, k, v, splits=4, causal=True)


def test_causal_more_queries_than_keys():
    """The first Nq - Nkv queries see no key: O = 0, lse = -inf."""
    q, k, v = I.make_general(1, 2, 2, 500, 200, 64, "bf16", seed=440)
    o, lse = check("bf16", q, k, v, causal=True)
    assert np.all(o[:, :, :300] == 0.0) and np.all(np.isneginf(lse[:, :, :300]))


def test_causal_split_with_empty_partitions():
    """Square causal with 8 key partitions: early query blocks see only the
    first partition, the others are empty and must not disturb the merge."""
    q, k, v = I.make_general(1, 2, 2, 2048, 2048, 128, "bf16", seed=450)
    check("bf16", q, k, v, splits=8, causal=True)


def test_causal_f16_gqa():
    q, k, v = I.make_general(2, 8, 4, 700, 700, 64, "f16", seed=460)
    check("f16", q, k, v, causal=True)


def test_causal_decode_equals_unmasked():
    q, k, v = I.make_general(1, 4, 4, 1, 1000, 128, "bf16", seed=470)
    o1, l1 = run_fa_ex(q, k, v, "bf16", 1, causal=True)
    o2, l2 = run_fa_ex(q, k, v, "bf16", 1, causal=False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
