"""Key partitions merged inside thread-block clusters (fa_fwd and the
automatic plan of fa_fwd_ex): the partitions of one 256-row query block run
as the CTAs of one cluster and combine their partial results through
distributed shared memory with the online-softmax rescaling ("FlashAttention
dissected", sections "The mathematical breakthrough: Tiling and Online
Softmax" and "Interaction with the KV cache during inference").

Every row is compared with the fp64 oracle at the stated bars.  The shapes
give clusters of 2 to 8 CTAs (odd sizes included), ragged last key tiles,
rows past N in the last query block, the causal mask (partitions that see no
key of a row), every input dtype and both head dimensions, and the split
last wave of multi-wave launches."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import (DTYPE_CODES, TOL_LSE, compare_ex, ensure_library, run_fa_ex, to_device,
                       tol_o_dtype)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def run_fwd(q, k, v, dtype, causal=False, scale=None):
    """fa_fwd through the C ABI on NaN-poisoned outputs."""
    B, H, N, d = q.shape
    tq, tk, tv = (to_device(x, dtype) for x in (q, k, v))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    sc = float(I.default_scale(d) if scale is None else scale)
    st = fab.fa_fwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                    sc, code, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    st = fab.fa_device_status(s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    return o.float().cpu().numpy(), lse.cpu().numpy()


# (B, H, N, d, dtype, causal): single launches whose blocks split in-cluster
SHAPES = [
    (1, 1, 512, 64, "f32", False),     # 2 blocks, clusters of 4 (one key tile each)
    (1, 1, 129, 64, "bf16", False),    # 1 block, 2 partitions (the second sees one key)
    (1, 1, 2048, 128, "bf16", False),  # 8 blocks, clusters of 3 (the d = 128 merge's limit)
    (1, 3, 1000, 64, "bf16", False),   # 12 blocks, clusters of 8, ragged keys and rows
    (2, 4, 1000, 64, "bf16", False),   # the tail-masking workload's shape: clusters of 4
    (1, 2, 777, 128, "f16", True),     # causal, clusters of 3, partitions with no visible key
    (1, 1, 700, 64, "f32", True),      # causal fp32, clusters of 6
    (1, 5, 300, 128, "bf16", False),   # 10 blocks, 3 key tiles: clusters of 3
    (1, 1, 384, 64, "bf16", True),     # causal, clusters of 3: block 0's last partition
    (1, 1, 384, 128, "bf16", True),    #   sees no key and finishes while its peers still run
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SHAPES)
def test_fa_fwd_cluster_merge_every_row(B, H, N, d, dtype, causal):
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    assert fab.fa_fwd_launches(B, H, N, d, code) == 1
    q, k, v = I.make_general(B, H, H, N, N, d, dtype, seed=700 + N + H + d)
    o, lse = run_fwd(q, k, v, dtype, causal=causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v, causal=causal)
    assert err_o <= tol_o_dtype(dtype) and err_l <= TOL_LSE, (err_o, err_l)
    # where fa_fwd_ex's automatic plan is the same single launch (at most 8
    # partitions wanted), it gives the same bits
    if fab.fa_fwd_ex_launches(B, H, H, N, N, d, code, 0) == 1:
        o2, l2 = run_fa_ex(q, k, v, dtype, 0, causal=causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, l2)


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_cluster_merge_scales(scale):
    q, k, v = I.make_general(1, 2, 2, 900, 900, 64, "bf16", seed=731)
    o, lse = run_fwd(q, k, v, "bf16", scale=np.float32(scale))
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v, scale=np.float32(scale))
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (err_o, err_l)


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (1, 10, 4096, 64, "bf16"),    # 160 blocks: 152 unsplit, the last 8 in clusters of 4
    (1, 10, 4500, 128, "bf16"),   # 180 blocks: the split tail crosses a head, ragged last blocks
    (1, 20, 4096, 64, "f16"),     # 320 blocks, a tail of 16
])
def test_fa_fwd_split_last_wave(B, H, N, d, dtype):
    """Several waves with a partly filled last one: the tail's blocks run in
    a second launch as clusters; every row against the oracle."""
    code = DTYPE_CODES[dtype]
    assert fab.fa_fwd_launches(B, H, N, d, code) == 2
    q, k, v = I.make_general(B, H, H, N, N, d, dtype, seed=990 + H + d)
    o, lse = run_fwd(q, k, v, dtype)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v)
    assert err_o <= tol_o_dtype(dtype) and err_l <= TOL_LSE, (err_o, err_l)


def test_cluster_merge_deterministic_and_lse_optional():
    q, k, v = I.make_general(2, 4, 4, 1000, 1000, 64, "bf16", seed=741)
    o1, l1 = run_fwd(q, k, v, "bf16")
    o2, l2 = run_fwd(q, k, v, "bf16")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    o3 = torch.full_like(tq, float("nan"))
    st = fab.fa_fwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o3.data_ptr(), None, 2, 4, 1000, 64,
                    float(I.default_scale(64)), fab.FA_DTYPE_BF16, None)
    assert st == fab.FA_OK
    assert fab.fa_device_status(None) == fab.FA_OK
    assert np.array_equal(o1, o3.float().cpu().numpy())


# (B, H, H_kv, N_q, N_kv, d, dtype, causal): fa_fwd_ex's automatic plan on
# general shapes whose partitions merge in-cluster (query heads not packed)
GENERAL = [
    (1, 8, 2, 1000, 1000, 64, "bf16", False),   # grouped heads, 32 blocks, clusters of 4
    (1, 10, 10, 500, 3000, 64, "bf16", False),  # N_q != N_kv, 20 blocks over 24 key tiles
    (1, 24, 24, 500, 1200, 64, "bf16", True),   # causal with N_kv - N_q = 700, clusters of 3
    (1, 4, 2, 700, 700, 64, "f32", False),      # fp32, grouped heads, 12 blocks
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nkv,d,dtype,causal", GENERAL)
def test_automatic_plan_cluster_general_shapes(B, H, H_kv, Nq, Nkv, d, dtype, causal):
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    assert fab.fa_fwd_ex_launches(B, H, H_kv, Nq, Nkv, d, code, 0) == 1  # merged in-cluster
    q, k, v = I.make_general(B, H, H_kv, Nq, Nkv, d, dtype, seed=760 + H + Nq)
    o, lse = run_fa_ex(q, k, v, dtype, 0, causal=causal)
    assert np.isfinite(o).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v, causal=causal)
    assert err_o <= tol_o_dtype(dtype) and err_l <= TOL_LSE, (err_o, err_l)
