"""fa_fwd_ex on the GPU against the fp64 oracle: key-range partitions
(split-KV) merged by the second kernel, query and key lengths that differ
(decode steps: one query against a long key cache), and grouped key/value
heads (GQA / MQA).  Same tolerances as the square parity tests."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_LSE, compare_ex, ensure_library, run_fa_ex, tol_o_dtype

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def check(dtype, q, k, v, splits, rows=None):
    o, lse = run_fa_ex(q, k, v, dtype, splits)
    if rows is None:
        assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v, rows=rows)
    assert err_o <= tol_o_dtype(dtype), (q.shape, k.shape, splits, err_o)
    assert err_l <= TOL_LSE, (q.shape, k.shape, splits, err_l)
    return o, lse


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 32])
@pytest.mark.parametrize("d", [64, 128])
def test_split_kv_bf16(splits, d):
    q, k, v = I.make_general(1, 2, 2, 300, 1000, d, "bf16", seed=50 + splits)
    check("bf16", q, k, v, splits)


@pytest.mark.parametrize("splits", [1, 4])
def test_split_kv_f32(splits):
    q, k, v = I.make_general(1, 2, 2, 200, 700, 64, "f32", seed=60 + splits)
    check("f32", q, k, v, splits)


@pytest.mark.parametrize("Nkv", [1, 127, 128, 4097])
@pytest.mark.parametrize("splits", [1, 16])
def test_decode_single_query(Nkv, splits):
    q, k, v = I.make_general(2, 8, 8, 1, Nkv, 128, "bf16", seed=70 + Nkv)
    check("bf16", q, k, v, splits)


@pytest.mark.parametrize("H,H_kv", [(8, 2), (8, 1), (6, 3)])
def test_grouped_kv_heads(H, H_kv):
    q, k, v = I.make_general(2, H, H_kv, 257, 511, 64, "bf16", seed=80 + H_kv)
    check("bf16", q, k, v, 1)
    check("bf16", q, k, v, 4)


def test_gqa_decode_long_cache():
    """A decode step of a grouped-query model against a 16k-key cache, split
    across 32 partitions; checked on every (b, h) row."""
    q, k, v = I.make_general(4, 32, 8, 1, 16384, 128, "bf16", seed=90)
    check("bf16", q, k, v, 32)


def test_more_queries_than_keys():
    q, k, v = I.make_general(1, 3, 3, 1000, 130, 128, "bf16", seed=91)
    check("bf16", q, k, v, 2)


def test_split_matches_unsplit_closely():
    q, k, v = I.make_general(2, 4, 4, 512, 2048, 128, "bf16", seed=92)
    o1, l1 = run_fa_ex(q, k, v, "bf16", 1)
    o8, l8 = run_fa_ex(q, k, v, "bf16", 8)
    assert np.max(np.abs(o1 - o8)) <= 2 ** -7 and np.max(np.abs(l1 - l8)) <= 1e-4


def test_fa_fwd_equals_fa_fwd_ex_automatic():
    """fa_fwd is fa_fwd_ex's automatic plan where that plan merges in-cluster
    (12 query blocks here: their keys split across clusters): the same bits."""
    w = I.custom(2, 3, 333, 128, "bf16", seed=93)
    q, k, v = I.make(w)
    from .gpu_util import compare, run_fa
    o_a, l_a = run_fa(w, q, k, v)
    o_b, l_b = run_fa_ex(q, k, v, "bf16", 0)
    assert np.array_equal(o_a, o_b) and np.array_equal(l_a, l_b)
    err_o, err_l = compare(w, o_a, l_a, q, k, v)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE


def test_workspace_too_small_is_rejected():
    q, k, v = I.make_general(1, 2, 2, 64, 1024, 64, "bf16", seed=94)
    need = fab.fa_fwd_ex_workspace_size(1, 2, 64, 1024, 64, 4)
    assert need == 4 * 1 * 2 * 64 * (64 + 4) * 4
    from .gpu_util import to_device
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    o = torch.empty_like(tq)
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    st = fab.fa_fwd_ex(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), None, 1, 2, 2, 64,
                       1024, 64, 0.125, fab.FA_DTYPE_BF16, 4, ws.data_ptr(), need - 16, None)
    assert st == fab.FA_ERR_INVALID_ARG


BENCH_FORWARD = [n for n, w in I.WORKLOADS.items() if not w.backward]


@pytest.mark.parametrize("name", BENCH_FORWARD)
def test_workloads_in_bench_launch_configuration(name):
    """Every forward workload as the benchmark launches it: fa_fwd where the
    workload fits its signature, else fa_fwd_ex with the workload's
    num_splits (0: the library's plan for this device, which on a 152-SM GPU
    splits the last wave of the headline shapes).  Every output row must be
    written; the small workloads are compared on every row, the large ones on
    seeded rows, the edge rows and rows of the last three heads (the ones a
    split last wave covers)."""
    from bench import uses_fa_fwd
    from .gpu_util import edge_rows, run_fa
    w = I.WORKLOADS[name]
    q, k, v = I.make(w)
    if uses_fa_fwd(w):
        o, lse = run_fa(w, q, k, v)
    else:
        o, lse = run_fa_ex(q, k, v, w.dtype, w.splits, causal=w.causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = None
    if w.oracle_rows is not None:
        tail = [(w.B - 1, h, i) for h in range(max(0, w.H - 3), w.H)
                for i in (0, 1, w.N // 2, w.N - 2, w.N - 1)]
        rows = np.concatenate([edge_rows(w, w.oracle_rows), np.array(tail, dtype=np.int64)])
    err_o, err_l = compare_ex(w.dtype, o, lse, q, k, v, rows=rows, causal=w.causal)
    assert err_o <= tol_o_dtype(w.dtype) and err_l <= TOL_LSE, (name, err_o, err_l)


@pytest.mark.parametrize("name", ["gqa_b2h32kv8_n8192_d128", "causal_b2h32_n8192_d128",
                                  "f16_b2h32_n8192_d128"])
def test_headline_variants_sampled_rows(name):
    from .gpu_util import edge_rows
    w = I.WORKLOADS[name]
    q, k, v = I.make(w)
    o, lse = run_fa_ex(q, k, v, w.dtype, 1, causal=w.causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = compare_ex(w.dtype, o, lse, q, k, v, rows=edge_rows(w, w.oracle_rows), causal=w.causal)
    assert err_o <= tol_o_dtype(w.dtype) and err_l <= TOL_LSE, (err_o, err_l)


@pytest.mark.parametrize("Nq,G", [(1, 2), (1, 8), (16, 4), (32, 4), (3, 5)])
@pytest.mark.parametrize("splits", [1, 4])
def test_packed_grouped_heads(Nq, G, splits):
    """Query heads of one key/value head packed into one tile (Nq * G <= 128),
    including exactly 128 packed rows and a group size that is not a power
    of two."""
    H_kv = 3
    q, k, v = I.make_general(2, H_kv * G, H_kv, Nq, 1500, 128, "bf16", seed=500 + Nq * G + splits)
    check("bf16", q, k, v, splits)


def test_packed_causal_and_fp32():
    from .gpu_util import compare_ex, run_fa_ex
    q, k, v = I.make_general(1, 8, 2, 16, 700, 64, "bf16", seed=520)
    o, lse = run_fa_ex(q, k, v, "bf16", 3, causal=True)
    err_o, err_l = compare_ex("bf16", o, lse, q, k, v, causal=True)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE
    q, k, v = I.make_general(1, 8, 2, 4, 900, 64, "f32", seed=521)
    check("f32", q, k, v, 2)
    q, k, v = I.make_general(2, 16, 4, 1, 3000, 64, "f16", seed=522)
    check("f16", q, k, v, 4)


def test_automatic_plan_launch_counts():
    """The plan on this device: the headline shape on a 152-SM GPU runs its
    13 full waves unsplit and its last 72 blocks in a second launch, split
    into clusters that merge in distributed shared memory (2 launches);
    causal and fp32 launches never take the split last wave; an underfilled
    launch splits every block, merged in-cluster (1 launch) or, for the
    decode kernel, through the workspace (2 launches)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bf16, f32, causal = fab.FA_DTYPE_BF16, fab.FA_DTYPE_F32, fab.FA_FLAG_CAUSAL
    blocks = 2 * 32 * 32
    last = blocks % sms
    expect = 2 if 0 < last and 2 * last <= sms else 1
    assert fab.fa_fwd_ex_launches(2, 32, 32, 8192, 8192, 128, bf16, 0) == expect
    assert fab.fa_fwd_launches(2, 32, 8192, 128, bf16) == expect
    assert fab.fa_fwd_ex_launches(2, 32, 32, 8192, 8192, 128, bf16 | causal, 0) == 1
    assert fab.fa_fwd_launches(2, 32, 8192, 128, bf16 | causal) == 1
    # 512 blocks of 16 key tiles: 3 full waves, a last wave of 56 split in clusters
    assert fab.fa_fwd_ex_launches(4, 16, 16, 2048, 2048, 64, bf16, 0) == (2 if 0 < 512 % sms and 2 * (512 % sms) <= sms else 1)
    assert fab.fa_fwd_ex_launches(8, 16, 16, 1024, 1024, 64, bf16, 0) == 1   # 8 key tiles: not split
    assert fab.fa_fwd_ex_launches(1, 1, 1, 512, 512, 64, f32, 0) == 1       # clusters of 4
    assert fab.fa_fwd_launches(1, 1, 512, 64, f32) == 1
    assert fab.fa_fwd_ex_launches(8, 32, 8, 1, 16384, 128, bf16, 0) == 2     # decode: 64 CTAs, 2 partitions


@pytest.mark.parametrize("B,H,H_kv,N,d,dtype", [
    (1, 10, 10, 4096, 64, "bf16"),    # 160 blocks: 152 unsplit, the last 8 of one head split
    (1, 10, 10, 4500, 128, "bf16"),   # 180 blocks: the split tail crosses a head, ragged last blocks
    (1, 20, 5, 4096, 64, "f16"),      # grouped heads, 320 blocks, a tail of 16
    (1, 6, 6, 3000, 64, "bf16"),      # 72 blocks (one partial wave): partitions of every block
])
def test_automatic_partitions(B, H, H_kv, N, d, dtype):
    """num_splits = 0: the library plans the partitions for the device (on a
    152-SM GB300 these shapes run their last wave as a split second launch
    merged over its rows); every output row matches the oracle."""
    q, k, v = I.make_general(B, H, H_kv, N, N, d, dtype, seed=980 + H + d)
    o, lse = run_fa_ex(q, k, v, dtype, 0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = compare_ex(dtype, o, lse, q, k, v)
    assert err_o <= tol_o_dtype(dtype) and err_l <= TOL_LSE, (err_o, err_l)


@pytest.mark.parametrize("B,H,N,d", [(2, 32, 2048, 128), (4, 16, 2048, 64)])
def test_dependent_last_wave_in_a_chain(B, H, N, d):
    """Where the plan runs its last wave as a second launch that may start
    while the full waves are still running, a later call on the same stream
    still sees the whole output: three calls chained through O (each call's
    output is the next call's queries) give the same bits with and without a
    synchronize between the calls, and the first step matches the oracle."""
    bf16 = fab.FA_DTYPE_BF16
    if fab.fa_fwd_launches(B, H, N, d, bf16) != 2:
        pytest.skip("the plan on this device has no split last wave for this shape")
    w = I.custom(B, H, N, d, "bf16", seed=1201 + d)
    q, k, v = I.make(w)
    from .gpu_util import compare, to_device
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    s = torch.cuda.current_stream()

    def chain(sync):
        outs, x = [], tq
        for _ in range(3):
            o = torch.full_like(tq, float("nan"))
            lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
            st = fab.fa_fwd(x.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, float(w.scale), bf16, s.cuda_stream)
            assert st == fab.FA_OK, (st, fab.fa_last_error_message())
            if sync:
                torch.cuda.synchronize()
            outs.append((o, lse))
            x = o
        torch.cuda.synchronize()
        assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
        return outs

    ref = chain(True)
    for _ in range(3):
        got = chain(False)
        for (o_r, l_r), (o_g, l_g) in zip(ref, got):
            assert torch.equal(o_r.view(torch.int16), o_g.view(torch.int16))
            assert torch.equal(l_r, l_g)
    o1, l1 = ref[0]
    last_head = np.stack([np.full(64, B - 1), np.full(64, H - 1), np.linspace(0, N - 1, 64).astype(np.int64)], 1)
    rows = np.concatenate([I.sample_rows(w, 192), last_head])   # the last head lies in the split last wave
    err_o, err_l = compare(w, o1.float().cpu().numpy(), l1.cpu().numpy(), q, k, v, rows=rows)
    assert err_o <= tol_o_dtype("bf16") and err_l <= TOL_LSE, (err_o, err_l)
