"""The allocation-free entry point, fa_fwd_ex_static, for callers that
cannot allocate device memory (plugins of engines that own the device memory
pool, per-step code that must not call cudaMalloc).  Its split partials live
in the library's static per-device array instead of a caller workspace.

Each case runs fa_fwd_ex with a caller-allocated workspace once and
fa_fwd_ex_static twice in a row on the same inputs (the array keeps the
previous call's contents).  Both static results must match the fa_fwd_ex
result and the fp64 oracle within the parity tolerance.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_LSE, TOL_O_BF16, compare_ex, ensure_library, run_fa_ex, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def run_static(q, k, v, splits):
    B, H, Nq, d = q.shape
    H_kv, Nkv = k.shape[1], k.shape[2]
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    st = fab.fa_fwd_ex_static(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, H, H_kv, Nq, Nkv, d, float(I.default_scale(d)),
                              fab.FA_DTYPE_BF16, splits, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
    return o.float().cpu().numpy(), lse.cpu().numpy()


# (name, shape (B, H, H_kv, N_q, N_kv, d), seed, num_splits, oracle rows)
#   rows None: every row; "tail": the last two heads (the last wave of the
#   automatic plan) and 256 seeded rows
CASES = [
    ("decode, 16 partitions", (2, 8, 2, 1, 8192, 128), 301, 16, None),
    ("prefill, 6 partitions", (1, 4, 4, 700, 1500, 64), 302, 6, None),
    ("decode, automatic plan", (1, 8, 1, 1, 16384, 128), 303, 0, None),
    ("several waves, automatic plan", (1, 40, 40, 1024, 4096, 128), 304, 0, "tail"),
]


def _rows(shape, which):
    B, H, _, Nq, _, _ = shape
    if which is None:
        return None
    tail = [(B - 1, h, i) for h in (H - 2, H - 1) for i in range(Nq)]
    rng = np.random.default_rng(7)
    sample = [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(Nq))) for _ in range(256)]
    return np.array(tail + sample, dtype=np.int64)


@pytest.mark.parametrize("name,shape,seed,splits,which", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_matches_caller_workspace_and_oracle_twice(name, shape, seed, splits, which):
    B, H, H_kv, Nq, Nkv, d = shape
    q, k, v = I.make_general(B, H, H_kv, Nq, Nkv, d, "bf16", seed=seed)
    need = fab.fa_fwd_ex_workspace_size(B, H, Nq, Nkv, d, splits)
    assert 0 < need <= fab.fa_fwd_ex_static_capacity()
    assert fab.fa_fwd_ex_launches(B, H, H_kv, Nq, Nkv, d, fab.FA_DTYPE_BF16, splits) >= 2
    o_ref, l_ref = run_fa_ex(q, k, v, "bf16", splits)
    rows = _rows(shape, which)
    for call in range(2):
        o_s, l_s = run_static(q, k, v, splits)
        assert np.isfinite(o_s).all() and np.isfinite(l_s).all(), (name, call)
        # the existing entry point on a caller workspace
        assert np.max(np.abs(o_s - o_ref)) <= TOL_O_BF16, (name, call)
        assert np.max(np.abs(l_s - l_ref)) <= TOL_LSE, (name, call)
        # the fp64 oracle
        err_o, err_l = compare_ex("bf16", o_s, l_s, q, k, v, rows=rows)
        assert err_o <= TOL_O_BF16 and err_l <= TOL_LSE, (name, call, err_o, err_l)


def test_oversized_request_is_rejected_before_any_work():
    cap = fab.fa_fwd_ex_static_capacity()
    # B*H*Nq rows x (d+4) floats x splits well beyond the capacity
    B, H, Nq, Nkv, d, splits = 8, 32, 4096, 8192, 128, 32
    assert fab.fa_fwd_ex_workspace_size(B, H, Nq, Nkv, d, splits) > cap
    # Real device memory, far smaller than the sizes claimed: q, k, v and o
    # sit 256 bytes apart in one buffer, so even if the capacity check were
    # lost, the overlap checks would refuse the call before any launch.
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    base = buf.data_ptr()
    st = fab.fa_fwd_ex_static(base, base + 256, base + 512, base + 768, None, B, H, H, Nq, Nkv, d,
                              0.088, fab.FA_DTYPE_BF16, splits, None)
    assert st == fab.FA_ERR_UNSUPPORTED
    assert "static workspace" in fab.fa_last_error_message()
    torch.cuda.synchronize()
    assert torch.count_nonzero(buf).item() == 0
