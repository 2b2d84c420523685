"""The allocation-free entry point, fa_fwd_ex_static, for callers that
cannot allocate device memory (plugins of engines that own the device memory
pool, per-step code that must not call cudaMalloc).  Its split partials live
in the library's static per-device array instead of a caller workspace.

Checked against fa_fwd_ex with a caller-allocated workspace on the same
inputs, within the parity tolerance, on two calls in a row (the array keeps
the previous call's contents).  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes alone in a fresh process."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_O_BF16, ensure_library, run_fa_ex, to_device

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


def test_static_workspace_matches_caller_workspace_twice():
    cases = [I.make_general(2, 8, 2, 1, 8192, 128, "bf16", seed=301),     # decode, 16 partitions
             I.make_general(1, 4, 4, 700, 1500, 64, "bf16", seed=302)]    # prefill, 6 partitions
    for (q, k, v), splits in zip(cases, (16, 6)):
        need = fab.fa_fwd_ex_workspace_size(q.shape[0], q.shape[1], q.shape[2], k.shape[2],
                                            q.shape[3], splits)
        assert 0 < need <= fab.fa_fwd_ex_static_capacity()
        o_ref, l_ref = run_fa_ex(q, k, v, "bf16", splits)
        o_s, l_s = run_static(q, k, v, splits)
        assert np.isfinite(o_s).all() and np.isfinite(l_s).all()
        assert np.max(np.abs(o_s - o_ref)) <= TOL_O_BF16
        assert np.max(np.abs(l_s - l_ref)) <= 1e-3


def test_oversized_request_is_rejected_before_any_work():
    cap = fab.fa_fwd_ex_static_capacity()
    # B*H*Nq rows x (d+4) floats x splits well beyond the capacity
    B, H, Nq, Nkv, d, splits = 8, 32, 4096, 8192, 128, 32
    assert fab.fa_fwd_ex_workspace_size(B, H, Nq, Nkv, d, splits) > cap
    st = fab.fa_fwd_ex_static(1 << 32, 2 << 32, 3 << 32, 4 << 32, None, B, H, H, Nq, Nkv, d, 0.088,
                              fab.FA_DTYPE_BF16, splits, None)
    assert st == fab.FA_ERR_UNSUPPORTED
    assert "static workspace" in fab.fa_last_error_message()
