"""Failure detection on the GPU without a fault: a kernel waits, with the
forward kernel's bounded barrier wait, on a barrier phase nothing completes.
The wait must give up (about 1 s), the kernel must exit normally, the host
must read FA_ERR_TIMEOUT once, and the context must stay usable."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_LSE, compare, ensure_library, run_fa, tol_o, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def test_barrier_timeout_is_reported_then_cleared():
    s = torch.cuda.current_stream()
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
    assert fab.fa_selftest_barrier_timeout(s.cuda_stream) == fab.FA_OK
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_ERR_TIMEOUT
    assert "device error word" in fab.fa_last_error_message()
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK  # read once, then clear
    # the context is still usable: a forward pass runs and is correct
    w = I.custom(1, 2, 300, 64, "bf16", seed=31)
    q, k, v = I.make(w)
    o, lse = run_fa(w, q, k, v)
    err_o, err_l = compare(w, o, lse, q, k, v)
    assert err_o <= tol_o(w) and err_l <= TOL_LSE


def test_timeout_does_not_stop_later_launches():
    """A timed-out launch only stops its own CTAs; a forward pass enqueued
    after it, before anyone reads the status, still computes everything."""
    s = torch.cuda.current_stream()
    w = I.custom(2, 3, 513, 128, "bf16", seed=32)
    q, k, v = I.make(w)
    tq, tk, tv = (to_device(x, w.dtype) for x in (q, k, v))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda")
    assert fab.fa_selftest_barrier_timeout(s.cuda_stream) == fab.FA_OK
    st = fab.fa_fwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    w.B, w.H, w.N, w.d, float(w.scale), fab.FA_DTYPE_BF16, s.cuda_stream)
    assert st == fab.FA_OK
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_ERR_TIMEOUT  # sticky until read
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(on).all() and np.isfinite(ln).all()
    err_o, err_l = compare(w, on, ln, q, k, v)
    assert err_o <= tol_o(w) and err_l <= TOL_LSE
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
