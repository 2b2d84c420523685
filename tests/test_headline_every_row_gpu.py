"""Every row of the compute-bound headline workload (B=2, H=32, N=8192,
d=128, bf16 inputs N(0,1) x 0.5) against the fp64 oracle, element by
element, in the launch configuration the benchmark times.

"CUDA Flash Attention: Online Softmax with Shared Memory Tiling",
Correctness Verification: the GPU output is compared with the CPU reference
on every element.  Here that is all 524,288 rows of O (128 values each) and
of lse, at the stated bars (O <= 1.5e-2 absolute for bf16 in/out, lse <=
1e-3).  The oracle runs once for the module (about 45 s on 16 host cores)
and serves both entry points: fa_fwd, the call the benchmark times, and
fa_fwd_ex with num_splits = 0 on a caller workspace (the same automatic
plan for the device)."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import TOL_LSE, TOL_O_BF16, ensure_library, o_allowance, run_fa, run_fa_ex, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def headline():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    w = I.WORKLOADS[I.HEADLINE]
    q, k, v = I.make(w)
    o_ref, l_ref = oracle.attention_f64(q, k, v, float(w.scale))
    return w, q, k, v, o_ref, l_ref


def _check_every_row(w, o, lse, o_ref, l_ref, what):
    assert o.shape == o_ref.shape and lse.shape == l_ref.shape
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    d_o = np.abs(o.astype(np.float64) - o_ref)
    err_o = float(np.max(d_o - o_allowance(o_ref, "bf16")))
    err_l = float(np.max(np.abs(lse.astype(np.float64) - l_ref)))
    print(f"{what}: {o.shape[0] * o.shape[1] * o.shape[2]} rows, max|dO| = {float(d_o.max()):.3e} "
          f"(with the rounding allowance {err_o:.3e}), max|dlse| = {err_l:.3e}")
    assert err_o <= TOL_O_BF16, (what, err_o)
    assert err_l <= TOL_LSE, (what, err_l)


def test_fa_fwd_every_row(headline):
    w, q, k, v, o_ref, l_ref = headline
    o, lse = run_fa(w, q, k, v)
    _check_every_row(w, o, lse, o_ref, l_ref, "fa_fwd")


def test_fa_fwd_ex_automatic_every_row(headline):
    w, q, k, v, o_ref, l_ref = headline
    o, lse = run_fa_ex(q, k, v, "bf16", 0)
    _check_every_row(w, o, lse, o_ref, l_ref, "fa_fwd_ex(num_splits=0)")
