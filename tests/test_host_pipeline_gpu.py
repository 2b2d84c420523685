"""fa_fwd_host: the forward pass on host tensors with overlapped copies.

Each chunk is an ordinary fa_fwd_ex launch (with the library's automatic key
partitions) on device copies of contiguous head ranges, so the outputs equal
fa_fwd_ex on the whole problem up to the summation order of the partitions
(bit for bit where no chunk is split); they are also compared with the oracle
on sampled rows."""
import numpy as np
import pytest

from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

from .gpu_util import DTYPE_CODES, TOL_LSE, compare_ex, ensure_library, run_fa_ex, to_device, tol_o_dtype

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_library()


def run_host(q, k, v, dtype, causal=False, with_lse=True, pinned=True, stream=None):
    B, H, Nq, d = q.shape
    H_kv, Nkv = k.shape[1], k.shape[2]
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    hq, hk, hv = (pin(to_device(x, dtype).cpu()) for x in (q, k, v))
    ho = pin(torch.full_like(hq, float("nan")))
    hl = pin(torch.full((B, H, Nq), float("nan"), dtype=torch.float32)) if with_lse else None
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    need = fab.fa_fwd_host_workspace_size(B, H, H_kv, Nq, Nkv, d, code)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    sc = float(np.float32(1.0 / np.sqrt(d)))
    s = stream if stream is not None else torch.cuda.current_stream()
    st = fab.fa_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(),
                         hl.data_ptr() if hl is not None else None, B, H, H_kv, Nq, Nkv, d, sc, code, base,
                         need, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
    return ho.float().numpy(), (hl.numpy() if hl is not None else None)


@pytest.mark.parametrize("B,H,H_kv,Nq,Nkv,d,dtype,causal", [
    (1, 1, 1, 300, 333, 64, "bf16", False),      # one chunk
    (1, 3, 3, 200, 200, 128, "bf16", True),      # fewer chunks than slots
    (3, 12, 6, 130, 260, 64, "f16", False),      # 18 units: 9 chunks of 2
    (2, 17, 17, 257, 129, 128, "bf16", True),    # ragged last chunk
    (4, 16, 4, 1, 700, 128, "bf16", False),      # decode: packed grouped heads
    (2, 4, 4, 160, 160, 64, "f32", False),       # TF32 path
    (2, 40, 40, 2048, 2048, 64, "bf16", False),  # 80 units: ramp chunks of 4 and 8 units, split
    (2, 40, 40, 2048, 2048, 128, "f16", True),   # ramp chunks of 2 and 4 units, causal
])
def test_matches_device_call(B, H, H_kv, Nq, Nkv, d, dtype, causal):
    q, k, v = I.make_general(B, H, H_kv, Nq, Nkv, d, dtype, seed=700 + H + Nq)
    o_h, l_h = run_host(q, k, v, dtype, causal)
    o_d, l_d = run_fa_ex(q, k, v, dtype, 1, causal=causal)
    # partitions change only the order of the fp32 sums: within an output
    # rounding step of the unsplit result
    # (rows that see no key: O = 0 and lse = -inf on both sides)
    assert not np.isnan(o_h).any() and not np.isnan(l_h).any()
    assert np.array_equal(np.isneginf(l_h), np.isneginf(l_d))
    seen = np.isfinite(l_d)
    assert np.max(np.abs(o_h - o_d)) <= 2 ** -7 and np.max(np.abs(l_h[seen] - l_d[seen])) <= 1e-4
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, B, 16), rng.integers(0, H, 16), rng.integers(0, Nq, 16)], axis=1)
    err_o, err_l = compare_ex(dtype, o_h, l_h, q, k, v, rows=rows, causal=causal)
    assert err_o <= tol_o_dtype(dtype) and err_l <= TOL_LSE


def test_pageable_host_memory():
    """Host tensors that are not pinned: the copies run through the
    driver's staging buffers, and the result is the same."""
    q, k, v = I.make_general(2, 8, 2, 300, 300, 128, "bf16", seed=730)
    o_p, l_p = run_host(q, k, v, "bf16")
    o_u, l_u = run_host(q, k, v, "bf16", pinned=False)
    assert np.array_equal(o_p, o_u) and np.array_equal(l_p, l_u)


def test_two_threads_two_streams():
    """Two host threads call fa_fwd_host at once on their own streams (the
    library serialises its internal streams per device); both results equal
    the single-threaded ones."""
    import threading
    shapes = [(2, 8, 2, 300, 300, 128, 740), (1, 6, 6, 500, 700, 64, 741)]
    inputs = [I.make_general(B, H, Hk, Nq, Nk, d, "bf16", seed=sd) for B, H, Hk, Nq, Nk, d, sd in shapes]
    ref = [run_host(q, k, v, "bf16") for q, k, v in inputs]
    got = [None, None]
    errors = []

    def work(i):
        try:
            with torch.cuda.device(0):
                s = torch.cuda.Stream()
                got[i] = run_host(*inputs[i], "bf16", stream=s)
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for (o_r, l_r), (o_g, l_g) in zip(ref, got):
        assert np.array_equal(o_r, o_g) and np.array_equal(l_r, l_g)


def test_without_lse_and_repeated():
    q, k, v = I.make_general(2, 8, 2, 300, 300, 128, "bf16", seed=710)
    o1, _ = run_host(q, k, v, "bf16", with_lse=False)
    o2, l2 = run_host(q, k, v, "bf16")
    assert np.array_equal(o1, o2) and np.isfinite(l2).all()


@pytest.mark.parametrize("B,H,H_kv,Nq,Nkv,d,dtype,causal", [
    (1, 2, 2, 300, 333, 64, "bf16", False),      # one chunk
    (2, 8, 2, 200, 260, 128, "bf16", True),      # grouped heads
    (4, 16, 16, 256, 1024, 64, "f16", False),    # several chunks
    (2, 36, 36, 1024, 1024, 64, "bf16", False),  # 72 units: ramp chunks
])
def test_backward_matches_device_call(B, H, H_kv, Nq, Nkv, d, dtype, causal):
    """fa_bwd_host equals fa_bwd on device copies up to the summation order
    of the dQ reductions (and the oracle within the gradient tolerance)."""
    import oracle
    from .gpu_util import grad_errors, run_bwd, tol_grad
    q, k, v = I.make_general(B, H, H_kv, Nq, Nkv, d, dtype, seed=720 + H + Nq)
    dout = I.make_dout(B, H, Nq, d, dtype, seed=720 + H + Nq)
    sc = float(np.float32(1.0 / np.sqrt(d)))
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    # forward on the device for o and lse, then both backward forms
    (gq, gk, gv), _ = run_bwd(q, k, v, dout, dtype, causal=causal)
    tq, tk, tv, tdo = (to_device(x, dtype) for x in (q, k, v, dout))
    o = torch.empty_like(tq)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    assert fab.fa_fwd_ex(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv,
                         Nq, Nkv, d, sc, code, 1, None, 0, s.cuda_stream) == fab.FA_OK
    hin = [t.cpu().pin_memory() for t in (tq, tk, tv, o, tdo, lse)]
    hout = [torch.full_like(t, float("nan")).pin_memory() for t in (hin[0], hin[1], hin[2])]
    need = fab.fa_bwd_host_workspace_size(B, H, H_kv, Nq, Nkv, d)
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    st = fab.fa_bwd_host(*(t.data_ptr() for t in hin), *(t.data_ptr() for t in hout), B, H, H_kv, Nq, Nkv, d,
                         sc, code, base, need, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    assert fab.fa_device_status(s.cuda_stream) == fab.FA_OK
    got = [t.float().numpy() for t in hout]
    for a, r in zip(got, (gq, gk, gv)):
        assert np.max(np.abs(a - r)) <= 1e-2 * max(np.max(np.abs(r)), 1e-30)  # a bf16/fp16 ulp or so
    errs = grad_errors(got, oracle.attention_bwd_f64(q, k, v, dout, sc, causal=causal))
    assert max(errs) <= tol_grad(dtype), errs
