"""Helpers of the GPU parity tests: upload seeded inputs, call the C ABI,
compare with the CPU oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle
from exact_tiled_attention_04_gb300 import binding as fab
from exact_tiled_attention_04_gb300 import inputs as I

# Tolerances against the fp64 oracle (absolute): O for bf16 in/out with fp32
# accumulation, O for fp32 in/out on the TF32 tensor-core path, and lse.
TOL_O_BF16 = 1.5e-2
TOL_O_F32 = 2e-3
TOL_LSE = 1e-3
# fp16 in/out (no stated bar): weights rounded to fp16 move O by at most
# 2^-11 * 2 max|v| (about 2e-3 for |v| <= 4) and the output rounding by half
# an fp16 ulp (<= 1e-3 for |O| < 2): 4e-3.
TOL_O_F16 = 4e-3

DTYPE_CODES = {"bf16": fab.FA_DTYPE_BF16, "f16": fab.FA_DTYPE_F16, "f32": fab.FA_DTYPE_F32}


def ensure_library():
    from exact_tiled_attention_04_gb300 import build
    build.build()
    return fab.load()


def to_device(x: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        bits = I.bf16_bits(x).view(np.int16)
        return torch.from_numpy(bits).cuda().view(torch.bfloat16)
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32).astype(np.float16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def run_fa(w, q, k, v, scale=None, with_lse=True, stream=None):
    """Run the CUDA path through the C ABI on poisoned outputs; returns
    (o float32 numpy, lse numpy or None)."""
    import torch
    tq, tk, tv = (to_device(x, w.dtype) for x in (q, k, v))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    s = stream if stream is not None else torch.cuda.current_stream()
    dt = DTYPE_CODES[w.dtype] | (fab.FA_FLAG_CAUSAL if getattr(w, "causal", False) else 0)
    sc = float(w.scale if scale is None else scale)
    st = fab.fa_fwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                    lse.data_ptr() if lse is not None else None,
                    w.B, w.H, w.N, w.d, sc, dt, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    st = fab.fa_device_status(s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    return o.float().cpu().numpy(), (lse.cpu().numpy() if lse is not None else None)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bfloat16 unit in the last place at |x| (8 significant bits):
    for |x| in [2^e, 2^(e+1)) it is 2^(e-8)."""
    _, e = np.frexp(np.abs(x))          # |x| = m * 2^e with m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 values rounded to the nearest bfloat16 (ties to even), as
    float64: the best a bf16 output can be."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                   # x = m 2^e, |m| in [0.5, 1)
    # 8 significant bits: m * 2^8 rounded to an integer (np.round: ties to even)
    return np.ldexp(np.round(m * 256.0), e - 8)


def half_ulp_f16(x: np.ndarray) -> np.ndarray:
    """Half an fp16 unit in the last place at |x| (11 significant bits)."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, e - 12)


def o_allowance(x: np.ndarray, dtype: str) -> np.ndarray:
    """Extra error allowed on top of the absolute O tolerance.  A bf16 output
    is rounded to the nearest bf16 value, which alone can be off by half a
    bf16 ulp of |O|: 2^-6 = 0.0156 for |O| in [4, 8), more than the 1.5e-2
    bar.  Where that happens the bar becomes half an ulp plus 1e-3 of
    arithmetic error; everywhere else (|O| < 4) the bar is 1.5e-2 as stated."""
    if dtype == "bf16":
        return np.maximum(0.0, half_ulp_bf16(x) + 1e-3 - TOL_O_BF16)
    if dtype == "f16":
        return np.maximum(0.0, half_ulp_f16(x) + 1e-3 - TOL_O_F16)
    return np.zeros_like(x)


def compare(w, o_gpu, lse_gpu, q, k, v, rows=None, scale=None):
    """Max |GPU - oracle| over every row (rows=None) or the given (b,h,i).
    The O figure is max(|dO| - allowance(O_ref)) (see o_allowance), which is
    the plain max |dO| wherever |O_ref| < 4."""
    sc = float(w.scale if scale is None else scale)
    if rows is None:
        o_ref, l_ref = oracle.attention_f64(q, k, v, sc)
        og, lg = o_gpu, lse_gpu
    else:
        rows = np.asarray(rows, dtype=np.int64)
        o_ref, l_ref = oracle.attention_f64(q, k, v, sc, rows=rows)
        og = o_gpu[rows[:, 0], rows[:, 1], rows[:, 2]]
        lg = lse_gpu[rows[:, 0], rows[:, 1], rows[:, 2]] if lse_gpu is not None else None
    err_o = float(np.max(np.abs(og.astype(np.float64) - o_ref) - o_allowance(o_ref, w.dtype)))
    err_l = float(np.max(np.abs(lg.astype(np.float64) - l_ref))) if lg is not None else 0.0
    return err_o, err_l


def tol_o(w) -> float:
    return tol_o_dtype(w.dtype)


def edge_rows(w, count: int) -> np.ndarray:
    """Seeded rows plus the first and last row of the first and last head and
    rows on both sides of every 128-row tile boundary of head 0."""
    rows = [I.sample_rows(w, count)]
    fixed = [(0, 0, 0), (0, 0, w.N - 1), (w.B - 1, w.H - 1, 0), (w.B - 1, w.H - 1, w.N - 1)]
    for t in range(128, w.N, 128 * max(1, w.N // 2048)):
        fixed += [(0, 0, t - 1), (0, 0, t)]
    rows.append(np.array(fixed, dtype=np.int64))
    return np.concatenate(rows)


def run_fa_ex(q, k, v, dtype: str, num_splits: int, scale=None, stream=None, with_lse=True,
              causal=False):
    """fa_fwd_ex through the C ABI on poisoned outputs, with a workspace the
    caller (this test) allocates.  Returns (o, lse) as numpy."""
    import torch
    B, H, Nq, d = q.shape
    H_kv, Nkv = k.shape[1], k.shape[2]
    tq, tk, tv = (to_device(x, dtype) for x in (q, k, v))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    wbytes = fab.fa_fwd_ex_workspace_size(B, H, Nq, Nkv, d, num_splits)
    ws = torch.full((max(wbytes, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream()
    dt = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    sc = float(I.default_scale(d) if scale is None else scale)
    st = fab.fa_fwd_ex(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                       lse.data_ptr() if lse is not None else None, B, H, H_kv, Nq, Nkv, d, sc, dt,
                       num_splits, ws.data_ptr() if wbytes else None, wbytes, s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    st = fab.fa_device_status(s.cuda_stream)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    return o.float().cpu().numpy(), (lse.cpu().numpy() if lse is not None else None)


def compare_ex(dtype: str, o_gpu, lse_gpu, q, k, v, scale=None, rows=None, causal=False):
    """Max |GPU - oracle| (O with the rounding allowance, lse).  Rows with no
    visible key must have lse = -inf on both sides (inf is reported if not)."""
    d = q.shape[3]
    sc = float(I.default_scale(d) if scale is None else scale)
    if rows is None:
        o_ref, l_ref = oracle.attention_f64_ex(q, k, v, sc, causal=causal)
        og, lg = o_gpu, lse_gpu
    else:
        rows = np.asarray(rows, dtype=np.int64)
        o_ref, l_ref = oracle.attention_f64_ex(q, k, v, sc, rows=rows, causal=causal)
        og = o_gpu[rows[:, 0], rows[:, 1], rows[:, 2]]
        lg = lse_gpu[rows[:, 0], rows[:, 1], rows[:, 2]] if lse_gpu is not None else None
    err_o = float(np.max(np.abs(og.astype(np.float64) - o_ref) - o_allowance(o_ref, dtype)))
    err_l = 0.0
    if lg is not None:
        lg = lg.astype(np.float64)
        empty = np.isneginf(l_ref)
        if not np.array_equal(empty, np.isneginf(lg)):
            return err_o, float("inf")
        err_l = float(np.max(np.abs(lg[~empty] - l_ref[~empty]))) if (~empty).any() else 0.0
    return err_o, err_l


def tol_o_dtype(dtype: str) -> float:
    return {"bf16": TOL_O_BF16, "f16": TOL_O_F16, "f32": TOL_O_F32}[dtype]


# Backward pass: error = max |g - g_ref| / max |g_ref| per gradient tensor.
# P and dS are rounded to the input dtype before their products (relative
# 2^-9 for bf16, 2^-12 for fp16) and the outputs once more; each gradient
# element sums many such terms with independent rounding errors, so the
# normalised error stays near one output rounding (2^-9 = 2e-3 for bf16,
# 2^-12 = 2.4e-4 for fp16).  The bars leave 5x and 10x room for the D_i
# formed from the rounded forward output and for fp32 accumulation order.
TOL_GRAD_BF16 = 1e-2
TOL_GRAD_F16 = 2.5e-3


def tol_grad(dtype: str) -> float:
    return TOL_GRAD_F16 if dtype == "f16" else TOL_GRAD_BF16


def run_bwd(q, k, v, dout, dtype: str, causal: bool = False, scale=None):
    """Forward (fa_fwd_ex, one partition) then fa_bwd on the GPU through the
    C ABI; returns (dq, dk, dv) as float32 numpy arrays and the scale used.
    Outputs and workspace are poisoned with NaN first."""
    import torch
    B, H, Nq, d = q.shape
    H_kv, Nkv = k.shape[1], k.shape[2]
    sc = float(np.float32(1.0 / np.sqrt(d))) if scale is None else float(scale)
    tq, tk, tv, tdo = (to_device(x, dtype) for x in (q, k, v, dout))
    o = torch.full_like(tq, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    code = DTYPE_CODES[dtype] | (fab.FA_FLAG_CAUSAL if causal else 0)
    st = fab.fa_fwd_ex(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv,
                       Nq, Nkv, d, sc, code, 1, None, 0, s)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    dq = torch.full_like(tq, float("nan"))
    dk = torch.full_like(tk, float("nan"))
    dv = torch.full_like(tv, float("nan"))
    need = fab.fa_bwd_workspace_size(B, H, Nq, d)
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda")
    st = fab.fa_bwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), tdo.data_ptr(), lse.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, Nq, Nkv, d, sc, code,
                    ws.data_ptr(), need, s)
    assert st == fab.FA_OK, (st, fab.fa_last_error_message())
    st = fab.fa_device_status(s)
    assert st == fab.FA_OK, (st, fab.fa_status_string(st), fab.fa_last_error_message())
    return (dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()), sc


def grad_errors(got, ref):
    """Normalised errors (max |g - ref| / max |ref|) of (dq, dk, dv)."""
    out = []
    for g, r in zip(got, ref):
        assert np.isfinite(g).all()
        den = max(float(np.max(np.abs(r))), 1e-30)
        out.append(float(np.max(np.abs(g.astype(np.float64) - r))) / den)
    return out
