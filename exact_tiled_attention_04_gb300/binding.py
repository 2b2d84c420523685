"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

The functions here carry the C names and pass plain integers (device
addresses, sizes) straight through; every step of the attention forward pass
runs in the CUDA library.  If the library is missing the calls raise: there is
no CPU fallback.

``attention()`` is a convenience for PyTorch callers: it checks tensor
shapes/dtypes, allocates the outputs with PyTorch (the library itself never
allocates) and calls ``fa_fwd`` on the current stream.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ALIGNMENT = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_DTYPE_F32 = 0
FA_DTYPE_BF16 = 1
FA_DTYPE_F16 = 2
FA_FLAG_CAUSAL = 0x100

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {fa_status_string(status)} (status {status})"
        detail = fa_last_error_message()
        if detail:
            msg += f"; {detail}"
        super().__init__(msg)


def library_path() -> str:
    return LIB_PATH


def load(path: str | None = None):
    """Load the CUDA library (once).  Raises if it was not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA attention library not found at {path}; build it with "
                "`python -m exact_tiled_attention_04_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        i64, vp, f32, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        lib.fa_fwd.restype = c_int
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, c_int, vp]
        lib.fa_fwd_validate.restype = c_int
        lib.fa_fwd_validate.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, c_int]
        lib.fa_device_status.restype = c_int
        lib.fa_device_status.argtypes = [vp]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_status_string.argtypes = [c_int]
        lib.fa_last_error_message.restype = ctypes.c_char_p
        lib.fa_last_error_message.argtypes = []
        lib.fa_version.restype = c_int
        lib.fa_version.argtypes = []
        lib.fa_selftest_barrier_timeout.restype = c_int
        lib.fa_selftest_barrier_timeout.argtypes = [vp]
        sz = ctypes.c_size_t
        lib.fa_fwd_ex.restype = c_int
        lib.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, c_int, c_int,
                                  vp, sz, vp]
        lib.fa_fwd_ex_validate.restype = c_int
        lib.fa_fwd_ex_validate.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, c_int,
                                           c_int, vp, sz]
        lib.fa_fwd_ex_workspace_size.restype = sz
        lib.fa_fwd_ex_workspace_size.argtypes = [i64, i64, i64, i64, i64, c_int]
        lib.fa_fwd_ex_splits.restype = c_int
        lib.fa_fwd_ex_splits.argtypes = [i64, i64, i64, i64, i64, c_int]
        lib.fa_fwd_ex_launches.restype = c_int
        lib.fa_fwd_ex_launches.argtypes = [i64, i64, i64, i64, i64, i64, c_int, c_int]
        lib.fa_fwd_launches.restype = c_int
        lib.fa_fwd_launches.argtypes = [i64, i64, i64, i64, c_int]
        lib.fa_fwd_ex_static.restype = c_int
        lib.fa_fwd_ex_static.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, c_int,
                                         c_int, vp]
        lib.fa_fwd_ex_static_capacity.restype = sz
        lib.fa_fwd_ex_static_capacity.argtypes = []
        lib.fa_fwd_host.restype = c_int
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, c_int, vp, sz, vp]
        lib.fa_fwd_host_workspace_size.restype = sz
        lib.fa_fwd_host_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, c_int]
        bwd_args = [vp] * 9 + [i64] * 6 + [f32, c_int, vp, sz]
        lib.fa_bwd.restype = c_int
        lib.fa_bwd.argtypes = bwd_args + [vp]
        lib.fa_bwd_validate.restype = c_int
        lib.fa_bwd_validate.argtypes = bwd_args
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.fa_bwd_host.restype = c_int
        lib.fa_bwd_host.argtypes = bwd_args + [vp]
        lib.fa_bwd_host_workspace_size.restype = sz
        lib.fa_bwd_host_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64]
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/fa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(", text, flags=re.M)


# ----------------------------------------------------------- C-ABI mirrors
def fa_fwd(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, N: int, d: int,
           scale: float, dtype: int, stream: int | None) -> int:
    return load().fa_fwd(q, k, v, o, lse or None, B, H, N, d, scale, dtype, stream or None)


def fa_fwd_validate(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, N: int,
                    d: int, scale: float, dtype: int) -> int:
    return load().fa_fwd_validate(q, k, v, o, lse or None, B, H, N, d, scale, dtype)


def fa_fwd_ex(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int,
              N_q: int, N_kv: int, d: int, scale: float, dtype: int, num_splits: int,
              workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    return load().fa_fwd_ex(q, k, v, o, lse or None, B, H, H_kv, N_q, N_kv, d, scale, dtype,
                            num_splits, workspace or None, workspace_bytes, stream or None)


def fa_fwd_ex_validate(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int,
                       H_kv: int, N_q: int, N_kv: int, d: int, scale: float, dtype: int,
                       num_splits: int, workspace: int | None, workspace_bytes: int) -> int:
    return load().fa_fwd_ex_validate(q, k, v, o, lse or None, B, H, H_kv, N_q, N_kv, d, scale,
                                     dtype, num_splits, workspace or None, workspace_bytes)


def fa_fwd_ex_workspace_size(B: int, H: int, N_q: int, N_kv: int, d: int, num_splits: int) -> int:
    return int(load().fa_fwd_ex_workspace_size(B, H, N_q, N_kv, d, num_splits))


def fa_fwd_ex_splits(B: int, H: int, H_kv: int, N_q: int, N_kv: int, num_sms: int) -> int:
    return int(load().fa_fwd_ex_splits(B, H, H_kv, N_q, N_kv, num_sms))


def fa_fwd_ex_launches(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int, dtype: int,
                       num_splits: int) -> int:
    return load().fa_fwd_ex_launches(B, H, H_kv, N_q, N_kv, d, dtype, num_splits)


def fa_fwd_launches(B: int, H: int, N: int, d: int, dtype: int) -> int:
    return load().fa_fwd_launches(B, H, N, d, dtype)


def fa_fwd_ex_static(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int,
                     N_q: int, N_kv: int, d: int, scale: float, dtype: int, num_splits: int,
                     stream: int | None) -> int:
    """fa_fwd_ex for callers that cannot allocate device memory: the split
    partials live in the library's static per-device array (see include/fa.h)."""
    return load().fa_fwd_ex_static(q, k, v, o, lse or None, B, H, H_kv, N_q, N_kv, d, scale, dtype,
                                   num_splits, stream or None)


def fa_fwd_ex_static_capacity() -> int:
    return int(load().fa_fwd_ex_static_capacity())


def fa_fwd_host(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int, N_q: int,
                N_kv: int, d: int, scale: float, dtype: int, workspace: int | None, workspace_bytes: int,
                stream: int | None) -> int:
    return load().fa_fwd_host(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, workspace,
                              workspace_bytes, stream)


def fa_fwd_host_workspace_size(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int, dtype: int) -> int:
    return load().fa_fwd_host_workspace_size(B, H, H_kv, N_q, N_kv, d, dtype)


def fa_bwd(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int,
           H: int, H_kv: int, N_q: int, N_kv: int, d: int, scale: float, dtype: int,
           workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    return load().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype,
                         workspace, workspace_bytes, stream)


def fa_bwd_validate(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int,
                    B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int, scale: float, dtype: int,
                    workspace: int | None, workspace_bytes: int) -> int:
    return load().fa_bwd_validate(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale,
                                  dtype, workspace, workspace_bytes)


def fa_bwd_workspace_size(B: int, H: int, N_q: int, d: int) -> int:
    return load().fa_bwd_workspace_size(B, H, N_q, d)


def fa_bwd_host(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int,
                H: int, H_kv: int, N_q: int, N_kv: int, d: int, scale: float, dtype: int,
                workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    return load().fa_bwd_host(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype,
                              workspace, workspace_bytes, stream)


def fa_bwd_host_workspace_size(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int) -> int:
    return load().fa_bwd_host_workspace_size(B, H, H_kv, N_q, N_kv, d)


def fa_device_status(stream: int | None) -> int:
    return load().fa_device_status(stream or None)


def fa_selftest_barrier_timeout(stream: int | None) -> int:
    return load().fa_selftest_barrier_timeout(stream or None)


def fa_status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def fa_last_error_message() -> str:
    return load().fa_last_error_message().decode()


def fa_version() -> int:
    return load().fa_version()


# ------------------------------------------------------- PyTorch convenience
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float16:
        return FA_DTYPE_F16
    if t.dtype == torch.float32:
        return FA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16, float16 or float32")


def attention(q, k, v, scale: float | None = None, out=None, lse=None, with_lse: bool = True,
              stream=None, causal: bool = False, num_splits: int | None = None, workspace=None):
    """O = softmax(scale * Q K^T) V for CUDA tensors q [B, H, N_q, d] and k, v
    [B, H_kv, N_kv, d]: H a multiple of H_kv (query head h reads key/value
    head h // (H // H_kv)), N_q and N_kv independent (a decode step has
    N_q = 1).  bf16, fp16 (d = 64, 128) or fp32 (d = 64, TF32 tensor cores).

    Returns (out, lse); lse is fp32 [B, H, N_q] (natural log) or None when
    with_lse is False.  scale defaults to 1/sqrt(d) in fp32.  causal: query i
    sees keys j <= i + N_kv - N_q.  num_splits: key-range partitions (None:
    the library's automatic plan for the device, num_splits = 0 of
    fa_fwd_ex); their workspace is allocated when not given.  Enqueued on `stream` (default:
    PyTorch's current stream); raises FAError on a non-OK status.
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError(f"q must be [B,H,N_q,d] and k, v one [B,H_kv,N_kv,d] shape: {q.shape} {k.shape} {v.shape}")
    if q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3] or q.shape[1] % k.shape[1] != 0:
        raise ValueError(f"incompatible q and k/v shapes: {q.shape} {k.shape}")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    B, H, N_q, d = (int(x) for x in q.shape)
    H_kv, N_kv = int(k.shape[1]), int(k.shape[2])
    if scale is None:
        scale = float(torch.tensor(1.0, dtype=torch.float32) / torch.sqrt(torch.tensor(float(d), dtype=torch.float32)))
    if not math.isfinite(scale):
        raise ValueError("scale must be finite")
    if num_splits is None:
        num_splits = 0  # the library's automatic plan for this device
    with torch.cuda.device(q.device):
        need = fa_fwd_ex_workspace_size(B, H, N_q, N_kv, d, num_splits)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr() if lse is not None else None, B, H, H_kv, N_q, N_kv, d, float(scale),
                       _dtype_code(q) | (FA_FLAG_CAUSAL if causal else 0), num_splits,
                       workspace.data_ptr() if need > 0 else None,
                       workspace.numel() * workspace.element_size() if need > 0 else 0, s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_ex")
    return out, lse


def attention_backward(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
                       dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of O = softmax(scale * Q K^T) V for CUDA
    tensors q, o, dout [B, H, N_q, d] and k, v [B, H_kv, N_kv, d] (bf16 or
    fp16), given the forward's o and fp32 lse [B, H, N_q].  scale defaults to
    1/sqrt(d) in fp32.  `workspace` (uint8, at least fa_bwd_workspace_size
    bytes) is allocated when not given.  Enqueued on `stream` (default:
    PyTorch's current stream); raises FAError on a non-OK status."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError(f"incompatible shapes: q {q.shape} k {k.shape} v {v.shape} o {o.shape} "
                         f"dout {dout.shape}")
    for t in (q, k, v, o, dout, lse):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("every tensor must be a contiguous CUDA tensor")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise TypeError("q, k, v, o, dout must share a dtype")
    if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("lse must be fp32 [B, H, N_q]")
    B, H, N_q, d = (int(x) for x in q.shape)
    H_kv, N_kv = int(k.shape[1]), int(k.shape[2])
    if scale is None:
        scale = float(torch.tensor(1.0, dtype=torch.float32) / torch.sqrt(torch.tensor(float(d), dtype=torch.float32)))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size(B, H, N_q, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, N_q, N_kv,
                    d, float(scale), _dtype_code(q) | (FA_FLAG_CAUSAL if causal else 0),
                    workspace.data_ptr(), workspace.numel() * workspace.element_size(), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv
