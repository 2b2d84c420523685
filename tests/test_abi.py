"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function include/fa.h declares, and its
argument validation returns the documented status codes before any CUDA
call."""
import ctypes
import math
import subprocess

import pytest

from exact_tiled_attention_04_gb300 import binding as fab


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_04_gb300 import build
    build.build()
    return fab.load()


def test_header_declares_expected_entry_points():
    names = fab.header_functions()
    for n in ("fa_fwd", "fa_fwd_validate", "fa_device_status", "fa_status_string",
              "fa_last_error_message", "fa_version"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fab.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in fab.header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for st in range(6):
        assert fab.fa_status_string(st)
    assert fab.fa_status_string(99) == "unknown status"
    assert fab.fa_version() >= 100


# fake, aligned, non-overlapping device addresses: validation never dereferences
Q, K, V, O, L = 1 << 32, 2 << 32, 3 << 32, 4 << 32, 5 << 32
GOOD = dict(B=2, H=4, N=1000, d=64, scale=0.125, dtype=fab.FA_DTYPE_BF16)


def validate(q=Q, k=K, v=V, o=O, lse=L, **kw):
    a = dict(GOOD)
    a.update(kw)
    return fab.fa_fwd_validate(q, k, v, o, lse, a["B"], a["H"], a["N"], a["d"], a["scale"], a["dtype"])


def test_valid_arguments(lib):
    assert validate() == fab.FA_OK
    assert validate(lse=None) == fab.FA_OK
    assert validate(d=128) == fab.FA_OK
    assert validate(dtype=fab.FA_DTYPE_F32) == fab.FA_OK
    assert validate(scale=0.0) == fab.FA_OK and validate(scale=-3.0) == fab.FA_OK
    # inputs may alias one another
    assert validate(k=Q, v=Q) == fab.FA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), fab.FA_ERR_INVALID_ARG),
    (dict(k=None), fab.FA_ERR_INVALID_ARG),
    (dict(v=None), fab.FA_ERR_INVALID_ARG),
    (dict(o=None), fab.FA_ERR_INVALID_ARG),
    (dict(B=0), fab.FA_ERR_INVALID_ARG),
    (dict(H=-1), fab.FA_ERR_INVALID_ARG),
    (dict(N=0), fab.FA_ERR_INVALID_ARG),
    (dict(scale=math.inf), fab.FA_ERR_INVALID_ARG),
    (dict(scale=math.nan), fab.FA_ERR_INVALID_ARG),
    (dict(d=96), fab.FA_ERR_UNSUPPORTED),
    (dict(d=128, dtype=fab.FA_DTYPE_F32), fab.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fab.FA_ERR_UNSUPPORTED),
    (dict(q=Q + 8), fab.FA_ERR_ALIGNMENT),
    (dict(o=O + 4), fab.FA_ERR_ALIGNMENT),
    (dict(lse=L + 2), fab.FA_ERR_ALIGNMENT),
    (dict(o=Q + 1024), fab.FA_ERR_INVALID_ARG),      # output overlaps an input
    (dict(lse=O + 4096), fab.FA_ERR_INVALID_ARG),    # lse overlaps the output
    (dict(B=1 << 40, H=1 << 30), fab.FA_ERR_INVALID_ARG),  # element count overflows
    (dict(H=1 << 31, B=1), fab.FA_ERR_UNSUPPORTED),  # beyond 32-bit TMA coordinates
])
def test_invalid_arguments(lib, kw, status):
    assert validate(**kw) == status


def test_fa_fwd_rejects_bad_arguments_without_cuda(lib):
    # same checks, same codes, and no CUDA call is made (this machine may
    # have no GPU at all)
    assert fab.fa_fwd(Q, K, V, O, L, 2, 4, 1000, 96, 0.125, fab.FA_DTYPE_BF16, None) == fab.FA_ERR_UNSUPPORTED
    assert fab.fa_fwd(None, K, V, O, L, 2, 4, 1000, 64, 0.125, fab.FA_DTYPE_BF16, None) == fab.FA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(fab, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        fab.load(str(tmp_path / "absent.so"))


def validate_ex(q=Q, k=K, v=V, o=O, lse=L, B=2, H=8, H_kv=2, Nq=1, Nkv=4096, d=128, scale=0.088,
                dtype=fab.FA_DTYPE_BF16, splits=1, ws=None, wbytes=0):
    return fab.fa_fwd_ex_validate(q, k, v, o, lse, B, H, H_kv, Nq, Nkv, d, scale, dtype, splits, ws,
                                  wbytes)


def test_ex_validation(lib):
    WS = 6 << 32
    assert validate_ex() == fab.FA_OK
    assert validate_ex(H_kv=3) == fab.FA_ERR_INVALID_ARG          # 8 query heads, 3 kv heads
    assert validate_ex(H_kv=0) == fab.FA_ERR_INVALID_ARG
    assert validate_ex(Nq=0) == fab.FA_ERR_INVALID_ARG
    assert validate_ex(splits=-1) == fab.FA_ERR_INVALID_ARG
    assert validate_ex(splits=0) == fab.FA_OK  # automatic (no device here: one partition)
    need = fab.fa_fwd_ex_workspace_size(2, 8, 1, 4096, 128, 8)
    assert need == 8 * 2 * 8 * 1 * (128 + 4) * 4
    assert validate_ex(splits=8) == fab.FA_ERR_INVALID_ARG          # workspace missing
    assert validate_ex(splits=8, ws=WS, wbytes=need - 1) == fab.FA_ERR_INVALID_ARG
    assert validate_ex(splits=8, ws=WS, wbytes=need) == fab.FA_OK
    assert validate_ex(splits=8, ws=WS + 8, wbytes=need) == fab.FA_ERR_ALIGNMENT
    assert validate_ex(splits=8, ws=O, wbytes=need) == fab.FA_ERR_INVALID_ARG  # overlaps o


def test_split_planning(lib):
    # capped at one partition per 128 keys and at 32
    assert fab.fa_fwd_ex_workspace_size(1, 1, 10, 200, 64, 8) == 2 * 10 * 68 * 4
    assert fab.fa_fwd_ex_workspace_size(1, 1, 10, 100, 64, 8) == 0
    assert fab.fa_fwd_ex_workspace_size(1, 1, 10, 1 << 20, 64, 64) == 32 * 10 * 68 * 4
    # no empty partition: 5 tiles in 4 requested -> 3 partitions of 2, 2, 1 tiles
    assert fab.fa_fwd_ex_workspace_size(1, 1, 1, 5 * 128, 64, 4) == 3 * 1 * 68 * 4
    assert fab.fa_fwd_ex_splits(1, 1, 1, 512, 512, 152) == 4        # 2 CTAs; capped at 4 key tiles
    assert fab.fa_fwd_ex_splits(2, 32, 32, 8192, 8192, 152) == 1    # 2048 CTAs fill the GPU
    assert fab.fa_fwd_ex_splits(2, 4, 4, 1000, 1000, 152) == 4
    # packed grouped heads: one CTA per key/value head
    assert fab.fa_fwd_ex_splits(8, 32, 8, 1, 16384, 152) == 2       # 64 CTAs
    assert fab.fa_fwd_ex_splits(8, 32, 32, 1, 16384, 152) == 1      # no grouping: 256 CTAs
    assert fab.fa_fwd_ex_splits(1, 8, 2, 64, 4096, 152) == 16       # 64 x 4 rows > 128: 8 CTAs; 19 wanted, 2 of 32 tiles each


def test_launch_counts(lib):
    bf16 = fab.FA_DTYPE_BF16
    # explicit partitions: one launch, or the split launch and its merge
    assert fab.fa_fwd_ex_launches(1, 1, 1, 100, 1000, 64, bf16, 1) == 1
    assert fab.fa_fwd_ex_launches(1, 1, 1, 100, 1000, 64, bf16, 4) == 2
    assert fab.fa_fwd_ex_launches(1, 1, 1, 100, 100, 64, bf16, 4) == 1   # one key tile: no split
    # automatic plan without a device to ask: one partition
    assert fab.fa_fwd_ex_launches(2, 32, 32, 8192, 8192, 128, bf16, 0) == 1
    assert fab.fa_fwd_launches(2, 32, 8192, 128, bf16) == 1
    assert fab.fa_fwd_launches(0, 32, 8192, 128, bf16) == 0
    # invalid sizes
    assert fab.fa_fwd_ex_launches(1, 3, 2, 100, 100, 64, bf16, 1) == 0
    assert fab.fa_fwd_ex_launches(1, 1, 1, 100, 100, 64, bf16, -1) == 0
    assert fab.fa_fwd_ex_launches(0, 1, 1, 100, 100, 64, bf16, 1) == 0


def test_dtype_flags(lib):
    assert validate(dtype=fab.FA_DTYPE_F16) == fab.FA_OK
    assert validate(dtype=fab.FA_DTYPE_F16, d=128) == fab.FA_OK
    assert validate(dtype=fab.FA_DTYPE_F16, d=96) == fab.FA_ERR_UNSUPPORTED
    assert validate(dtype=fab.FA_DTYPE_BF16 | fab.FA_FLAG_CAUSAL) == fab.FA_OK
    assert validate(dtype=fab.FA_DTYPE_BF16 | 0x200) == fab.FA_ERR_INVALID_ARG  # unknown flag
    assert validate_ex(dtype=fab.FA_DTYPE_F16 | fab.FA_FLAG_CAUSAL) == fab.FA_OK


def validate_bwd(q=Q, k=K, v=V, o=O, dout=6 << 32, lse=L, dq=7 << 32, dk=8 << 32, dv=9 << 32, B=2, H=8,
                 H_kv=2, Nq=300, Nkv=333, d=64, scale=0.125, dtype=fab.FA_DTYPE_BF16, ws=10 << 32,
                 wbytes=None):
    if wbytes is None:
        wbytes = fab.fa_bwd_workspace_size(B, H, Nq, d)
    return fab.fa_bwd_validate(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, Nq, Nkv, d, scale, dtype,
                               ws, wbytes)


def test_bwd_validation(lib):
    # statistics: 8 bytes per padded query row (3 tiles of 128), then fp32 dQ
    assert fab.fa_bwd_workspace_size(2, 8, 300, 64) == 2 * 8 * 384 * 8 + 2 * 8 * 300 * 64 * 4
    assert fab.fa_bwd_workspace_size(1, 1, 1, 96) == 0
    assert validate_bwd() == fab.FA_OK
    assert validate_bwd(dtype=fab.FA_DTYPE_F16 | fab.FA_FLAG_CAUSAL, d=128) == fab.FA_OK
    assert validate_bwd(dtype=fab.FA_DTYPE_F32) == fab.FA_ERR_UNSUPPORTED
    assert validate_bwd(d=96) == fab.FA_ERR_UNSUPPORTED
    assert validate_bwd(dtype=fab.FA_DTYPE_BF16 | 0x200) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(H_kv=3) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(lse=None) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(ws=None) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(wbytes=fab.fa_bwd_workspace_size(2, 8, 300, 64) - 1) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(dq=(7 << 32) + 8) == fab.FA_ERR_ALIGNMENT
    assert validate_bwd(ws=(10 << 32) + 4) == fab.FA_ERR_ALIGNMENT
    assert validate_bwd(lse=L + 2) == fab.FA_ERR_ALIGNMENT
    assert validate_bwd(dk=Q + 64) == fab.FA_ERR_INVALID_ARG     # output overlaps an input
    assert validate_bwd(dv=8 << 32) == fab.FA_ERR_INVALID_ARG    # dv overlaps dk
    assert validate_bwd(ws=O) == fab.FA_ERR_INVALID_ARG          # workspace overlaps o
    assert validate_bwd(scale=float("nan")) == fab.FA_ERR_INVALID_ARG
    assert validate_bwd(k=Q, v=Q) == fab.FA_OK                   # inputs may alias
    # rejected before any CUDA call
    assert fab.fa_bwd(Q, K, V, O, 6 << 32, L, 7 << 32, 8 << 32, 9 << 32, 2, 8, 2, 300, 333, 96, 0.125,
                      fab.FA_DTYPE_BF16, 10 << 32, 1 << 30, None) == fab.FA_ERR_UNSUPPORTED


def test_host_pipeline_validation(lib):
    code = fab.FA_DTYPE_BF16
    need = fab.fa_fwd_host_workspace_size(2, 8, 2, 300, 300, 128, code)
    assert need > 0 and fab.fa_fwd_host_workspace_size(2, 8, 3, 300, 300, 128, code) == 0
    WS = 6 << 32
    args = (Q, K, V, O, L, 2, 8, 2, 300, 300, 128, 0.088, code)
    # rejected before any CUDA call
    assert fab.fa_fwd_host(*args, None, need, None) == fab.FA_ERR_INVALID_ARG
    assert fab.fa_fwd_host(*args, WS, need - 1, None) == fab.FA_ERR_INVALID_ARG
    assert fab.fa_fwd_host(*args, WS + 16, need, None) == fab.FA_ERR_ALIGNMENT
    assert fab.fa_fwd_host(Q, K, V, O, L, 2, 8, 2, 300, 300, 96, 0.088, code, WS, need, None) == \
        fab.FA_ERR_UNSUPPORTED


def test_host_pipeline_workspace_is_checked_with_its_own_size(lib):
    """The host pipelines check their device workspace with the size they
    need, not the workspace of the device entry point on the whole problem
    (a different size): a tensor placed right after the pipeline workspace
    is accepted, one that reaches into its last bytes is rejected."""
    B, H, N, d = 2, 32, 8192, 128
    code = fab.FA_DTYPE_BF16
    need = fab.fa_bwd_host_workspace_size(B, H, H, N, N, d)
    assert 0 < need and need != fab.fa_bwd_workspace_size(B, H, N, d)
    qb = B * H * N * d * 2
    lb = B * H * N * 4
    ws = 1 << 40
    # q, k, v, o, dout, lse, dq, dk, dv one after another, the first one
    # `start` bytes after the workspace
    def ptrs(start):
        sizes = [qb] * 5 + [lb] + [qb] * 3
        out, a = [], ws + start
        for sz in sizes:
            out.append(a)
            a += (sz + 255) // 256 * 256
        return out
    overlapping = ptrs(need - 256)
    assert fab.fa_bwd_host(*overlapping, B, H, H, N, N, d, 0.088, code, ws, need, None) == fab.FA_ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("the accepted case would run the pipeline on fake host pointers")
    adjacent = ptrs(need)
    assert fab.fa_bwd_host(*adjacent, B, H, H, N, N, d, 0.088, code, ws, need, None) == fab.FA_ERR_CUDA
