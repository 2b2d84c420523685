// C-ABI entry points of the backward pass (declared in include/fa.h):
// argument checks, workspace layout, TMA tensor maps and the three launches
// (prep, main, dQ conversion) on the caller's stream.
#include <cmath>
#include <cstddef>
#include <cstdint>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_bwd_internal.h"
#include "fa_host.h"

using namespace fa::host;

namespace {

constexpr int64_t kInt32Max = 2147483647;
constexpr size_t kWsAlign = 256;

int64_t pad128(int64_t n) { return (n + 127) / 128 * 128; }

// Workspace: [row statistics: 2 floats per padded query row, padded to 256 bytes]
//            [dQ accumulator: B*H*Nq*d fp32]
size_t stats_bytes(int64_t B, int64_t H, int64_t N_q) {
    const size_t n = static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(pad128(N_q)) *
                     2 * sizeof(float);
    return (n + kWsAlign - 1) / kWsAlign * kWsAlign;
}
size_t workspace_bytes(int64_t B, int64_t H, int64_t N_q, int64_t d) {
    return stats_bytes(B, H, N_q) +
           static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(N_q) * static_cast<size_t>(d) *
               sizeof(float);
}

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

namespace fa {
// The argument checks of fa_bwd that concern the tensors: sizes, dtype, flags,
// alignment and overlaps (the outputs dq, dk, dv overlap no input and no other
// output).  The workspace is checked by the caller.
int validate_bwd_tensors(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, const void* dq, const void* dk, const void* dv, int64_t B, int64_t H,
                         int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype_arg) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype_arg & ~(0xFF | FA_FLAG_CAUSAL)) return FA_ERR_INVALID_ARG;  // unknown flag
    const int dtype = dtype_arg & 0xFF;
    // fp32 inputs: the TF32 tensor-core kind takes K-major operands only, and
    // four of the five backward products read an operand MN-major
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (B > INT64_MAX / H) return FA_ERR_INVALID_ARG;
    const int64_t BH = B * H, BHkv = B * H_kv;
    if (BH > INT64_MAX / (N_q + 128) || BH * (N_q + 128) > INT64_MAX / (d * 4)) return FA_ERR_INVALID_ARG;
    if (BHkv > INT64_MAX / N_kv || BHkv * N_kv > INT64_MAX / (d * 4)) return FA_ERR_INVALID_ARG;
    // TMA coordinates are 32-bit; the grid is B * H_kv * ceil(N_kv / 128) CTAs
    if (BH > kInt32Max || N_q > kInt32Max - 128 || N_kv > kInt32Max - 128) return FA_ERR_UNSUPPORTED;
    if (BHkv > kInt32Max / ((N_kv + 127) / 128)) return FA_ERR_UNSUPPORTED;
    if (misaligned16(q) || misaligned16(k) || misaligned16(v) || misaligned16(o) || misaligned16(dout) ||
        misaligned16(dq) || misaligned16(dk) || misaligned16(dv))
        return FA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGNMENT;
    const void* in_ptr[6] = {q, k, v, o, dout, lse};
    size_t in_len[6];
    bwd_tensor_bytes(B, H, H_kv, N_q, N_kv, d, in_len);
    const void* out_ptr[3] = {dq, dk, dv};
    const size_t out_len[3] = {in_len[0], in_len[1], in_len[2]};
    for (int a = 0; a < 3; ++a) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(out_ptr[a], out_len[a], in_ptr[i], in_len[i])) return FA_ERR_INVALID_ARG;
        for (int b2 = a + 1; b2 < 3; ++b2)
            if (overlaps(out_ptr[a], out_len[a], out_ptr[b2], out_len[b2])) return FA_ERR_INVALID_ARG;
    }
    return FA_OK;
}

// Bytes of q, k, v, o, dout, lse (in that order; dq, dk, dv are the sizes of
// q, k, v) for 16-bit inputs.
void bwd_tensor_bytes(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, size_t* len) {
    const size_t qbytes = static_cast<size_t>(B * H * N_q * d * 2);
    const size_t kvbytes = static_cast<size_t>(B * H_kv * N_kv * d * 2);
    len[0] = qbytes;
    len[1] = kvbytes;
    len[2] = kvbytes;
    len[3] = qbytes;
    len[4] = qbytes;
    len[5] = static_cast<size_t>(B * H * N_q) * sizeof(float);
}
}  // namespace fa

namespace {

int validate_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, const void* dq, const void* dk, const void* dv, int64_t B, int64_t H,
                 int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype_arg,
                 const void* workspace, size_t workspace_bytes_given) {
    if (!workspace) return FA_ERR_INVALID_ARG;
    const int st = fa::validate_bwd_tensors(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale,
                                            dtype_arg);
    if (st != FA_OK) return st;
    if (misaligned16(workspace)) return FA_ERR_ALIGNMENT;
    const size_t need = workspace_bytes(B, H, N_q, d);
    if (workspace_bytes_given < need) return FA_ERR_INVALID_ARG;
    // the workspace overlaps no input and no output
    const void* ptr[9] = {q, k, v, o, dout, lse, dq, dk, dv};
    size_t len[9];
    fa::bwd_tensor_bytes(B, H, H_kv, N_q, N_kv, d, len);
    len[6] = len[0];
    len[7] = len[1];
    len[8] = len[2];
    for (int i = 0; i < 9; ++i)
        if (overlaps(workspace, need, ptr[i], len[i])) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

int launch_bwd_all(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                   int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype_arg, void* workspace,
                   void* stream) {
    const int dtype = dtype_arg & 0xFF;
    const bool causal = (dtype_arg & FA_FLAG_CAUSAL) != 0;
    const int64_t BH = B * H, BHkv = B * H_kv;
    const int64_t Nq_pad = pad128(N_q);
    CUtensorMap mq, mk, mv, mdo, mdk, mdv, mdq;
    int st;
    if ((st = encode_map(&mq, q, dtype, BH, N_q, d)) != FA_OK) return st;
    if ((st = encode_map(&mdo, dout, dtype, BH, N_q, d)) != FA_OK) return st;
    if ((st = encode_map(&mk, k, dtype, BHkv, N_kv, d)) != FA_OK) return st;
    if ((st = encode_map(&mv, v, dtype, BHkv, N_kv, d)) != FA_OK) return st;
    if ((st = encode_map(&mdk, dk, dtype, BHkv, N_kv, d)) != FA_OK) return st;
    if ((st = encode_map(&mdv, dv, dtype, BHkv, N_kv, d)) != FA_OK) return st;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* stats = reinterpret_cast<float*>(ws);
    float* dq_acc = reinterpret_cast<float*>(ws + stats_bytes(B, H, N_q));
    if ((st = encode_map(&mdq, dq_acc, FA_DTYPE_F32, BH, N_q, d)) != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    fa::BwdPrepParams pp{};
    pp.o = o;
    pp.dout = dout;
    pp.lse = lse;
    pp.stats = stats;
    pp.dq_acc = dq_acc;
    pp.rows_pad = static_cast<long long>(BH * Nq_pad);
    pp.Nq = static_cast<int>(N_q);
    pp.Nq_pad = static_cast<int>(Nq_pad);
    cudaError_t e = fa::launch_bwd_prep(pp, static_cast<int>(d), dtype, s);
    if (e != cudaSuccess) {
        set_error("backward prep launch", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }

    fa::BwdParams p{};
    p.status = device_status_words(&st);
    if (st != FA_OK) return st;
    p.gen = next_generation();
    p.stats = stats;
    p.Nq = static_cast<int>(N_q);
    p.Nkv = static_cast<int>(N_kv);
    p.Nq_pad = static_cast<int>(Nq_pad);
    p.n_q_tiles = static_cast<int>(Nq_pad / 128);
    p.n_kv_blocks = static_cast<int>((N_kv + 127) / 128);
    p.H = static_cast<int>(H);
    p.H_kv = static_cast<int>(H_kv);
    p.group = static_cast<int>(H / H_kv);
    p.causal = causal ? 1 : 0;
    p.causal_offset = static_cast<int>(N_kv - N_q);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale = scale;
    const unsigned int grid = static_cast<unsigned int>(BHkv * p.n_kv_blocks);
    e = (dtype == FA_DTYPE_BF16)
            ? fa::launch_bwd_bf16(static_cast<int>(d), mq, mk, mv, mdo, mdk, mdv, mdq, p, grid, s)
            : fa::launch_bwd_f16(static_cast<int>(d), mq, mk, mv, mdo, mdk, mdv, mdq, p, grid, s);
    if (e != cudaSuccess) {
        set_error("backward kernel launch", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }

    fa::BwdDqParams dp{};
    dp.dq_acc = dq_acc;
    dp.dq = dq;
    dp.n = static_cast<long long>(BH * N_q * d);
    dp.scale = scale;
    e = fa::launch_bwd_dq(dp, dtype, s);
    if (e != cudaSuccess) {
        set_error("backward dQ conversion launch", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N_q, int64_t d) {
    if (B < 1 || H < 1 || N_q < 1 || (d != 64 && d != 128)) return 0;
    if (B > INT64_MAX / H || B * H > INT64_MAX / (N_q + 128) || B * H * (N_q + 128) > INT64_MAX / (d * 4))
        return 0;
    return workspace_bytes(B, H, N_q, d);
}

int fa_bwd_validate(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                    int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype, const void* workspace,
                    size_t workspace_bytes_given) {
    return validate_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype, workspace,
                        workspace_bytes_given);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
           int64_t d, float scale, int dtype, void* workspace, size_t workspace_bytes_given, void* stream) {
    const int st = validate_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype,
                                workspace, workspace_bytes_given);
    if (st != FA_OK) return st;
    return launch_bwd_all(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype, workspace,
                          stream);
}

}  // extern "C"
