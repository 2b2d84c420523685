// Merge of key-partition partial results (split-KV launches).
//
// A split launch sweeps disjoint key ranges of one query row in different
// CTAs; each leaves an unnormalised accumulator O_s relative to its own
// reference maximum m_s (base-2, scaled units) and the sums l_s (fp32
// weights) and lq_s (weights as normalised in the fused kernel).  They combine
// exactly like consecutive tiles of the online softmax ("FlashAttention
// dissected", section "The mathematical breakthrough: Tiling and Online
// Softmax": rescale by the correction factor e^(m_s - m_new) and add; section
// "Interaction with the KV cache during inference": FlashDecoding splits the
// key sequence across cores):
//   M = max_s m_s,  w_s = 2^(m_s - M),
//   O = sum_s w_s O_s / sum_s w_s lq_s,   lse = ln 2 * (M + log2 sum_s w_s l_s).
// One warp per query row; lane s holds partition s's statistics (at most 32
// partitions), lanes split the head dimension for the weighted sum.
#include <cmath>
#include <cstdint>

#include "fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D, int kDtype>
__global__ void __launch_bounds__(256) fa_merge_kernel(const MergeParams m) {
    constexpr int kPer = D / 32;  // columns per lane
    const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
    const int lane = static_cast<int>(threadIdx.x % 32);
    if (row >= m.rows) return;
    const size_t slab = static_cast<size_t>(m.rows);

    float ms = -INFINITY, ls = 0.0f, lqs = 0.0f;
    if (lane < m.splits) {
        const float4 st = *reinterpret_cast<const float4*>(m.ml_part + (static_cast<size_t>(lane) * slab + row) * 4);
        ms = st.x;
        ls = st.y;
        lqs = st.z;
    }
    float M = ms;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float mref = (M == -INFINITY) ? 0.0f : M;
    const float ws = (lane < m.splits) ? ex2(ms - mref) : 0.0f;
    float L = ws * ls, LQ = ws * lqs;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, off);
        LQ += __shfl_xor_sync(0xffffffffu, LQ, off);
    }

    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.0f;
    for (int sp = 0; sp < m.splits; ++sp) {
        const float w = __shfl_sync(0xffffffffu, ws, sp);
        if (w == 0.0f) continue;  // a partition with no visible key (its O slot is not written)
        const float* src = m.o_part + (static_cast<size_t>(sp) * slab + row) * D + lane * kPer;
        if constexpr (kPer == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        }
    }
    const float inv = LQ > 0.0f ? 1.0f / LQ : 0.0f;
    const size_t out = static_cast<size_t>(row) * D + lane * kPer;
    if constexpr (kDtype == FA_DTYPE_BF16 || kDtype == FA_DTYPE_F16) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(m.o) + out);
#pragma unroll
        for (int i = 0; i < kPer; i += 2)
            dst[i / 2] = pack_16x2<kDtype == FA_DTYPE_F16>(acc[i] * inv, acc[i + 1] * inv);
    } else {
        float* dst = static_cast<float*>(m.o) + out;
#pragma unroll
        for (int i = 0; i < kPer; ++i) dst[i] = acc[i] * inv;
    }
    if (m.lse != nullptr && lane == 0)
        m.lse[row] = (L > 0.0f) ? (mref + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

cudaError_t launch_merge(const MergeParams& m, int d, int dtype, cudaStream_t stream) {
    const unsigned int blocks = static_cast<unsigned int>((m.rows + 7) / 8);
    if (d == 128 && dtype == FA_DTYPE_BF16)
        fa_merge_kernel<128, FA_DTYPE_BF16><<<blocks, 256, 0, stream>>>(m);
    else if (d == 64 && dtype == FA_DTYPE_BF16)
        fa_merge_kernel<64, FA_DTYPE_BF16><<<blocks, 256, 0, stream>>>(m);
    else if (d == 64 && dtype == FA_DTYPE_F32)
        fa_merge_kernel<64, FA_DTYPE_F32><<<blocks, 256, 0, stream>>>(m);
    else if (d == 128 && dtype == FA_DTYPE_F16)
        fa_merge_kernel<128, FA_DTYPE_F16><<<blocks, 256, 0, stream>>>(m);
    else if (d == 64 && dtype == FA_DTYPE_F16)
        fa_merge_kernel<64, FA_DTYPE_F16><<<blocks, 256, 0, stream>>>(m);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace fa
