// Backward pass, the two memory-bound kernels around the main one:
//   prep: per query row, D_i = dO_i . O_i (the row sum of dP o P that the
//         gradient of the softmax needs, formed from the forward output
//         instead of the N scores), the negated base-2 log-sum-exp, and a
//         zeroed row of the fp32 dQ accumulator;
//   dq:   dQ = scale * accumulator in the input dtype.
#include <cmath>
#include <cstdint>

#include "fa.h"
#include "fa_bwd_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// One warp per padded query row; lane l holds elements [l*D/32, (l+1)*D/32).
template <int D, bool F16>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdPrepParams p) {
    constexpr int kPer = D / 32;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
    const int lane = static_cast<int>(threadIdx.x % 32);
    if (row >= p.rows_pad) return;
    const long long bh = row / p.Nq_pad;
    const int i = static_cast<int>(row % p.Nq_pad);
    // rows of a tile are consecutive (Nq_pad is a multiple of 128)
    float* st = p.stats + (row / 128) * kStatFloatsPerTile + (row % 128);
    if (i >= p.Nq) {  // padding row of the last query tile: weight 0, no gradient
        if (lane == 0) {
            st[0] = -INFINITY;
            st[128] = 0.0f;
        }
        return;
    }
    const size_t r = static_cast<size_t>(bh) * static_cast<size_t>(p.Nq) + static_cast<size_t>(i);
    const uint16_t* o = static_cast<const uint16_t*>(p.o) + r * D + lane * kPer;
    const uint16_t* g = static_cast<const uint16_t*>(p.dout) + r * D + lane * kPer;
    float acc = 0.0f;
    if constexpr (kPer == 4) {
        const uint2 ov = *reinterpret_cast<const uint2*>(o);
        const uint2 gv = *reinterpret_cast<const uint2*>(g);
        acc = widen_lo16<F16>(ov.x) * widen_lo16<F16>(gv.x) + widen_lo16<F16>(ov.x >> 16) * widen_lo16<F16>(gv.x >> 16) +
              widen_lo16<F16>(ov.y) * widen_lo16<F16>(gv.y) + widen_lo16<F16>(ov.y >> 16) * widen_lo16<F16>(gv.y >> 16);
    } else {
        const uint32_t ov = *reinterpret_cast<const uint32_t*>(o);
        const uint32_t gv = *reinterpret_cast<const uint32_t*>(g);
        acc = widen_lo16<F16>(ov) * widen_lo16<F16>(gv) + widen_lo16<F16>(ov >> 16) * widen_lo16<F16>(gv >> 16);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    float* z = p.dq_acc + r * D + lane * kPer;
    if constexpr (kPer == 4)
        *reinterpret_cast<float4*>(z) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    else
        *reinterpret_cast<float2*>(z) = make_float2(0.0f, 0.0f);
    if (lane == 0) {
        const float lse = p.lse[r];
        // a row with no visible key (lse = -inf) gets weight 0 everywhere
        st[0] = (lse == -INFINITY) ? -INFINITY : -lse * 1.4426950408889634f;
        st[128] = acc;
    }
}

// Eight elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdDqParams p) {
    const long long i = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) * 8;
    if (i >= p.n) return;
    const float4 a = *reinterpret_cast<const float4*>(p.dq_acc + i);
    const float4 b = *reinterpret_cast<const float4*>(p.dq_acc + i + 4);
    const float s = p.scale;
    uint4 out;
    out.x = pack_16x2<F16>(a.x * s, a.y * s);
    out.y = pack_16x2<F16>(a.z * s, a.w * s);
    out.z = pack_16x2<F16>(b.x * s, b.y * s);
    out.w = pack_16x2<F16>(b.z * s, b.w * s);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + i) = out;
}

cudaError_t launch_bwd_prep(const BwdPrepParams& p, int d, int dtype, cudaStream_t stream) {
    const unsigned int blocks = static_cast<unsigned int>((p.rows_pad + 7) / 8);
    if (d == 128 && dtype == FA_DTYPE_BF16)
        fa_bwd_prep_kernel<128, false><<<blocks, 256, 0, stream>>>(p);
    else if (d == 64 && dtype == FA_DTYPE_BF16)
        fa_bwd_prep_kernel<64, false><<<blocks, 256, 0, stream>>>(p);
    else if (d == 128 && dtype == FA_DTYPE_F16)
        fa_bwd_prep_kernel<128, true><<<blocks, 256, 0, stream>>>(p);
    else if (d == 64 && dtype == FA_DTYPE_F16)
        fa_bwd_prep_kernel<64, true><<<blocks, 256, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdDqParams& p, int dtype, cudaStream_t stream) {
    const unsigned int blocks = static_cast<unsigned int>((p.n / 8 + 255) / 256);
    if (dtype == FA_DTYPE_BF16)
        fa_bwd_dq_kernel<false><<<blocks, 256, 0, stream>>>(p);
    else if (dtype == FA_DTYPE_F16)
        fa_bwd_dq_kernel<true><<<blocks, 256, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace fa
