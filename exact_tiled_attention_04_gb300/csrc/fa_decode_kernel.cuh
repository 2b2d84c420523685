// Forward kernel for short query blocks (decode steps), sm_103a.
//
// What it computes is the forward pass of fa_fwd_kernel.cuh (the online
// softmax of "FlashAttention dissected", section "Algorithmic core in
// pseudocode", with the key partitions of its section "Interaction with the
// KV cache during inference") for the case where the query rows of one
// key/value head, R = N_q x (H / H_kv) of them, number at most 32.  In the
// general kernel a 128-row query tile then holds mostly padding, and every
// key tile costs a full 128 x 128 softmax for those few rows.
//
// Here the products are transposed so that the keys, not the query rows,
// sit on the 128 tensor-memory lanes:
//   S^T = K_j Q^T      (128 keys x NR rows, NR = R rounded up to 16 or 32)
//   O^T += V_j^T P^T   (d x NR; at d = 64 the MMA's M of 128 is padded with
//                       rows that are never read)
// so thread t of the softmax warpgroup owns key t of every tile and
// exponentiates NR scores per tile instead of 128.  The reference maxima
// (one per query row) are shared by the whole warpgroup: a tile whose
// scores exceed a row's reference by more than 8 (base 2) triggers, through
// one barrier vote, a reduction of the tile's row maxima across the 128
// threads and a rescale of O^T, l and lq; other tiles need no cross-thread
// step.  The sums l (exact weights, for lse) and lq (the weights as rounded
// for the product, which normalises O) are kept per thread and reduced once
// at the end.
//
// Organisation (one CTA = one key/value head and key partition, 192 threads):
//   warps 0-3  softmax warpgroup (thread t = TMEM lane t)
//   warp 4     tensor-core issuer (one thread) and TMEM owner
//   warp 5     TMA producer (one thread; the warp zeroes the padding rows)
// Tensor memory: S^T in two buffers of NR columns, O^T in NR columns.
// Shared memory: the V ring, the K ring, Q (NR rows), P^T in two buffers
// (NR rows x 128 keys, 16-bit, K-major), reduction scratch, mbarriers.
// Tensor-core order: S(0), S(1); then per tile j: O^T += V_j^T P^T(j) once
// P(j) is written, then S(j + 2) into S(j)'s buffer.
//
// Every mbarrier wait is bounded (the forward kernel's wait_phase), and the
// softmax warpgroup's named barriers are reached by all of its threads on
// every path: a failed wait is carried into the next vote and the
// warpgroup leaves its loop together.
#pragma once

#include <cmath>
#include <cstdint>

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kDecThreads = 192;
constexpr int kDecMmaWarp = 4;
constexpr int kDecLoadWarp = 5;
constexpr uint32_t kDecNamedBar = 1;  // the softmax warpgroup's named barrier

template <int D, bool F16, int NR>
struct DecCfg {
    static_assert(NR == 16 || NR == 32, "rows per CTA: 16 or 32");
    static constexpr int kAtomElems = 64;
    static constexpr int kAtoms = D / kAtomElems;
    static constexpr int kAtomBytes = 128 * 128;              // 128 keys x 128 bytes
    static constexpr int kTileBytes = kAtoms * kAtomBytes;    // 128 keys x D
    static constexpr int kRowAtomBytes = NR * 128;            // NR rows x 128 bytes
    static constexpr int kUmmaK = 16;
    static constexpr int kQkSteps = D / kUmmaK;
    static constexpr int kPvSteps = 128 / kUmmaK;
    static constexpr int kStages = D == 128 ? 3 : 6;          // K+V stages
    static constexpr uint32_t kFmt = F16 ? 0u : 1u;
    static constexpr uint32_t kIdescQK = instr_desc(kFmt, false, false, 128, NR);  // S^T = K Q^T
    static constexpr uint32_t kIdescPV = instr_desc(kFmt, true, false, 128, NR);   // O^T += V^T P^T
    // tensor memory
    static constexpr uint32_t kColS = 0;                      // [2] x NR
    static constexpr uint32_t kColO = 2 * NR;                 // NR
    static constexpr uint32_t kTmemCols = 3 * NR <= 64 ? 64 : 128;
    // shared memory; V first: at d = 64 the padded half of V^T is read
    // 16 KB past a V tile, which stays inside the V and K rings
    static constexpr int kOffV = 0;                                       // [kStages]
    static constexpr int kOffK = kOffV + kStages * kTileBytes;            // [kStages]
    static constexpr int kOffQ = kOffK + kStages * kTileBytes;            // kAtoms x NR rows
    static constexpr int kOffP = kOffQ + kAtoms * kRowAtomBytes;          // [2] x 2 atoms x NR rows
    static constexpr int kOffRed = kOffP + 2 * 2 * kRowAtomBytes;         // float [3][4 warps][NR]
    static constexpr int kOffBar = kOffRed + 3 * 4 * NR * 4;
    // barriers
    static constexpr int kBarQFull = 0;                   // Q landed (TMA) and padding zeroed
    static constexpr int kBarFull = 1;                    // [kStages] K and V of a tile landed
    static constexpr int kBarEmpty = kBarFull + kStages;  // [kStages] both consumed
    static constexpr int kBarS = kBarEmpty + kStages;     // [2] S^T buffer ready
    static constexpr int kBarP = kBarS + 2;               // [2] P^T buffer written (4 warps)
    static constexpr int kBarPFree = kBarP + 2;           // [2] the product reading it is done
    static constexpr int kBarO = kBarPFree + 2;           // every product done
    static constexpr int kBarDrain = kBarO + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemUsed = kOffAbort + 4;
    static constexpr size_t kSmemBytes = static_cast<size_t>(kSmemUsed) + 1024;  // alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
    static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "operand tiles must be 1024-byte aligned");
};

// NR consecutive TMEM columns of this warp's 32 lanes (one per thread).
template <int NR>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[NR]) {
    if constexpr (NR == 32) {
        tmem_ld32(taddr, r);
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
              "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
}
// Wait for this thread's outstanding tcgen05.ld; the registers are named so
// that no use of them is scheduled above the wait.
template <int NR>
__device__ __forceinline__ void tmem_ld_cols_wait(uint32_t (&r)[NR]) {
    if constexpr (NR == 32) {
        tmem_ld_wait(r);
    } else {
        asm volatile("tcgen05.wait::ld.sync.aligned;"
                     : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                       "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                       "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                     :
                     : "memory");
    }
}
template <int NR>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[NR]) {
    if constexpr (NR == 32) {
        tmem_st32(taddr, r);
    } else {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
            "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
            "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
            : "memory");
    }
}

// OR of a predicate over the `nthreads` threads of named barrier `id`
// (every one of them must call it).
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0u;
}

// Reduce-scatter of NR values per lane across the 32 lanes of a warp (max
// or sum): each exchange step halves the values a lane keeps, so NR - 1
// shuffles (plus 32 / NR - 1 plain ones) leave lane L holding the
// warp-wide result for row L / (32 / NR).
template <int NR, bool kMax>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[NR], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
    for (int cnt = NR, o = 16; cnt > 1; cnt /= 2, o /= 2) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < cnt / 2; ++i) {
            const float send = upper ? v[i] : v[i + cnt / 2];
            const float keep = upper ? v[i + cnt / 2] : v[i];
            v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
#pragma unroll
    for (int o = 16 / NR; o >= 1; o /= 2) v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
    return v[0];
}

// One CTA per (key/value head, key partition): grid = B * H_kv * p.splits.
// The key/value head's p.Nq * p.group <= NR query rows are row n = g * Nq + i
// (query head g of the group, query index i); their outputs are the rows
// kvh * Nq * group + n of [B*H, Nq].
template <int D, bool F16, bool kCausal, int NR>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
    using C = DecCfg<D, F16, NR>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_u32 + pad;

    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;
    const unsigned int split = blockIdx.x % static_cast<unsigned>(p.splits);
    const int kvh = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.splits));  // b * H_kv + key/value head
    const int rows = p.Nq * p.group;
    // key tiles any row sees (causal: up to the last query's diagonal)
    int n_tiles = p.n_kv_tiles;
    if (kCausal) {
        const long long lim = min(static_cast<long long>(p.Nkv), static_cast<long long>(p.Nq) + p.causal_offset);
        n_tiles = lim <= 0 ? 0 : static_cast<int>((lim + 127) / 128);
    }
    const int t_begin = static_cast<int>(split) * p.tiles_per_split;
    const int T = max(0, min(p.tiles_per_split, n_tiles - t_begin));
    const bool has_work = T > 0;

    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarQFull), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarFull + s), 1);
            mbar_init(bar(C::kBarEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::kBarS + b), 1);
            mbar_init(bar(C::kBarP + b), 4);
            mbar_init(bar(C::kBarPFree + b), 1);
        }
        mbar_init(bar(C::kBarO), 1);
        mbar_init(bar(C::kBarDrain), 1);
        *abort_flag = (*reinterpret_cast<volatile unsigned int*>(&p.status->abort_gen) == p.gen) ? 1u : 0u;
        mbar_init_fence();
    }
    if (warp == kDecMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0u;  // an earlier CTA of this launch gave up

    if (skip) {
        // nothing (the device error word already reports the failure)
    } else if (warp == kDecLoadWarp) {
        // ---------------------------------------------------------- producer
        if (has_work) {
            // Q rows rows .. NR-1 are zero (whole 128-byte rows, so the
            // swizzle does not matter), then rows 0 .. rows-1 by TMA
            for (int a = 0; a < C::kAtoms; ++a) {
                uint4* q4 = reinterpret_cast<uint4*>(smem + C::kOffQ + a * C::kRowAtomBytes);
                for (int i = rows * 8 + lane; i < NR * 8; i += 32) q4[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        if (has_work && lane == 0) {
            const uint64_t once = policy_evict_first();  // every byte here is read once
            mbar_arrive_expect_tx(bar(C::kBarQFull), static_cast<uint32_t>(C::kAtoms * rows * 128));
            for (int a = 0; a < C::kAtoms; ++a)
                tma_load_3d(sbase + C::kOffQ + a * C::kRowAtomBytes, &map_q, bar(C::kBarQFull), a * C::kAtomElems,
                            0, kvh * p.group, once);
            int issued = 0;
            for (int j = 0; j < T; ++j) {
                const int s = j % C::kStages;
                if (!wait_phase(bar(C::kBarEmpty + s), ((j / C::kStages) & 1) ^ 1, abort_flag, p, 60)) break;
                mbar_arrive_expect_tx(bar(C::kBarFull + s), 2u * C::kTileBytes);
                const int key0 = (t_begin + j) * 128;
                for (int a = 0; a < C::kAtoms; ++a) {
                    tma_load_3d(sbase + C::kOffK + s * C::kTileBytes + a * C::kAtomBytes, &map_k,
                                bar(C::kBarFull + s), a * C::kAtomElems, key0, kvh, once);
                    tma_load_3d(sbase + C::kOffV + s * C::kTileBytes + a * C::kAtomBytes, &map_v,
                                bar(C::kBarFull + s), a * C::kAtomElems, key0, kvh, once);
                }
                issued = j + 1;
            }
            // every issued load has landed before the CTA may exit
            for (int s = 0; s < C::kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
                wait_phase(bar(C::kBarFull + s), (last / C::kStages) & 1, abort_flag, p, 61, false);
            }
        }
    } else if (warp == kDecMmaWarp) {
        // ------------------------------------------------------------ issuer
        if (has_work && lane == 0) {
            const uint32_t sQ = sbase + C::kOffQ;
            auto issue_s = [&](int j) {  // S^T(j) = K_j Q^T into buffer j & 1
                const uint32_t sK = sbase + C::kOffK + (j % C::kStages) * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < C::kQkSteps; ++kk) {
                    const uint32_t koff = (kk * 32) / 128 * C::kAtomBytes + (kk * 32) % 128;
                    const uint32_t qoff = (kk * 32) / 128 * C::kRowAtomBytes + (kk * 32) % 128;
                    mma_ss<false>(tmem + C::kColS + NR * (j & 1), smem_desc_sw128(sK + koff, 16, 1024),
                                  smem_desc_sw128(sQ + qoff, 16, 1024), C::kIdescQK, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(C::kBarS + (j & 1)));
            };
            bool ok = wait_phase(bar(C::kBarQFull), 0, abort_flag, p, 62);
            for (int j = 0; ok && j < 2 && j < T; ++j) {
                ok = wait_phase(bar(C::kBarFull + j % C::kStages), (j / C::kStages) & 1, abort_flag, p, 63);
                if (!ok) break;
                tc_fence_after();
                issue_s(j);
            }
            for (int j = 0; ok && j < T; ++j) {
                const int b = j & 1;
                ok = wait_phase(bar(C::kBarP + b), (j >> 1) & 1, abort_flag, p, 64);
                if (!ok) break;
                tc_fence_after();
                // O^T += V_j^T P^T(j): A = V_j read MN-major (d contiguous, its
                // two 64-element blocks 16 KB apart), B = P^T K-major
                const uint32_t sV = sbase + C::kOffV + (j % C::kStages) * C::kTileBytes;
                const uint32_t sP = sbase + C::kOffP + b * 2 * C::kRowAtomBytes;
#pragma unroll
                for (int kk = 0; kk < C::kPvSteps; ++kk) {
                    const uint32_t poff = (kk * 32) / 128 * C::kRowAtomBytes + (kk * 32) % 128;
                    mma_ss<false>(tmem + C::kColO, smem_desc_sw128(sV + kk * C::kUmmaK * 128, C::kAtomBytes, 1024),
                                  smem_desc_sw128(sP + poff, 16, 1024), C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(C::kBarPFree + b));
                tc_commit(bar(C::kBarEmpty + j % C::kStages));  // K_j and V_j are no longer read
                if (j + 2 < T) {
                    ok = wait_phase(bar(C::kBarFull + (j + 2) % C::kStages), ((j + 2) / C::kStages) & 1, abort_flag,
                                    p, 63);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j + 2);  // buffer b: S^T(j) was read before P(j) was published
                }
            }
            if (ok) tc_commit(bar(C::kBarO));
            tc_commit(bar(C::kBarDrain));
            wait_phase(bar(C::kBarDrain), 0, abort_flag, p, 65, false);
        }
    } else {
        // ------------------------------------------------ softmax warpgroup
        const int t = static_cast<int>(threadIdx.x);  // key t of each tile; lane t of O^T in the epilogue
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS;
        const uint32_t tO = tmem + lane_base + C::kColO;
        const float c = p.scale_log2;
        float* red = reinterpret_cast<float*>(smem + C::kOffRed);  // [3][4 warps][NR]
        constexpr int kLanesPerRow = 32 / NR;                      // after warp_reduce_rows
        // key t's 16-bit slot in row n of a P^T buffer: atom t / 64, byte
        // 2 (t % 64) of the row, whose 16-byte chunks are permuted by n % 8
        const int pch = (t % 64) / 8;
        uint8_t* pkey = smem + C::kOffP + (t / 64) * C::kRowAtomBytes + (t % 8) * 2;

        float m[NR], l[NR], lq[NR];  // reference maxima (base 2, scaled), sums
#pragma unroll
        for (int n = 0; n < NR; ++n) {
            m[n] = -INFINITY;
            l[n] = 0.0f;
            lq[n] = 0.0f;
        }
        // is key `key` visible to row n (padding rows see every key)
        auto visible = [&](int n, int key) -> bool {
            if (key >= p.Nkv) return false;
            if (kCausal && n < rows) return key <= n % p.Nq + p.causal_offset;
            return true;
        };
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const int b = j & 1;
            const int key0 = (t_begin + j) * 128;
            const int key = key0 + t;
            // a tile with a key some row may not see: the partial last tile,
            // or (causal) keys past the first row's diagonal
            const bool masked = key0 + 128 > p.Nkv || (kCausal && key0 + 127 > p.causal_offset);
            uint32_t s[NR];
            if (ok) ok = wait_phase(bar(C::kBarS + b), (j >> 1) & 1, abort_flag, p, 66);
            ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-wide
            if (ok) {
                tc_fence_after();
                tmem_ld_cols<NR>(tS + NR * b, s);
                tmem_ld_cols_wait<NR>(s);
            } else {
#pragma unroll
                for (int n = 0; n < NR; ++n) s[n] = 0u;
            }
            // x = t - m: the exponent of each weight against the current reference
            float x[NR];
            bool need = j == 0 || !ok;
#pragma unroll
            for (int n = 0; n < NR; ++n) {
                x[n] = fmaf(u2f(s[n]), c, -m[n]);
                if (masked && !visible(n, key)) x[n] = -INFINITY;
                need |= x[n] > kRescaleThreshold;
            }
            if (named_barrier_or(kDecNamedBar, 128, need)) {
                if (named_barrier_or(kDecNamedBar, 128, !ok)) {  // every thread leaves together
                    ok = false;
                    break;
                }
                // the tile's row maxima over its 128 keys
                float v[NR];
#pragma unroll
                for (int n = 0; n < NR; ++n) v[n] = (masked && !visible(n, key)) ? -INFINITY : u2f(s[n]) * c;
                const float r = warp_reduce_rows<NR, true>(v, lane);
                if (lane % kLanesPerRow == 0) red[warp * NR + lane / kLanesPerRow] = r;
                named_barrier_sync(kDecNamedBar, 128);
                float alpha[NR];
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    const float tmax = fmaxf(fmaxf(red[n], red[NR + n]), fmaxf(red[2 * NR + n], red[3 * NR + n]));
                    float mn = fmaxf(m[n], tmax);
                    if (mn == -INFINITY) mn = 0.0f;  // no visible key yet: any finite reference
                    alpha[n] = ex2(m[n] - mn);      // 0 while m was -inf
                    l[n] *= alpha[n];
                    lq[n] *= alpha[n];
                    m[n] = mn;
                    x[n] = (masked && !visible(n, key)) ? -INFINITY : fmaf(u2f(s[n]), c, -mn);
                }
                if (j > 0) {  // O^T holds tiles < j: rescale it once the last product into it is done
                    ok = __all_sync(0xffffffffu,
                                    wait_phase(bar(C::kBarPFree + (b ^ 1)), ((j - 1) >> 1) & 1, abort_flag, p, 67));
                    if (ok) {
                        tc_fence_after();
                        uint32_t o[NR];
                        tmem_ld_cols<NR>(tO, o);
                        tmem_ld_cols_wait<NR>(o);
#pragma unroll
                        for (int n = 0; n < NR; ++n) o[n] = f2u(u2f(o[n]) * alpha[n]);
                        tmem_st_cols<NR>(tO, o);
                        tmem_st_wait();
                    }
                }
            }
            // P^T buffer b was last read by the product of tile j - 2
            if (ok && j >= 2) ok = wait_phase(bar(C::kBarPFree + b), ((j - 2) >> 1) & 1, abort_flag, p, 68);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                uint8_t* pbuf = pkey + b * 2 * C::kRowAtomBytes;
#pragma unroll
                for (int n = 0; n < NR; n += 2) {
                    const float p0 = ex2(x[n]), p1 = ex2(x[n + 1]);
                    l[n] += p0;
                    l[n + 1] += p1;
                    const uint32_t w2 = pack_16x2<F16>(p0, p1);
                    lq[n] += widen_lo16<F16>(w2);
                    lq[n + 1] += widen_lo16<F16>(w2 >> 16);
                    *reinterpret_cast<uint16_t*>(pbuf + n * 128 + ((pch ^ (n & 7)) << 4)) =
                        static_cast<uint16_t>(w2 & 0xFFFFu);
                    *reinterpret_cast<uint16_t*>(pbuf + (n + 1) * 128 + ((pch ^ ((n + 1) & 7)) << 4)) =
                        static_cast<uint16_t>(w2 >> 16);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarP + b));
            }
        }

        // ------------------------------------------------------- epilogue
        if (ok && has_work) ok = wait_phase(bar(C::kBarO), 0, abort_flag, p, 69);
        ok = __all_sync(0xffffffffu, ok);
        if (!named_barrier_or(kDecNamedBar, 128, !ok)) {
            tc_fence_after();
            // l and lq over the 128 keys of the warpgroup
            {
                float v[NR], w[NR];
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    v[n] = l[n];
                    w[n] = lq[n];
                }
                const float rl = warp_reduce_rows<NR, false>(v, lane);
                const float rq = warp_reduce_rows<NR, false>(w, lane);
                if (lane % kLanesPerRow == 0) {
                    red[4 * NR + warp * NR + lane / kLanesPerRow] = rl;
                    red[8 * NR + warp * NR + lane / kLanesPerRow] = rq;
                }
            }
            named_barrier_sync(kDecNamedBar, 128);
            float L[NR], LQ[NR];
#pragma unroll
            for (int n = 0; n < NR; ++n) {
                const float* rl = red + 4 * NR + n;
                const float* rq = red + 8 * NR + n;
                L[n] = (rl[0] + rl[NR]) + (rl[2 * NR] + rl[3 * NR]);
                LQ[n] = (rq[0] + rq[NR]) + (rq[2 * NR] + rq[3 * NR]);
            }
            uint32_t o[NR];
            if (has_work) {
                tmem_ld_cols<NR>(tO, o);
                tmem_ld_cols_wait<NR>(o);
            } else {
#pragma unroll
                for (int n = 0; n < NR; ++n) o[n] = 0u;
            }
            const long long row0 = static_cast<long long>(kvh) * rows;  // output row of row 0
            if (p.splits > 1) {
                // unnormalised partial of this key partition (the merge's input);
                // a row with no visible key gets weight 0 there (m = -inf)
                const size_t slab = static_cast<size_t>(gridDim.x / p.splits) * rows;
                const size_t r0 = split * slab + static_cast<size_t>(row0);
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    if (n < rows) {
                        if (t < D) p.o_part[(r0 + n) * D + t] = u2f(o[n]);
                        if (t == n)
                            *reinterpret_cast<float4*>(p.ml_part + (r0 + n) * 4) =
                                make_float4(L[n] > 0.0f ? m[n] : -INFINITY, L[n], LQ[n], 0.0f);
                    }
                }
            } else {
                uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    if (n < rows) {
                        const float inv = LQ[n] > 0.0f ? 1.0f / LQ[n] : 0.0f;
                        if (t < D)
                            out[(row0 + n) * D + t] =
                                static_cast<uint16_t>(pack_16x2<F16>(u2f(o[n]) * inv, 0.0f) & 0xFFFFu);
                        if (t == n && p.lse != nullptr)
                            p.lse[row0 + n] =
                                L[n] > 0.0f ? (m[n] + log2f(L[n])) * 0.69314718055994531f : -INFINITY;
                    }
                }
            }
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kDecMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool F16, bool kCausal, int NR>
cudaError_t launch_decode_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const FwdParams& p, unsigned int grid, cudaStream_t stream) {
    using C = DecCfg<D, F16, NR>;
    auto kern = fa_decode_kernel<D, F16, kCausal, NR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecThreads, C::kSmemBytes, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

// Rows per CTA (p.Nq * p.group) <= 32; q over [B*H, Nq, d] with boxes of
// Nq rows x group heads; k, v over [B*H_kv, Nkv, d].
template <int D, bool F16>
cudaError_t launch_decode(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p,
                          unsigned int grid, cudaStream_t stream) {
    const int rows = p.Nq * p.group;
    if (rows <= 16)
        return p.causal ? launch_decode_variant<D, F16, true, 16>(q, k, v, p, grid, stream)
                        : launch_decode_variant<D, F16, false, 16>(q, k, v, p, grid, stream);
    return p.causal ? launch_decode_variant<D, F16, true, 32>(q, k, v, p, grid, stream)
                    : launch_decode_variant<D, F16, false, 32>(q, k, v, p, grid, stream);
}

}  // namespace fa
