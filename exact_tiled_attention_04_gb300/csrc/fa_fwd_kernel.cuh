// Fused exact-attention forward kernel for sm_103a (GB300).
//
// What it computes ("How Did I Write My First FlashAttention Kernel in
// CUDA?", pseudo-algorithm steps 1-5; "FlashAttention dissected", section
// "Algorithmic core in pseudocode"): for a block of query rows, sweep the
// key/value sequence tile by tile, keeping per row a running maximum m, a
// running denominator l and an unnormalised output accumulator O that is
// rescaled by exp(m_old - m_new) whenever m moves; divide O by l once at the
// end ("FlashAttention dissected", the final normalisation after the inner
// loop; the deferred division of "CUDA Flash Attention: Online Softmax with
// Shared Memory Tiling", Kernel 2).  The N x N score matrix never leaves the
// SM.
//
// Organisation (one CTA = 256 query rows of one (batch, head), 384 threads):
//   warps 0-3  softmax warpgroup 0: query tile 0 (rows 0-127 of the block)
//   warps 4-7  softmax warpgroup 1: query tile 1 (rows 128-255)
//   warp  8    tensor-core issuer of tile 0 (one thread) and TMEM owner
//   warp  9    TMA producer (one thread; the whole warp for fp32 inputs,
//              which also rounds each K tile to TF32)
//   warp 10    tensor-core issuer of tile 1 (one thread)
//   warp 11    fp32 inputs: writes each V tile transposed (V^T, TF32);
//              otherwise idle (completes warpgroup 2 for the register
//              reallocation)
// (fp32 inputs: the softmax warpgroups round their query tiles to TF32
// before the first scores.)
// Split launches whose partitions form a thread-block cluster merge them
// after the roles finish, in every warp (cluster_merge).
// Tensor memory (512 columns x 128 lanes, fp32):
//   S_w  columns [128w, 128w+128)   scores of tile w; P_w overwrites its
//                                   first columns (bf16 pairs or tf32)
//   O_w  columns [256 + Dw, 256 + D(w+1))   output accumulator of tile w
// Shared memory (128-byte-swizzled TMA tiles, 1024-byte aligned):
//   Q_0, Q_1 (reused as the output staging tiles), a ring of K tiles and a
//   ring of V tiles, then the mbarriers.
// Tensor-core work per key tile j and tile w, enqueued by tile w's issuer:
//   O_w += P_w(j) V_j as soon as P_w(j) is ready, then S_w(j+1) = Q_w K_{j+1}^T
//   (which overwrites P_w(j) in TMEM: same thread, so the tensor core runs
//   them in order).  While one tile's softmax runs, the other tile's
//   products keep the tensor core busy.

// Online-softmax details:
//   * scores are handled in base 2: t = s * scale * log2(e), p = 2^(t - m);
//   * the reference maximum m is only moved when the tile maximum exceeds
//     it by more than 8 (a factor 256): O and l are rescaled then, and
//     otherwise p <= 2^8 with the stale m.  The final O / l and
//     lse = (m + log2 l) ln 2 are exact for any reference maximum;
//   * keys past N in the last tile get weight exactly 0 (the "tile masking"
//     of "CUDA Flash Attention: Online Softmax with Shared Memory Tiling",
//     Design decisions, with the masked keys excluded rather than given a
//     large negative score); a reference maximum of -inf is replaced by 0
//     so that (-inf) - (-inf) never occurs (that page's NaN guard).
//
// Every wait on an mbarrier is bounded: after about a second the waiting
// thread raises a CTA-wide abort flag and sets the device error word; every
// role then leaves its loop, in-flight tensor-core work and TMA loads are
// drained, and tensor memory is freed before the CTA exits.
#pragma once

#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr int kTileM = 128;  // query rows per softmax warpgroup = TMEM lanes
constexpr int kTileN = 128;  // keys per K/V tile
// Three warpgroups: two softmax warpgroups and one holding the two
// tensor-core issuer warps, the TMA warp and one idle warp.  Registers are
// allocated per warpgroup, so the launch gets 384 x 168; setmaxnreg then
// moves them from warpgroup 2 to the softmax warpgroups (per variant, see
// FwdCfg: the split always sums to 384 x 168).
constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;   // tensor-core issuer of query tile 0, TMEM owner
constexpr int kMmaWarp2 = 10; // tensor-core issuer of query tile 1
constexpr int kLoadWarp = 9;
constexpr int kTransposeWarp = 11;  // fp32 inputs: writes the V^T tiles (otherwise idle)
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;             // log2 units
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

template <bool TF32, int D, bool F16 = false>
struct FwdCfg {
    static constexpr int kElem = TF32 ? 4 : 2;
    static constexpr int kAtomElems = 128 / kElem;      // elements in one 128-byte swizzle row
    static constexpr int kAtoms = D / kAtomElems;       // swizzle atoms across the head dim
    static constexpr int kAtomBytes = 128 * 128;        // 128 rows x 128 bytes
    static constexpr int kTileBytes = kAtoms * kAtomBytes;
    static constexpr int kUmmaK = 32 / kElem;           // K of one MMA instruction (32 bytes)
    static constexpr int kQkSteps = D / kUmmaK;
    static constexpr int kPvSteps = kTileN / kUmmaK;
    // fp32 inputs: the K ring holds TF32-rounded tiles, the V ring holds
    // transposed V^T tiles (the TF32 kind takes K-major operands only), and
    // one extra buffer receives the raw V tile from TMA.
    static constexpr int kKStages = TF32 ? 2 : (kTileBytes <= 16384 ? 4 : 3);
    static constexpr int kVStages = TF32 ? 2 : (kTileBytes <= 16384 ? 4 : 2);
    static constexpr int kVtAtomBytes = D * 128;  // V^T: D rows x 32 keys (128 bytes)
    // instruction-descriptor operand format: 0 = fp16, 1 = bf16, 2 = tf32
    static constexpr uint32_t kFmt = TF32 ? 2u : (F16 ? 0u : 1u);
    // S = Q K^T: M = 128, N = 128, A and B K-major.
    static constexpr uint32_t kIdescQK = instr_desc(kFmt, false, false, kTileM, kTileN);
    // O += P V: A (P) from TMEM, B (V) MN-major, M = 128.  bf16: one
    // instruction per k-step covers the whole head dimension (N = D; the
    // 64-column blocks of V are kAtomBytes apart, the descriptor's leading
    // byte offset).  Every tcgen05.mma costs about the same time for any
    // N <= 128, so fewer, wider instructions are faster.
    static constexpr int kPvN = D;
    static constexpr int kPvSplit = 1;
    static constexpr uint32_t kIdescPV = instr_desc(kFmt, false, !TF32, kTileM, kPvN);

    // Where the two softmax warpgroups take turns (kTakeTurns), the other
    // one may start once this one has published half kTurnAfterHalf of P.
    // d = 128: after the whole tile (strict alternation keeps the tensor
    // core fed); fp32 inputs at d = 64: after the first half (overlapping
    // the two warpgroups' exponentials wins there; measured +7 % at d = 64,
    // -7 % at d = 128).
    static constexpr int kTurnAfterHalf = (D == 64) ? 0 : 1;

    // Early scores (16-bit inputs at d = 64, where the four tiles of S, P
    // and O fit the 512 TMEM columns side by side): P has columns of its
    // own, so S(j+1) = Q K_{j+1}^T is enqueued as soon as the softmax has
    // read S(j) into registers, ahead of O += P(j) V.  The next tile's
    // scores are then ready when the softmax finishes a tile, instead of a
    // product's latency later.  Elsewhere P overwrites S (d = 128 needs
    // the columns) and S(j+1) follows O += P(j) V.
    static constexpr bool kEarlyS = !TF32 && D == 64;
    static constexpr uint32_t kColP = 256;                  // kEarlyS: P_w at 256 + 64 w
    static constexpr uint32_t kColO = kEarlyS ? 384 : 256;  // O_w at kColO + D w
    // With early scores each warpgroup's next tile is ready when it needs
    // it, and turns would only serialise the two softmaxes: they run freely
    // (measured at d = 64: early scores alone +4 %, and without turns
    // +24 % on top).
    static constexpr bool kTakeTurns = !kEarlyS;
    // With early scores the two tiles run in step, and each softmax
    // warpgroup waits on the release barriers of the K and V stages (both
    // tiles' products) instead of completion barriers of its own tile: two
    // tcgen05.commit fewer per tile and issuer, each of which costs the
    // tensor pipe time (measured: two extra commits per tile and issuer
    // cost 5 %; this saves 5 % at d = 64.  Release barriers per tile,
    // waited for by their own tile's softmax, measured 4 % slower at
    // d = 128 and gained less at d = 64.)
    static constexpr bool kStageDone = kEarlyS;
    // row maxima from the reducing TMEM load (see the softmax loop)
    static constexpr bool kHwMax = D == 64;

    // register split (setmaxnreg): softmax warpgroups / warpgroup 2, chosen
    // so that neither side spills
    static constexpr uint32_t kSoftmaxRegs = TF32 ? 200 : 208;
    static constexpr uint32_t kOtherRegs = TF32 ? 104 : 88;
    static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs == kThreads * kLaunchRegs,
                  "register split must equal the launch allocation");

    // shared-memory map (offsets from the 1024-aligned base)
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffVRaw = kOffV + kVStages * kTileBytes;
    static constexpr int kOffBar = kOffVRaw + (TF32 ? kTileBytes : 0);
    // barrier slots
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kBarSFull = kBarVEmpty + kVStages;  // [2] (not kStageDone)
    static constexpr int kBarPFull = kBarSFull + 2;          // [2 tiles][2 halves]
    static constexpr int kBarOFull = kBarPFull + 4;          // [2]
    static constexpr int kBarEpi = kBarOFull + 2;            // [2]
    static constexpr int kBarDrain = kBarEpi + 2;            // [2]
    static constexpr int kBarQRaw = kBarDrain + 2;  // fp32 only: TMA landed, not yet rounded
    static constexpr int kBarKRaw = kBarQRaw + 1;   // [kKStages]
    static constexpr int kBarVRaw = kBarKRaw + kKStages;
    static constexpr int kBarTurn = kBarVRaw + 1;  // [2]: softmax warpgroup w may start a tile
    static constexpr int kBarSFree = kBarTurn + 2;   // [2] kEarlyS: S_w read (4 warps)
    static constexpr int kBarPVDone = kBarSFree + 2; // [2] kEarlyS, not kStageDone: O_w += P_w V done
    static constexpr int kBarVRawFree = kBarPVDone + 2;  // fp32 only: the raw V buffer was transposed
    static constexpr int kBarMerge = kBarVRawFree + 1;    // in-cluster merge: the peers' rows landed
    static constexpr int kNumBars = kBarMerge + 1;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffTurnFlags = kOffAbort + 4;  // [2][4] u32: turns each softmax warp has received
    static constexpr int kSmemUsed = kOffTurnFlags + 32;
    static constexpr size_t kSmemBytes = static_cast<size_t>(kSmemUsed) + 1024;  // alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
    // In-cluster merge of split partials: the unnormalised O (256 rows x D
    // fp32) and (m, l, lq) per row, written over the K and V rings once every
    // product of the CTA has completed.
    // In-cluster merge (cluster_merge): a padded row per query row (D fp32,
    // then m, l, lq, 0); the send buffer (256 rows) at the top of the operand
    // area, the receive slots ((S - 1) x ceil(256 / S) rows) from its start.
    static constexpr int kMergeRowBytes = D * 4 + 16;
    static constexpr int kOffSend = kOffBar - 256 * kMergeRowBytes;
    static_assert(kOffSend >= kOffQ + 2 * 2048, "send buffer over the row statistics");
    static_assert(kOffSend % 16 == 0, "bulk copies need 16-byte alignment");
    // the largest cluster whose receive slots fit below the send buffer
    static constexpr int max_merge_parts() {
        int s = 8;
        while (s > 2 && (s - 1) * ((256 + s - 1) / s) * kMergeRowBytes > kOffSend - kOffQ) --s;
        return s;
    }
    static constexpr int kMaxMergeParts = max_merge_parts();
    static_assert((kMaxMergeParts - 1) * ((256 + kMaxMergeParts - 1) / kMaxMergeParts) * kMergeRowBytes <=
                      kOffSend - kOffQ,
                  "receive slots do not fit");
    static_assert(kColO + 2 * D <= kTmemCols, "tensor memory budget exceeded");
};

// Bounded spin until *flag >= target, a shared counter that one warp of the
// other softmax warpgroup advances; the same give-up rule as wait_phase.
// (A spinning warp wakes within a few tens of clocks of the store, where an
// mbarrier wait took about 150.)
__device__ __forceinline__ bool wait_flag(volatile uint32_t* flag, uint32_t target,
                                          volatile uint32_t* abort_flag, const FwdParams& fp,
                                          unsigned int where) {
    if (*flag >= target) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (*flag >= target) return true;
        if ((++spins & 31u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1u;
                atomicOr(&fp.status->word, kDevErrTimeout | (where << 8));
                atomicExch(&fp.status->abort_gen, fp.gen);
                return false;
            }
        }
    }
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (if `honor_abort`) or when this wait itself gave up after kWaitLimitNs, in
// which case it raises the CTA's abort flag, sets the sticky device error
// bits (with the waiting role in bits 8-15) and marks this launch's
// generation as aborted, so CTAs of the same launch that start later skip
// their work.  Later launches are not affected.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile uint32_t* abort_flag, const FwdParams& fp,
                                           unsigned int where, bool honor_abort = true) {
    DevStatus* const status = fp.status;
    const unsigned int gen = fp.gen;
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if ((++spins & 31u) == 0u) {
            if (honor_abort && *abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1u;
                atomicOr(&status->word, kDevErrTimeout | (where << 8));
                atomicExch(&status->abort_gen, gen);
                return false;
            }
        }
    }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Maximum (kMax) or minimum of a 128-key score row held in registers: eight
// running accumulators over keys k = a (mod 8), three-input max/min, so only
// eight values are live beside the row and the dependent chain is 8 long.
template <bool kMax>
__device__ __forceinline__ float row_extreme(const uint32_t (&s)[4][32]) {
    auto v = [&](int e) { return u2f(s[e / 32][e % 32]); };
    auto two = [](float a, float b) { return kMax ? fmaxf(a, b) : fminf(a, b); };
    auto three = [](float a, float b, float c) { return kMax ? fmax3(a, b, c) : fmin3(a, b, c); };
    float acc[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) acc[a] = two(v(a), v(a + 8));
#pragma unroll
    for (int r = 2; r < 16; r += 2)
#pragma unroll
        for (int a = 0; a < 8; ++a) acc[a] = three(acc[a], v(a + 8 * r), v(a + 8 * (r + 1)));
    return two(three(acc[0], acc[1], acc[2]), three(acc[3], acc[4], two(acc[5], three(acc[6], acc[7], acc[7]))));
}

// Softmax numerators of one half (keys 64h .. 64h+63) of a 128-key score row
// held in registers: p_j = 2^(s_j * c - shift), keys >= `valid` get p = 0
// (kMasked, last tile only).  Writes P into tensor memory over the scores
// (bf16 pairs in 32 columns, or TF32 values in 64 columns) and adds p (fp32)
// into acc, per packed lane pair.  Pairs of keys go through the packed
// f32x2 FMA / add.
template <bool TF32, bool F16, bool kMasked>
__device__ __forceinline__ void exp_half(const uint32_t (&s)[4][32], uint64_t c2, uint64_t ns2,
                                         int valid, uint32_t tS, int h, uint64_t (&acc)[4]) {
    if constexpr (TF32) {
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            const int q = 2 * h + qq;
            uint32_t pw[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float t0, t1;
                f2_unpack(f2_fma(f2_pack(u2f(s[q][i]), u2f(s[q][i + 1])), c2, ns2), t0, t1);
                float p0 = ex2(t0), p1 = ex2(t1);
                if constexpr (kMasked) {
                    if (q * 32 + i >= valid) p0 = 0.0f;
                    if (q * 32 + i + 1 >= valid) p1 = 0.0f;
                }
                pw[i] = round_tf32(p0);
                pw[i + 1] = round_tf32(p1);
                acc[(i / 2) & 3] = f2_add(acc[(i / 2) & 3], f2_pack(p0, p1));
            }
            tmem_st32(tS + 32u * q, pw);
        }
    } else {
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c0 = h * 64 + 2 * i;  // keys c0, c0 + 1
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(u2f(s[c0 / 32][c0 % 32]), u2f(s[c0 / 32][c0 % 32 + 1])), c2, ns2),
                      t0, t1);
            float p0 = ex2(t0), p1 = ex2(t1);
            if constexpr (kMasked) {
                if (c0 >= valid) p0 = 0.0f;
                if (c0 + 1 >= valid) p1 = 0.0f;
            }
            const uint32_t pk = pack_16x2<F16>(p0, p1);
            pw[i] = pk;
            acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
        }
        tmem_st32(tS + 32u * h, pw);
    }
}

// One unmasked half of P as 16-bit pairs into registers (for the
// speculative path of the softmax loop; exp_half's arithmetic, no store).
template <bool F16>
__device__ __forceinline__ void exp_half_regs(const uint32_t (&s)[4][32], uint64_t c2, uint64_t ns2, int h,
                                              uint32_t (&pw)[32], uint64_t (&acc)[4]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int c0 = h * 64 + 2 * i;  // keys c0, c0 + 1
        float t0, t1;
        f2_unpack(f2_fma(f2_pack(u2f(s[c0 / 32][c0 % 32]), u2f(s[c0 / 32][c0 % 32 + 1])), c2, ns2), t0, t1);
        const float p0 = ex2(t0), p1 = ex2(t1);
        pw[i] = pack_16x2<F16>(p0, p1);
        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
    }
}

// Sum of the eight fp32 lanes of four packed pairs.
__device__ __forceinline__ float sum8(const uint64_t (&a)[4]) {
    float x[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) f2_unpack(a[k], x[2 * k], x[2 * k + 1]);
    return ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
}

// Epilogue of one key partition of a split launch (one thread = one query
// row): the unnormalised accumulator, relative to the reference maximum m,
// and m, l, lq go to the partition's slab of the workspace (or, for an
// in-cluster merge, m, l, lq to shared memory).  Not inlined: it runs once
// per CTA, and keeping it a call keeps the softmax loop's register
// allocation as it is (the same statistics stored inline there made ptxas
// spill ten times more in the d = 128 kernel).
template <int D>
__device__ __noinline__ void store_partial(const FwdParams& p, uint32_t tO, long long qrow, float m_ref,
                                           float l, float lq, uint8_t* cluster_stats) {
    if (p.cluster) {
        // in-cluster merge: the row's statistics go to this CTA's shared
        // memory (`cluster_stats`, in its query tile, whose products have all
        // completed); O stays in tensor memory until cluster_merge
        *reinterpret_cast<float4*>(cluster_stats) = make_float4(m_ref, l, lq, 0.0f);
        return;
    }
    // qrow: the query row's output row (of B*H*Nq), or -1 for a tile row
    // that is not a query row; a partition's slab holds rows part_row0 ..
    // part_row0 + part_rows - 1
    const unsigned int split = blockIdx.x % static_cast<unsigned>(p.splits);
    const size_t r = split * static_cast<size_t>(p.part_rows) + static_cast<size_t>(qrow - p.part_row0);
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(tO + 32u * q, o);
        tmem_ld_wait(o);
        if (qrow >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.o_part + r * D + q * 32);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                dst[ch] = make_uint4(o[4 * ch], o[4 * ch + 1], o[4 * ch + 2], o[4 * ch + 3]);
        }
    }
    if (qrow >= 0) *reinterpret_cast<float4*>(p.ml_part + r * 4) = make_float4(m_ref, l, lq, 0.0f);
}

// Zero the rows of the two query tiles that a packed launch does not load
// (row >= `rows` of tile 0, all of tile 1), one warp, before the Q load.
template <int kTileBytes, int kAtoms, int kAtomBytes>
__device__ __forceinline__ void zero_unloaded_q(uint8_t* q_tiles, int rows, int lane) {
    for (int a = 0; a < kAtoms; ++a) {
        uint4* t0 = reinterpret_cast<uint4*>(q_tiles + a * kAtomBytes);
        for (int i = rows * 8 + lane; i < 128 * 8; i += 32) t0[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    uint4* t1 = reinterpret_cast<uint4*>(q_tiles + kTileBytes);
    for (int i = lane; i < kTileBytes / 16; i += 32) t1[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    __syncwarp();
}

// Round `n16` 16-byte groups of fp32 in shared memory to TF32 in place
// (round to nearest, ties away), by `nthreads` threads (thread `tid`).  The
// loads of eight groups are issued before their stores, so their latencies
// overlap.
__device__ __forceinline__ void round_tf32_inplace(uint8_t* base, int n16, int tid, int nthreads) {
    uint4* p4 = reinterpret_cast<uint4*>(base);
    for (int i0 = tid; i0 < n16; i0 += 8 * nthreads) {
        uint4 v[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (i0 + b * nthreads < n16) v[b] = p4[i0 + b * nthreads];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (i0 + b * nthreads < n16) {
                uint4 r;
                r.x = round_tf32(u2f(v[b].x));
                r.y = round_tf32(u2f(v[b].y));
                r.z = round_tf32(u2f(v[b].z));
                r.w = round_tf32(u2f(v[b].w));
                p4[i0 + b * nthreads] = r;
            }
        }
    }
}

// fp32 V tile as loaded by TMA ([D/32 atoms][128 keys][128 bytes], swizzled)
// -> TF32-rounded V^T in the K-major swizzled operand layout
// ([4 atoms of 32 keys][D rows][128 bytes]), one warp.  Step i: lanes cover
// 32 consecutive d of one group of four keys, so the reads are 4
// row-contiguous 128-byte lines and the 16-byte writes take the minimum 4
// wavefronts.  Eight steps' loads are issued before their stores (the two
// buffers are distinct, which the compiler cannot see).
template <int D>
__device__ __forceinline__ void transpose_v_tf32(const uint8_t* vraw, uint8_t* vt, int lane) {
    constexpr int kDBlocks = D / 32;
    constexpr int kSteps = 32 * kDBlocks;
    static_assert(kSteps % 8 == 0, "whole batches of steps");
    for (int i0 = 0; i0 < kSteps; i0 += 8) {
        uint32_t r[8][4];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int i = i0 + b;
            const int d = (i % kDBlocks) * 32 + lane;
            const int kg = i / kDBlocks;  // keys 4kg .. 4kg+3
            const int atom_in = d / 32, c_in = (d % 32) / 4, w_in = (d % 4) * 4;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int key = 4 * kg + t;
                r[b][t] = *reinterpret_cast<const uint32_t*>(vraw + atom_in * 16384 + key * 128 +
                                                             ((c_in ^ (key & 7)) << 4) + w_in);
            }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int i = i0 + b;
            const int d = (i % kDBlocks) * 32 + lane;
            const int kg = i / kDBlocks;
            uint8_t* dst = vt + (kg / 8) * (D * 128) + d * 128 + (((kg % 8) ^ (d & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = make_uint4(round_tf32(u2f(r[b][0])), round_tf32(u2f(r[b][1])),
                                                        round_tf32(u2f(r[b][2])), round_tf32(u2f(r[b][3])));
        }
    }
}

// Producer warp of the fp32 (TF32) variant: TMA loads as in the 16-bit path
// (Q, K and V land "raw" on their own barriers), then the whole warp rounds
// each K tile in place and publishes it after a proxy fence.  The softmax
// warpgroups round Q (they are idle until the first scores), and warp 11
// writes the V^T tiles (transpose_tf32), so the three run side by side.  The
// raw V buffer is single: the load of tile j waits until the transposer has
// read tile j - 1 out of it.
template <int D>
__device__ void produce_tf32(const CUtensorMap& map_q, const CUtensorMap& map_k,
                             const CUtensorMap& map_v, const FwdParams& p, uint8_t* smem,
                             uint32_t sbase, int lane, int row0, int bh, int kvh, int t_begin, int T,
                             volatile uint32_t* abort_flag) {
    using C = FwdCfg<true, D>;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    auto all_ok = [&](bool ok) { return __all_sync(0xffffffffu, ok); };
    const uint64_t keep = policy_evict_last();
    const uint64_t once = policy_evict_first();
    int nk = 0, nv = 0;  // K and V tiles whose loads were issued
    bool ok = true;
    if (p.pack) zero_unloaded_q<C::kTileBytes, C::kAtoms, C::kAtomBytes>(smem + C::kOffQ, p.Nq * p.group, lane);
    if (lane == 0) {
        if (p.pack) {
            mbar_arrive_expect_tx(bar(C::kBarQRaw), static_cast<uint32_t>(C::kAtoms * p.Nq * p.group * 128));
            for (int a = 0; a < C::kAtoms; ++a)
                tma_load_3d(sbase + C::kOffQ + a * C::kAtomBytes, &map_q, bar(C::kBarQRaw),
                            a * C::kAtomElems, 0, bh * p.group, once);
        } else {
            mbar_arrive_expect_tx(bar(C::kBarQRaw), 2u * C::kTileBytes);
            for (int w = 0; w < 2; ++w)
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffQ + w * C::kTileBytes + a * C::kAtomBytes, &map_q,
                                bar(C::kBarQRaw), a * C::kAtomElems, row0 + w * kTileM, bh, once);
        }
    }
    for (int j = 0; ok && j < T; ++j) {
        const int ks = j % C::kKStages;
        ok = all_ok(wait_phase(bar(C::kBarKEmpty + ks), ((j / C::kKStages) & 1) ^ 1, abort_flag, p, 21));
        if (!ok) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::kBarKRaw + ks), C::kTileBytes);
            for (int a = 0; a < C::kAtoms; ++a)
                tma_load_3d(sbase + C::kOffK + ks * C::kTileBytes + a * C::kAtomBytes, &map_k,
                            bar(C::kBarKRaw + ks), a * C::kAtomElems, (t_begin + j) * kTileN, kvh, keep);
        }
        nk = j + 1;
        // the raw V buffer is free once tile j - 1 was transposed out of it
        if (j > 0) ok = all_ok(wait_phase(bar(C::kBarVRawFree), (j - 1) & 1, abort_flag, p, 24));
        if (!ok) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::kBarVRaw), C::kTileBytes);
            for (int a = 0; a < C::kAtoms; ++a)
                tma_load_3d(sbase + C::kOffVRaw + a * C::kAtomBytes, &map_v, bar(C::kBarVRaw),
                            a * C::kAtomElems, (t_begin + j) * kTileN, kvh, keep);
        }
        nv = j + 1;
        ok = all_ok(wait_phase(bar(C::kBarKRaw + ks), (j / C::kKStages) & 1, abort_flag, p, 22));
        if (!ok) break;
        round_tf32_inplace(smem + C::kOffK + ks * C::kTileBytes, C::kTileBytes / 16, lane, 32);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarKFull + ks));
    }
    // Drain every TMA load this warp issued (see the 16-bit producer).  At
    // most one raw V load is in flight (each waits for the previous one's
    // transpose), so the last issued one's phase is the one to wait for.
    if (lane == 0) {
        wait_phase(bar(C::kBarQRaw), 0, abort_flag, p, 25, false);
        for (int s = 0; s < C::kKStages && s < nk; ++s) {
            const int last = s + ((nk - 1 - s) / C::kKStages) * C::kKStages;
            wait_phase(bar(C::kBarKRaw + s), (last / C::kKStages) & 1, abort_flag, p, 25, false);
        }
        if (nv > 0) wait_phase(bar(C::kBarVRaw), (nv - 1) & 1, abort_flag, p, 25, false);
    }
}

// Warp 11 of the fp32 variant: each raw V tile -> the V^T operand tile of
// its stage (once the products of the tile that used the stage before have
// completed), published after a proxy fence; then the raw buffer is handed
// back to the producer.
template <int D>
__device__ void transpose_tf32(const FwdParams& p, uint8_t* smem, uint32_t sbase, int lane, int T,
                               volatile uint32_t* abort_flag) {
    using C = FwdCfg<true, D>;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    for (int j = 0; j < T; ++j) {
        const int vs = j % C::kVStages;
        if (!__all_sync(0xffffffffu, wait_phase(bar(C::kBarVRaw), j & 1, abort_flag, p, 23))) break;
        if (!__all_sync(0xffffffffu, wait_phase(bar(C::kBarVEmpty + vs), ((j / C::kVStages) & 1) ^ 1, abort_flag, p,
                                                26)))
            break;
        transpose_v_tf32<D>(smem + C::kOffVRaw, smem + C::kOffV + vs * C::kTileBytes, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(bar(C::kBarVFull + vs));
            mbar_arrive(bar(C::kBarVRawFree));
        }
    }
}

// In-cluster merge of the key partitions of one 256-row query block (p.cluster):
// the `splits` CTAs of a thread-block cluster swept disjoint key ranges of
// the same query rows.  They combine like consecutive tiles of the online
// softmax ("FlashAttention dissected", section "The mathematical
// breakthrough: Tiling and Online Softmax": rescale by the correction factor
// and add; section "Interaction with the KV cache during inference": the key
// sequence split across cores), with M = max_s m_s, w_s = 2^(m_s - M):
//   O = sum_s w_s O_s / sum_s w_s lq_s,   lse = ln 2 (M + log2 sum_s w_s l_s).
// CTA r of the cluster owns rows [256 r / S, 256 (r + 1) / S) of the block.
// Distributed shared memory moves about 20 bytes per clock between two SMs
// (measured: 64 KB in 3.3k clocks as one bulk copy, 4.2k as contiguous
// 16-byte stores by the threads, 7.3k as stores scattered over rows), so the
// rows travel as one bulk copy per peer.  Run by all 384 threads of every
// CTA of the cluster, after every role has finished (every product has
// completed and every TMA load has landed), on every path:
//   1. stage: the warps copy this CTA's unnormalised O of both tiles out of
//      tensor memory (warp w reads TMEM lane quarter w % 4) into a send
//      buffer at the top of its shared memory, one padded row per query row
//      (D fp32 and then (m, l, lq, 0), the statistics the softmax threads
//      left in the query tiles), so each owner's rows are contiguous; and
//      announce the bytes this CTA will receive on its merge barrier;
//   2. cluster barrier: every CTA has staged and is done with its K/V rings,
//      where the receive slots lie (a CTA whose partition sees no key gets
//      here at once, and must not be written to while a peer still streams
//      tiles);
//   3. one thread sends each peer its rows in one bulk copy, into the peer's
//      slot for this partition, completing on the peer's merge barrier;
//   4. wait (bounded) for the peers' rows, combine the owned rows (own rows
//      read from the send buffer) and write O (input dtype) and lse to global
//      memory, 8 columns per thread;
//   5. cluster barrier: every copy out of this CTA's send buffer has landed
//      (each CTA passed step 4 only after its own copies arrived).
// `write`: this CTA's partials are valid (no role gave up on a wait); a CTA
// without valid partials still sends (meaningless rows of an already failed
// launch), so no peer waits in vain.  The code runs outside the role
// branches and holds nothing in registers across them, so the softmax
// loop's register allocation does not see it.
template <bool TF32, int D, bool F16>
__device__ __forceinline__ void cluster_merge(const FwdParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                                              bool write, bool has_work, int row0, int bh,
                                              volatile uint32_t* abort_flag) {
    using C = FwdCfg<TF32, D, F16>;
    constexpr int kRowBytes = C::kMergeRowBytes;  // D fp32 + (m, l, lq, 0)
    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;
    const int S = p.splits;
    const int rmax = (256 + S - 1) / S;  // rows owned by one CTA, at most
    const int me = static_cast<int>(cluster_ctarank());
    const int rb0 = (256 * me) / S, rb1 = (256 * (me + 1)) / S;
    // receive slots [S - 1][rmax rows] from the start of the Q tiles; the
    // send buffer [256 rows] at the top of the operand area
    uint8_t* recv = smem + C::kOffQ;
    uint8_t* send = smem + C::kOffSend;
    const uint32_t merge_bar = sbase + C::kOffBar + 8u * static_cast<uint32_t>(C::kBarMerge);

    if (write) {
        if (has_work) {
            const int quarter = warp % 4;
            const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
            // (tile, 32-column chunk) items of this lane quarter, dealt to its three warps
            for (int item = warp / 4; item < 2 * (D / 32); item += 3) {
                const int tile = item / (D / 32), q = item % (D / 32);
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + C::kColO + static_cast<uint32_t>(D * tile + 32 * q), o);
                tmem_ld_wait(o);
                // padded rows: a warp's 32 rows start 16 bytes apart in the
                // banks, so its 16-byte stores take the minimum 4 wavefronts
                uint4* dst = reinterpret_cast<uint4*>(send + (128 * tile + 32 * quarter + lane) * kRowBytes + 128 * q);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) dst[ch] = make_uint4(o[4 * ch], o[4 * ch + 1], o[4 * ch + 2], o[4 * ch + 3]);
            }
        }
        if (threadIdx.x < 256) {
            const int r = static_cast<int>(threadIdx.x);
            *reinterpret_cast<uint4*>(send + r * kRowBytes + D * 4) =
                *reinterpret_cast<const uint4*>(smem + C::kOffQ + (r / 128) * C::kTileBytes + (r % 128) * 16);
        }
    }
    if (threadIdx.x == 0)  // this CTA receives its owned rows from every peer
        mbar_arrive_expect_tx(merge_bar, static_cast<uint32_t>((S - 1) * (rb1 - rb0) * kRowBytes));
    fence_proxy_async_smem();  // the staged rows are read by the bulk copies
    cluster_sync_all();

    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            if (k == me) continue;
            const int k0 = (256 * k) / S, k1 = (256 * (k + 1)) / S;
            const int slot = me < k ? me : me - 1;  // the peer's slot for this partition
            bulk_copy_to_peer(mapa_shared(sbase + C::kOffQ + static_cast<uint32_t>(slot * rmax * kRowBytes),
                                          static_cast<uint32_t>(k)),
                              smem_u32(send + k0 * kRowBytes), static_cast<uint32_t>((k1 - k0) * kRowBytes),
                              mapa_shared(merge_bar, static_cast<uint32_t>(k)));
        }
    }
    const bool arrived = __all_sync(0xffffffffu, wait_phase(merge_bar, 0, abort_flag, p, 17, false));

    constexpr int kTpr = D / 8;  // threads per row (8 output columns each)
    constexpr int kRowsPerPass = kThreads / kTpr;
    const int i = static_cast<int>(threadIdx.x);
    const int col0 = (i % kTpr) * 8;
    for (int rb = rb0 + i / kTpr; arrived && rb < rb1; rb += kRowsPerPass) {
        const long long qi = static_cast<long long>(row0) + rb;
        if (qi >= p.Nq) break;  // rows only grow along this loop
        const int rr = rb - rb0;
        // partition s's row: this CTA's own in the send buffer, a peer's in its slot
        auto row_of = [&](int s) -> const uint8_t* {
            return s == me ? send + rb * kRowBytes : recv + ((s < me ? s : s - 1) * rmax + rr) * kRowBytes;
        };
        float M = -INFINITY;
        for (int s = 0; s < S; ++s) M = fmaxf(M, reinterpret_cast<const float4*>(row_of(s) + D * 4)->x);
        const float mref = (M == -INFINITY) ? 0.0f : M;
        float L = 0.0f, LQ = 0.0f;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        for (int s = 0; s < S; ++s) {
            const uint8_t* row = row_of(s);
            const float4 st = *reinterpret_cast<const float4*>(row + D * 4);
            const float wgt = ex2(st.x - mref);  // ex2(-inf) = 0: no visible key
            L += wgt * st.y;
            LQ += wgt * st.z;
            if (wgt != 0.0f) {  // a partition with no visible key staged no O
                const float4 x0 = *reinterpret_cast<const float4*>(row + col0 * 4);
                const float4 x1 = *reinterpret_cast<const float4*>(row + col0 * 4 + 16);
                acc[0] += wgt * x0.x;
                acc[1] += wgt * x0.y;
                acc[2] += wgt * x0.z;
                acc[3] += wgt * x0.w;
                acc[4] += wgt * x1.x;
                acc[5] += wgt * x1.y;
                acc[6] += wgt * x1.z;
                acc[7] += wgt * x1.w;
            }
        }
        const float inv = LQ > 0.0f ? 1.0f / LQ : 0.0f;
        const size_t out_row = static_cast<size_t>(bh) * static_cast<size_t>(p.Nq) + static_cast<size_t>(qi);
        if constexpr (TF32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row * D + col0);
            dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
        } else {
            uint4 v4;
            v4.x = pack_16x2<F16>(acc[0] * inv, acc[1] * inv);
            v4.y = pack_16x2<F16>(acc[2] * inv, acc[3] * inv);
            v4.z = pack_16x2<F16>(acc[4] * inv, acc[5] * inv);
            v4.w = pack_16x2<F16>(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + out_row * D + col0) = v4;
        }
        if (p.lse != nullptr && col0 == 0)
            p.lse[out_row] = (L > 0.0f) ? (mref + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    cluster_sync_all();
}

// kOneTile: a packed launch (p.pack = 1), where query tile 1 holds no row;
// a template parameter so that unpacked launches carry none of its checks.
template <bool TF32, int D, bool F16 = false, bool kCausal = false, bool kOneTile = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                  const FwdParams p) {
    using C = FwdCfg<TF32, D, F16>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_u32 + pad;

    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;
    // blockIdx.x = cta * splits + split; cta = bh * n_q_blocks + qb, or
    // (causal) the heavy-first order of lpt_item over (bh, block)
    // grouped heads packed into query tile 0 (p.pack; always set when kOneTile)
    const bool pack = kOneTile || p.pack != 0;
    const unsigned int split = blockIdx.x % static_cast<unsigned>(p.splits);
    // (a tail launch starts at query block p.item_offset; unmasked launches only)
    const unsigned int cta = blockIdx.x / static_cast<unsigned>(p.splits) + static_cast<unsigned>(p.item_offset);
    int qb, bh;
    if (kCausal) {
        // later query blocks see more keys: heaviest first, by groups of heads
        // (packed launches have one block per key/value head)
        const int units = static_cast<int>(gridDim.x / static_cast<unsigned>(p.splits)) / p.n_q_blocks;
        int rank;
        lpt_item(cta, units, p.n_q_blocks, bh, rank);
        qb = p.n_q_blocks - 1 - rank;
    } else {
        qb = static_cast<int>(cta % static_cast<unsigned>(p.n_q_blocks));
        bh = static_cast<int>(cta / static_cast<unsigned>(p.n_q_blocks));
    }
    // key/value head of this query head (grouped-query attention: H / H_kv
    // query heads share one key/value head)
    // packed: bh is the key/value head itself; otherwise its query head's
    const int kvh = pack ? bh : (bh / p.H) * p.H_kv + (bh % p.H) / p.group;
    // rows of query tile 0 that hold query rows in a packed launch
    const int pack_rows = pack ? p.Nq * p.group : 0;
    // packed launches hold no query row in tile 1: its issuer and softmax
    // warpgroup sit out, and K/V stages are released by tile 0 alone
    constexpr bool one_tile = kOneTile;
    const int row0 = qb * 2 * kTileM;
    // key tiles this query block can see: all, or under the causal mask
    // those up to the last key its last row sees
    int n_tiles_block = p.n_kv_tiles;
    if (kCausal) {
        // last query index of the block (packed: every row has i < Nq)
        const long long last_i = pack ? p.Nq - 1 : static_cast<long long>(row0) + 2 * kTileM - 1;
        const long long lim = min(static_cast<long long>(p.Nkv), last_i + 1 + p.causal_offset);
        n_tiles_block = lim <= 0 ? 0 : static_cast<int>((lim + kTileN - 1) / kTileN);
    }
    const int t_begin = static_cast<int>(split) * p.tiles_per_split;
    // <= 0: this partition sees no key (causal mask); only its epilogue runs
    const int T = min(p.tiles_per_split, n_tiles_block - t_begin);
    const bool has_work = !kCausal || T > 0;  // without the mask every partition has a tile

    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        // read first: its latency (a cold line at the start of a launch)
        // overlaps the barrier setup below
        const unsigned int abort_gen = *reinterpret_cast<volatile unsigned int*>(&p.status->abort_gen);
        // fp32: the eight softmax warps round Q and arrive; else the TMA load
        mbar_init(bar(C::kBarQFull), TF32 ? 8 : 1);
        const uint32_t issuers = one_tile ? 1u : 2u;
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKEmpty + s), issuers);  // every active issuer's commit
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), issuers);
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(bar(C::kBarSFull + w), 1);
            mbar_init(bar(C::kBarPFull + 2 * w + 0), 4);  // one arrival per softmax warp
            mbar_init(bar(C::kBarPFull + 2 * w + 1), 4);
            mbar_init(bar(C::kBarTurn + w), 4);
            mbar_init(bar(C::kBarSFree + w), 4);
            mbar_init(bar(C::kBarPVDone + w), 1);
            mbar_init(bar(C::kBarOFull + w), 1);
            mbar_init(bar(C::kBarEpi + w), kTileM);
        }
        mbar_init(bar(C::kBarDrain + 0), 1);
        mbar_init(bar(C::kBarDrain + 1), 1);
        mbar_init(bar(C::kBarQRaw), 1);
        for (int s = 0; s < C::kKStages; ++s) mbar_init(bar(C::kBarKRaw + s), 1);
        mbar_init(bar(C::kBarVRaw), 1);
        mbar_init(bar(C::kBarVRawFree), 1);
        mbar_init(bar(C::kBarMerge), 1);
        {
            // turn counters of the flag turns: warpgroup 0 holds the first turn
            volatile uint32_t* tf = reinterpret_cast<volatile uint32_t*>(smem + C::kOffTurnFlags);
            for (int i = 0; i < 8; ++i) tf[i] = i < 4 ? 1u : 0u;
        }
        // A CTA starting after another CTA of this launch timed out does no work.
        *abort_flag = (abort_gen == p.gen) ? 1u : 0u;
        mbar_init_fence();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        tma_prefetch_desc(&map_o);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0u;

    if (skip) {
        // nothing issued: go straight to the teardown
    } else if (warp >= 8) {
        // warpgroup 2: TMA producer, two tensor-core issuers, one idle warp
        regs_decrease<C::kOtherRegs>();
      if (!has_work) {
        // no visible key: nothing to load or multiply
      } else if (warp == kLoadWarp) {
        // ------------------------------------------------------ TMA producer
        // a launch that follows in the stream with programmatic serialization
        // (the split last wave) may place its CTAs as this grid's leave the SMs
        if (lane == 0) asm volatile("griddepcontrol.launch_dependents;");
        if (!TF32 && pack) zero_unloaded_q<C::kTileBytes, C::kAtoms, C::kAtomBytes>(smem + C::kOffQ, pack_rows, lane);
        if constexpr (TF32) {
            produce_tf32<D>(map_q, map_k, map_v, p, smem, sbase, lane, row0, bh, kvh, t_begin, T, abort_flag);
        } else if (lane == 0) {
            const uint64_t keep = policy_evict_last();   // K/V: read by every query block of the head
            const uint64_t once = policy_evict_first();  // Q: read once
            if (pack) {
                // Nq rows x group heads into the first rows of tile 0
                mbar_arrive_expect_tx(bar(C::kBarQFull), static_cast<uint32_t>(C::kAtoms * pack_rows * 128));
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffQ + a * C::kAtomBytes, &map_q, bar(C::kBarQFull),
                                a * C::kAtomElems, 0, bh * p.group, once);
            } else {
                mbar_arrive_expect_tx(bar(C::kBarQFull), 2u * C::kTileBytes);
                for (int w = 0; w < 2; ++w)
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d(sbase + C::kOffQ + w * C::kTileBytes + a * C::kAtomBytes, &map_q,
                                    bar(C::kBarQFull), a * C::kAtomElems, row0 + w * kTileM, bh, once);
            }
            int nk = 0, nv = 0;  // K and V tiles whose loads were issued
            for (int j = 0; j < T; ++j) {
                const int ks = j % C::kKStages;
                if (!wait_phase(bar(C::kBarKEmpty + ks), ((j / C::kKStages) & 1) ^ 1, abort_flag, p, 1))
                    break;
                mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kTileBytes);
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffK + ks * C::kTileBytes + a * C::kAtomBytes, &map_k,
                                bar(C::kBarKFull + ks), a * C::kAtomElems, (t_begin + j) * kTileN, kvh, keep);
                nk = j + 1;
                const int vs = j % C::kVStages;
                if (!wait_phase(bar(C::kBarVEmpty + vs), ((j / C::kVStages) & 1) ^ 1, abort_flag, p, 2))
                    break;
                mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kTileBytes);
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffV + vs * C::kTileBytes + a * C::kAtomBytes, &map_v,
                                bar(C::kBarVFull + vs), a * C::kAtomElems, (t_begin + j) * kTileN, kvh, keep);
                nv = j + 1;
            }
            // Drain: wait until every issued load has landed, so that no TMA
            // write reaches shared memory after the CTA exits.  On the normal
            // path these phases completed long ago.  The last tile loaded
            // into stage s is the largest index below the issued count that
            // is congruent to s.
            wait_phase(bar(C::kBarQFull), 0, abort_flag, p, 3, false);
            for (int s = 0; s < C::kKStages && s < nk; ++s) {
                const int last = s + ((nk - 1 - s) / C::kKStages) * C::kKStages;
                wait_phase(bar(C::kBarKFull + s), (last / C::kKStages) & 1, abort_flag, p, 3, false);
            }
            for (int s = 0; s < C::kVStages && s < nv; ++s) {
                const int last = s + ((nv - 1 - s) / C::kVStages) * C::kVStages;
                wait_phase(bar(C::kBarVFull + s), (last / C::kVStages) & 1, abort_flag, p, 3, false);
            }
        }
    } else if (warp == kTransposeWarp) {
        // ------------------------------------------ fp32: V^T tiles (else idle)
        if constexpr (TF32) transpose_tf32<D>(p, smem, sbase, lane, T, abort_flag);
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ------------------------------------------------ tensor-core issuers
        // One issuing thread per query tile (warp 8: tile 0, warp 10: tile 1),
        // so each tile's products are enqueued as soon as its P is ready,
        // never behind the other tile's instructions.  Both read the same K/V
        // stages; each stage is released when both issuers' products that
        // read it have completed (empty barriers count two commits).
        if (lane == 0 && !(one_tile && warp == kMmaWarp2)) {
            const int w = (warp == kMmaWarp) ? 0 : 1;
            const uint32_t dS = tmem + 128u * static_cast<uint32_t>(w);
            const uint32_t dO = tmem + C::kColO + static_cast<uint32_t>(D * w);
            // P_w: over S_w, or its own columns (kEarlyS)
            const uint32_t dP = C::kEarlyS ? tmem + C::kColP + 64u * static_cast<uint32_t>(w) : dS;
            const uint32_t sQ = sbase + C::kOffQ + w * C::kTileBytes;
            // A k-step's descriptor at d = 128: the tile's, plus the step's
            // byte offset / 16 in the start-address field (no carry: shared
            // memory lies below 256 KB), fewer instructions for the issuing
            // thread, which shares its scheduler with a softmax warp
            // (measured +1 % on the headline shape; -1 % at d = 64, which
            // keeps the per-step descriptor).
            constexpr bool kDescAdd = D == 128 && !TF32;
            const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024);
            auto issue_qk = [&](int ks) {
                const uint32_t sK = sbase + C::kOffK + ks * C::kTileBytes;
                const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < C::kQkSteps; ++kk) {
                    const uint32_t off = (kk * 32) / 128 * C::kAtomBytes + (kk * 32) % 128;
                    const uint64_t da = kDescAdd ? dQ0 + (off >> 4) : smem_desc_sw128(sQ + off, 16, 1024);
                    const uint64_t db = kDescAdd ? dK0 + (off >> 4) : smem_desc_sw128(sK + off, 16, 1024);
                    mma_ss<TF32>(dS, da, db, C::kIdescQK, kk > 0 ? 1u : 0u);
                }
            };
            // k-steps [k0, k1) of O_w += P_w V
            auto issue_pv = [&](int vs, bool accumulate, int k0, int k1) {
                const uint32_t sV = sbase + C::kOffV + vs * C::kTileBytes;
#pragma unroll
                for (int kk = k0; kk < k1; ++kk) {
                    uint64_t db;
                    if constexpr (TF32) {
                        // V^T, K-major: 32-key atoms of D rows; a k-step is 8 keys (32 bytes)
                        db = smem_desc_sw128(sV + (kk / 4) * C::kVtAtomBytes + (kk % 4) * 32, 16, 1024);
                    } else {
                        // V, MN-major: 8-row groups 1024 bytes apart, 64-column blocks
                        // kAtomBytes apart; a k-step is 16 rows
                        db = kDescAdd ? smem_desc_sw128(sV, C::kAtomBytes, 1024) + ((kk * C::kUmmaK * 128) >> 4)
                                      : smem_desc_sw128(sV + kk * C::kUmmaK * 128, C::kAtomBytes, 1024);
                    }
                    mma_ts<TF32>(dO, dP + kk * 8, db, C::kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
                }
            };

            bool ok = wait_phase(bar(C::kBarQFull), 0, abort_flag, p, 4);
            if (ok) ok = wait_phase(bar(C::kBarKFull + 0), 0, abort_flag, p, 4);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
                if (!C::kStageDone) tc_commit(bar(C::kBarSFull + w));
                tc_commit(bar(C::kBarKEmpty + 0));
            }
            for (int j = 0; ok && j < T; ++j) {
                const int vs = j % C::kVStages;
                const int ks = (j + 1) % C::kKStages;
                if (C::kEarlyS && j + 1 < T) {
                    // S(j+1) as soon as the softmax has read S(j)
                    ok = wait_phase(bar(C::kBarSFree + w), j & 1, abort_flag, p, 14);
                    if (!ok) break;
                    ok = wait_phase(bar(C::kBarKFull + ks), ((j + 1) / C::kKStages) & 1, abort_flag, p, 7);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(ks);
                    if (!C::kStageDone) tc_commit(bar(C::kBarSFull + w));
                    tc_commit(bar(C::kBarKEmpty + ks));
                }
                ok = wait_phase(bar(C::kBarVFull + vs), (j / C::kVStages) & 1, abort_flag, p, 5);
                if (!ok) break;
                // the first half of P (keys 0-63) is published before the
                // second, so its products start while the softmax finishes
                ok = wait_phase(bar(C::kBarPFull + 2 * w), j & 1, abort_flag, p, 6);
                if (!ok) break;
                tc_fence_after();
                issue_pv(vs, j > 0, 0, C::kPvSteps / 2);
                ok = wait_phase(bar(C::kBarPFull + 2 * w + 1), j & 1, abort_flag, p, 6);
                if (!ok) break;
                tc_fence_after();
                issue_pv(vs, true, C::kPvSteps / 2, C::kPvSteps);
                tc_commit(bar(C::kBarVEmpty + vs));
                if (C::kEarlyS) {
                    if (!C::kStageDone) tc_commit(bar(C::kBarPVDone + w));
                    if (j + 1 == T) tc_commit(bar(C::kBarOFull + w));
                } else if (j + 1 < T) {
                    ok = wait_phase(bar(C::kBarKFull + ks), ((j + 1) / C::kKStages) & 1, abort_flag, p, 7);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(ks);
                    tc_commit(bar(C::kBarSFull + w));
                    tc_commit(bar(C::kBarKEmpty + ks));
                } else {
                    tc_commit(bar(C::kBarOFull + w));
                }
            }
            // Drain every tensor-core operation this thread issued before the
            // tensor memory is released.
            tc_commit(bar(C::kBarDrain + w));
            wait_phase(bar(C::kBarDrain + w), 0, abort_flag, p, 9, false);
        }
      }
        // The in-cluster merge after the role branches runs in every warp:
        // back to the launch allocation first (this waits until the softmax
        // warpgroups have returned theirs, which they do after their last
        // wait).
        if (!kOneTile && p.cluster) regs_increase<kLaunchRegs>();
    } else {
        // ------------------------------------------------ softmax warpgroups
        regs_increase<C::kSoftmaxRegs>();
        const int w = warp / 4;   // query tile of this warpgroup
        const int wi = warp % 4;  // TMEM lane quarter this warp may access
        const int t = wi * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wi * 32) << 16;
        const uint32_t tS = tmem + lane_off + 128u * static_cast<uint32_t>(w);
        const uint32_t tO = tmem + lane_off + C::kColO + static_cast<uint32_t>(D * w);
        // where this warp writes P: over its scores, or P_w's own columns (kEarlyS)
        const uint32_t tP = C::kEarlyS ? tmem + lane_off + C::kColP + 64u * static_cast<uint32_t>(w) : tS;
        const float c = p.scale_log2;
        const bool active = !(one_tile && w == 1);  // this warpgroup's tile has rows
        const bool take_turns = C::kTakeTurns && !one_tile;

        // keys of this row's head visible to this row: all Nkv, or under the
        // causal mask those up to i + causal_offset (may be none)
        // this thread's query row: (query head, query index i) and its row in
        // the [B*H, Nq] outputs (-1: a tile row that holds no query row)
        long long qi = row0 + w * kTileM + t;
        long long out_row = qi < p.Nq ? static_cast<long long>(bh) * p.Nq + qi : -1;
        if (pack) {
            const int r = w * kTileM + t;
            qi = r < pack_rows ? r % p.Nq : 0;
            out_row = r < pack_rows ? (static_cast<long long>(bh) * p.group + r / p.Nq) * p.Nq + qi : -1;
        }
        int row_limit = p.Nkv;
        if (kCausal) {
            const long long lim = qi + p.causal_offset + 1;
            row_limit = static_cast<int>(max(-1ll, min(static_cast<long long>(p.Nkv), lim)));
        }
        float m_ref = -INFINITY;  // reference maximum, base-2 scaled units
        float l = 0.0f;           // running sum of the weights p (fp32): gives lse
        float lq = 0.0f;          // running sum used to normalise O: l with each
                                  // tile's largest weight as rounded for P V
        bool ok = true;

        if constexpr (TF32) {
            // fp32 inputs: this warpgroup rounds its query tile to TF32 in
            // place (it is idle until the first scores); the issuers start
            // once all eight softmax warps have arrived
            if (has_work) {
                ok = __all_sync(0xffffffffu, wait_phase(bar(C::kBarQRaw), 0, abort_flag, p, 16));
                if (ok) {
                    round_tf32_inplace(smem + C::kOffQ + w * C::kTileBytes, C::kTileBytes / 16, t, kTileM);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::kBarQFull));
                }
            }
        }

        // Where they take turns (kTakeTurns), the two softmax warpgroups go
        // 0, 1, 0, 1, ...: one runs its exponentials while the other tile's
        // products occupy the tensor core (see kTurnAfterHalf for how far the
        // turns overlap).  Unmasked 16-bit launches pass the turn warp to
        // warp (warp i of one warpgroup to warp i of the other, on the same
        // scheduler) through shared counters the waiting warp spins on
        // (+1 % on the headline shape); the others through mbarriers (the
        // counters measured 1 % slower on the causal headline).
        constexpr bool kFlagTurns = !TF32 && !kCausal;
        volatile uint32_t* const turn_mine = reinterpret_cast<volatile uint32_t*>(smem + C::kOffTurnFlags) + 4 * w + wi;
        volatile uint32_t* const turn_other =
            reinterpret_cast<volatile uint32_t*>(smem + C::kOffTurnFlags) + 4 * (1 - w) + wi;
        // hand the turn to the other warpgroup after this one's tile j
        auto pass_turn = [&](int j) {
            if (kFlagTurns) {
                *turn_other = static_cast<uint32_t>(j + 1 + w);
            } else {
                mbar_arrive(bar(C::kBarTurn + (1 - w)));
            }
        };
        if (!kFlagTurns && take_turns && w == 1 && lane == 0) mbar_arrive(bar(C::kBarTurn + 0));
        const int T_rows = active ? T : 0;
        for (int j = 0; j < T_rows; ++j) {  // T <= 0: no key tile
            // S_w(j) computed (kStageDone: both tiles' scores, which release K stage j)
            bool got = C::kStageDone ? wait_phase(bar(C::kBarKEmpty + j % C::kKStages), (j / C::kKStages) & 1,
                                                  abort_flag, p, 10)
                                     : wait_phase(bar(C::kBarSFull + w), j & 1, abort_flag, p, 10);
            ok = __all_sync(0xffffffffu, got);
            if (!ok) break;
            if (take_turns) {
                got = kFlagTurns ? wait_flag(turn_mine, static_cast<uint32_t>(j + 1), abort_flag, p, 13)
                                 : wait_phase(bar(C::kBarTurn + w), j & 1, abort_flag, p, 13);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) break;
            }
            tc_fence_after();

            // the scores; at d = 64 with each 32-key quarter's maximum (the
            // reducing load: the row maximum of an unmasked tile for c >= 0
            // then costs no instruction of this warp; measured +2 to +3 % at
            // d = 64, -1 % at d = 128, where the computed maximum overlaps
            // the speculative first-half exponentials)
            uint32_t s[4][32];
            float qmax[4];
            if constexpr (C::kHwMax) {
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32_max(tS + 32u * q, s[q], qmax[q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld_wait_red(s[q], qmax[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(tS + 32u * q, s[q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld_wait(s[q]);
            }
            // maximum of an unmasked tile's scores (c >= 0)
            auto unmasked_max = [&]() -> float {
                if constexpr (C::kHwMax) return fmaxf(fmax3(qmax[0], qmax[1], qmax[2]), qmax[3]);
                else return row_extreme<true>(s);
            };
            if constexpr (C::kEarlyS) {
                // S_w may be overwritten by the next tile's scores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarSFree + w));
            }
            // kEarlyS: P_w and O_w hold tile j-1's product until it completes
            // (that product is not ordered before this tile's scores)
            auto wait_prev_product = [&]() -> bool {
                if (!C::kEarlyS || j == 0) return true;
                // (kStageDone: both tiles' products, which release V stage j-1)
                const bool done = C::kStageDone ? wait_phase(bar(C::kBarVEmpty + (j - 1) % C::kVStages),
                                                             ((j - 1) / C::kVStages) & 1, abort_flag, p, 15)
                                                : wait_phase(bar(C::kBarPVDone + w), (j - 1) & 1, abort_flag, p, 15);
                return __all_sync(0xffffffffu, done);
            };

            // keys of this tile visible to this row (<= 0: none, >= 128: all);
            // masking is decided per warp (tcgen05.st is warp-collective)
            const int valid = row_limit - (t_begin + j) * kTileN;
            // (without the causal mask `valid` is the same for every row)
            const bool masked = kCausal ? __any_sync(0xffffffffu, valid < kTileN) : (valid < kTileN);
            if (masked) {
                // keys past N: copy key 0's score so they cannot win the max;
                // their weight is zeroed below
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (q * 32 + i >= valid) s[q][i] = s[0][0];
            }

            // Speculation (16-bit inputs, unmasked tiles after the first; at
            // d = 128 without the causal mask only): the first half's
            // exponentials against the current reference run while the row
            // maximum reduces.  When no row of the warp moves its reference
            // (the lazy threshold below), they are exactly the values the
            // path below would compute and are published as they are;
            // otherwise that path recomputes them.  (d = 64: +5 to +8 %;
            // d = 128: +1 % with the flag turns, -1 % on causal launches.)
            if constexpr (!TF32 && (D == 64 || !kCausal)) {
                if (!masked && j > 0) {
                    const float shift_s = (m_ref == -INFINITY) ? 0.0f : m_ref;
                    const uint64_t c2s = f2_pack(c, c);
                    const uint64_t ns2s = f2_pack(-shift_s, -shift_s);
                    uint32_t pw0[32];
                    uint64_t acc_s[4] = {0, 0, 0, 0};
                    exp_half_regs<F16>(s, c2s, ns2s, 0, pw0, acc_s);
                    const float mx_s = (c >= 0.0f) ? unmasked_max() : row_extreme<false>(s);
                    const bool need_s = mx_s * c > m_ref + kRescaleThreshold;
                    if (!__any_sync(0xffffffffu, need_s)) {
                        if (!wait_prev_product()) {
                            ok = false;
                            break;
                        }
                        tmem_st32(tP, pw0);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::kBarPFull + 2 * w + 0));
                        if (take_turns && C::kTurnAfterHalf == 0 && lane == 0) pass_turn(j);
                        exp_half<TF32, F16, false>(s, c2s, ns2s, valid, tP, 1, acc_s);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::kBarPFull + 2 * w + 1));
                        if (take_turns && C::kTurnAfterHalf == 1 && lane == 0) pass_turn(j);
                        const float tsum = sum8(acc_s);
                        const float pmax = ex2(fmaf(mx_s, c, -shift_s));
                        const float pmax_r = widen_lo16<F16>(pack_16x2<F16>(pmax, 0.0f));
                        l += tsum;
                        lq += tsum + (pmax_r - pmax);  // the exact path's order of operations
                        continue;
                    }
                }
            }

            // tile maximum of t = s * c (c may be negative or zero); a masked
            // tile's comes from the scores as masked above
            const float mx = (c >= 0.0f) ? (masked ? row_extreme<true>(s) : unmasked_max()) : row_extreme<false>(s);
            const float m_tile = (!kCausal || valid > 0) ? mx * c : -INFINITY;
            const float m_new = fmaxf(m_ref, m_tile);
            const bool need = m_new > m_ref + kRescaleThreshold;  // always true on the first tile

            // per-row factor for the accumulator (1 where the reference stays)
            const float alpha = need ? ex2(m_ref - m_new) : 1.0f;
            if (need) {
                l *= alpha;  // alpha = 0 on the first tile (l was 0 anyway)
                lq *= alpha;
                m_ref = m_new;
            }
            const float shift = (m_ref == -INFINITY) ? 0.0f : m_ref;

            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O holds the previous tiles' contributions (their products
                // completed before this tile's scores were signalled, or, with
                // kEarlyS, once the last one signals); the next product into
                // O waits for this warp's first arrival.
                if (!wait_prev_product()) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32u * q, o);
                    tmem_ld_wait(o);
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(u2f(o[i]), u2f(o[i + 1])), a2), x0, x1);
                        o[i] = f2u(x0);
                        o[i + 1] = f2u(x1);
                    }
                    tmem_st32(tO + 32u * q, o);
                }
            }

            // p = 2^(s*c - shift), two keys at a time (f32x2), written over
            // the scores in two halves; each half is published on its own
            // barrier so its products can start early
            const uint64_t c2 = f2_pack(c, c);
            const uint64_t ns2 = f2_pack(-shift, -shift);
            uint64_t acc[4] = {0, 0, 0, 0};
            if (!wait_prev_product()) {
                ok = false;
                break;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (masked) {
                    exp_half<TF32, F16, true>(s, c2, ns2, valid, tP, h, acc);
                } else {
                    exp_half<TF32, F16, false>(s, c2, ns2, valid, tP, h, acc);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPFull + 2 * w + h));
                if (take_turns && h == C::kTurnAfterHalf && lane == 0) pass_turn(j);
            }
            // l: fp32 sum of the weights (gives lse).  lq: the same sum with
            // the tile's largest weight replaced by its value as rounded for
            // the P V product (bf16 or TF32; same FMA, exponential and
            // rounding as the element itself).  A weight that dominates a
            // row then enters the normalisation exactly as it entered O.
            const float tsum = sum8(acc);
            const float pmax = ex2(fmaf(mx, c, -shift));
            const float pmax_r = TF32 ? u2f(round_tf32(pmax)) : widen_lo16<F16>(pack_16x2<F16>(pmax, 0.0f));
            l += tsum;
            lq += tsum + ((!kCausal || valid > 0) ? pmax_r - pmax : 0.0f);
        }

        // ------------------------------------------------------- epilogue
        if (ok && has_work && active) {
            bool got = wait_phase(bar(C::kBarOFull + w), 0, abort_flag, p, 11);
            ok = __all_sync(0xffffffffu, got);
        }
        uint8_t* stage = smem + C::kOffQ + w * C::kTileBytes;  // Q_w is free after its last S MMA
        const bool split_mode = p.splits > 1;
        if (ok && split_mode && active) {
            tc_fence_after();
            if (has_work) {
                store_partial<D>(p, tO, out_row, m_ref, l, lq, stage + t * 16);
            } else if (!kOneTile && p.cluster) {
                // no visible key: weight 0 in the in-cluster merge
                *reinterpret_cast<float4*>(stage + t * 16) = make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
            } else if (out_row >= 0) {
                // an empty partition: weight 0 in the merge (its O slot is not read)
                const size_t r = split * static_cast<size_t>(p.part_rows) + static_cast<size_t>(out_row - p.part_row0);
                *reinterpret_cast<float4*>(p.ml_part + r * 4) = make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
            }
        }
        if (ok && !split_mode && active) {
            tc_fence_after();
            const float inv_l = lq > 0.0f ? 1.0f / lq : 0.0f;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                if (has_work) {
                    tmem_ld32(tO + 32u * q, o);
                    tmem_ld_wait(o);
                } else {  // no visible key: O = 0 (and lse = -inf below)
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if constexpr (TF32) {
                    // 32 fp32 = one 128-byte swizzle row of atom q
                    uint8_t* rowp = stage + q * C::kAtomBytes + t * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 v4;
                        v4.x = f2u(u2f(o[4 * ch + 0]) * inv_l);
                        v4.y = f2u(u2f(o[4 * ch + 1]) * inv_l);
                        v4.z = f2u(u2f(o[4 * ch + 2]) * inv_l);
                        v4.w = f2u(u2f(o[4 * ch + 3]) * inv_l);
                        *reinterpret_cast<uint4*>(rowp + ((ch ^ (t & 7)) << 4)) = v4;
                    }
                } else {
                    // 32 bf16 / fp16 = half a swizzle row: chunks 4*(q%2) .. +3 of atom q/2
                    uint8_t* rowp = stage + (q / 2) * C::kAtomBytes + t * 128;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int ch = (q % 2) * 4 + cc;
                        uint4 v4;
                        v4.x = pack_16x2<F16>(u2f(o[8 * cc + 0]) * inv_l, u2f(o[8 * cc + 1]) * inv_l);
                        v4.y = pack_16x2<F16>(u2f(o[8 * cc + 2]) * inv_l, u2f(o[8 * cc + 3]) * inv_l);
                        v4.z = pack_16x2<F16>(u2f(o[8 * cc + 4]) * inv_l, u2f(o[8 * cc + 5]) * inv_l);
                        v4.w = pack_16x2<F16>(u2f(o[8 * cc + 6]) * inv_l, u2f(o[8 * cc + 7]) * inv_l);
                        *reinterpret_cast<uint4*>(rowp + ((ch ^ (t & 7)) << 4)) = v4;
                    }
                }
            }
            if (p.lse != nullptr && out_row >= 0) {
                const float lse2 = (l > 0.0f) ? (m_ref + log2f(l)) : -INFINITY;
                p.lse[out_row] = lse2 * 0.69314718055994531f;
            }
            fence_proxy_async_smem();
        }
        // Every thread of the warpgroup arrives exactly once, whatever happened.
        mbar_arrive(bar(C::kBarEpi + w));
        if (t == 0) {
            const bool all_in = wait_phase(bar(C::kBarEpi + w), 0, abort_flag, p, 12);
            // a tile lying entirely past Nq has nothing to store
            if (all_in && !split_mode && !*abort_flag) {
                if (pack) {
                    // the Nq x group query rows of tile 0 (tile 1 holds none)
                    if (w == 0) {
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_store_3d(&map_o, smem_u32(stage + a * C::kAtomBytes), a * C::kAtomElems, 0,
                                         bh * p.group);
                        tma_store_commit();
                        tma_store_wait_read();
                    }
                } else if (row0 + w * kTileM < p.Nq) {
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_store_3d(&map_o, smem_u32(stage + a * C::kAtomBytes), a * C::kAtomElems,
                                     row0 + w * kTileM, bh);
                    tma_store_commit();
                    tma_store_wait_read();
                }
            }
        }
        // back to the launch allocation for the in-cluster merge (see warpgroup 2)
        if (!kOneTile && p.cluster) regs_decrease<kLaunchRegs>();
    }

    // ------------------------------------------------ in-cluster merge
    if (!kOneTile && p.cluster) {
        // every role is done: both tiles' products completed (the softmax
        // warpgroups waited for them), every TMA load landed (the producer
        // drained), and the row statistics are in shared memory
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        cluster_merge<TF32, D, F16>(p, smem, sbase, tmem, !skip && *abort_flag == 0u, has_work, row0, bh,
                                    abort_flag);
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // launched with programmatic serialization (the split last wave): this
    // CTA completes only after the grid before it in the stream, so that
    // work after this launch still sees both (returns at once otherwise)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;");
}

template <bool TF32, int D, bool F16, bool kCausal, bool kOneTile>
cudaError_t launch_fwd_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                               cudaStream_t stream) {
    using C = FwdCfg<TF32, D, F16>;
    auto kern = fa_fwd_kernel<TF32, D, F16, kCausal, kOneTile>;
    // The register split above relies on the compiled kernel holding exactly
    // kLaunchRegs per thread; refuse to launch otherwise (a setmaxnreg.inc
    // without the registers behind it would never return).
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    if (p.cluster) {
        // the p.splits partitions of a query block form one cluster
        // (consecutive blockIdx.x, so a CTA's cluster rank is its partition)
        if (kOneTile || p.splits < 2 || p.splits > C::kMaxMergeParts || grid % static_cast<unsigned>(p.splits) != 0)
            return cudaErrorInvalidConfiguration;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr_cluster[2];
        attr_cluster[0].id = cudaLaunchAttributeClusterDimension;
        attr_cluster[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
        attr_cluster[0].val.clusterDim.y = 1;
        attr_cluster[0].val.clusterDim.z = 1;
        cfg.attrs = attr_cluster;
        cfg.numAttrs = 1;
        // the last wave of an automatic plan (item_offset > 0) follows the
        // full waves' launch and shares no data with it: its CTAs may start
        // as that launch's CTAs finish
        if (p.item_offset > 0) {
            attr_cluster[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr_cluster[1].val.programmaticStreamSerializationAllowed = 1;
            cfg.numAttrs = 2;
        }
        e = cudaLaunchKernelEx(&cfg, kern, q, k, v, o, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(q, k, v, o, p);
    return cudaGetLastError();
}

}  // namespace fa

namespace fa {
// Causal and unmasked kernels are separate instantiations (the unmasked one
// keeps a tile's key count uniform across rows), and so are packed and
// unpacked ones.
template <bool TF32, int D, bool F16 = false>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                       cudaStream_t stream) {
    if (p.pack)
        return p.causal ? launch_fwd_variant<TF32, D, F16, true, true>(q, k, v, o, p, grid, stream)
                        : launch_fwd_variant<TF32, D, F16, false, true>(q, k, v, o, p, grid, stream);
    return p.causal ? launch_fwd_variant<TF32, D, F16, true, false>(q, k, v, o, p, grid, stream)
                    : launch_fwd_variant<TF32, D, F16, false, false>(q, k, v, o, p, grid, stream);
}
}  // namespace fa
