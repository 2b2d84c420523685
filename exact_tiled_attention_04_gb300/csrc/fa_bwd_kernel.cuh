// Backward pass of exact attention for sm_103a (GB300).
//
// What it computes: the gradients of O = softmax(scale Q K^T) V for an
// upstream gradient dO, recomputing the attention blocks from Q, K, V and the
// saved softmax statistic (lse) instead of storing the N x N matrix
// ("FlashAttention dissected", section "Memory complexity: from O(N^2) to
// O(N)"), with the exact gradient of the softmax formula of the same page:
//   P = exp(scale S - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D),  D_i = dO_i . O_i (= sum_j P_ij dP_ij),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Organisation (one CTA = 128 keys of one (batch, key/value head); it sweeps
// every 128-row query tile of the head's query heads; 384 threads):
//   warps 0-3  gradient warpgroup 0: query columns 0-63 of each tile
//   warps 4-7  gradient warpgroup 1: query columns 64-127
//   warp  8    tensor-core issuer (one thread) and TMEM owner
//   warp  9    TMA producer (one thread)
//   warp 10    dQ reducer (one thread): TMA tensor reductions of the
//              staged dQ into the fp32 accumulator
//   warp 11    idle (completes warpgroup 2 for the register reallocation)
//   warps 12-15 (read-out layout only) dQ read-out warpgroup
// Each thread of a gradient warpgroup owns one key row (its TMEM lane) and
// half of the query columns.  The scores are computed transposed (keys on
// the lanes) so that dK and dV accumulate in tensor memory for the whole
// sweep, and P^T and dS^T are the A operands of their products straight
// from tensor memory.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0, 128)        S^T = K Q^T of the current tile; warpgroup w then writes
//                   P^T (bf16/fp16 pairs) over its columns [64w, 64w + 32).
//   [128, 256)      dP^T = V dO^T; warpgroup w then writes dS^T over
//                   [128 + 64w, 128 + 64w + 32).
//   [256, 256 + d)  dV accumulator;  [256 + d, 256 + 2d)  dK accumulator.
//   dQ = dS K of a tile (query rows on the lanes, d columns): columns
//   [384, 448) for d = 64; for d = 128 over the dP^T columns, so the next
//   tile's dP^T waits until this dQ has been read out.
// Per query tile j the issuer enqueues dP^T(j), dV(j) += P^T dO once P^T(j)
// is written, S^T(j+1) (over P^T(j), which dV(j) has consumed: one issuing
// thread, executed in order), then dK(j) += dS^T Q and dQ(j) = dS K once
// dS(j) is written.  The gradient warpgroups form dS(j), then P^T(j+1) while
// dK(j) and dQ(j) run, then read dQ(j) out: staged (fp32) in the stage's Q
// and dO tiles, free once dQ(j) is computed, and added into an fp32
// accumulator in global memory with TMA tensor reductions (whole 128-byte
// lines); the stage goes back to the producer when both reductions have read
// it.  A last kernel scales and converts the accumulator.
//
// Read-out layout (d = 128 without the causal mask; 512 threads): warps
// 12-15 form a fourth warpgroup that reads each tile's dQ out of tensor
// memory, one query row a thread, so the gradient warpgroups go straight
// from dS(j) to P^T(j+1).  The issuer then enqueues dQ(j) before dK(j), and
// the next tile's scores after both (issued earlier they would wait in
// front of dQ(j) for the next Q tile, whose stage is still being reduced
// from).  The read-out warpgroup stages dQ columns [d/2, d) in the dO tile
// as soon as dQ(j) is computed (dV(j) ran before it) and [0, d/2) in the
// Q tile once dK(j) is; the reducer adds each half as soon as it is staged.
// With the causal mask (short sweeps, where a CTA's fixed cost weighs
// more) and at d = 64 (dQ in its own columns, so the next scores go early)
// the 384-thread layout measured faster.
//
// Shared memory (128-byte-swizzled TMA tiles, 1024-byte aligned): K and V of
// the key block (reused as the dK / dV output staging), a two-stage ring of
// Q, dO and row-statistics tiles, and dS (128 keys x 128 queries, the
// MN-major A operand of dQ = dS K).
//
// Every wait on an mbarrier is bounded as in the forward kernel: after about
// a second the CTA raises its abort flag and the device error word, every
// role leaves its loop, in-flight tensor-core work and TMA loads are
// drained, and tensor memory is freed before the CTA exits.
#pragma once

#include <cmath>
#include <cstdint>

#include "fa_bwd_internal.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr int kBwdMmaWarp = 8;
constexpr int kBwdLoadWarp = 9;
constexpr int kBwdReduceWarp = 10;
constexpr int kBwdReadWarp0 = 12;  // read-out layout: first warp of the dQ read-out warpgroup
constexpr uint32_t kBwdTmemCols = 512;
constexpr uint64_t kBwdWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s
constexpr int kBwdStatBytes = kStatFloatsPerTile * static_cast<int>(sizeof(float));  // one query tile

// The read-out layout (a dQ read-out warpgroup of its own) for d = 128
// without the causal mask; the 384-thread layout otherwise.
template <int D, bool kCausal>
constexpr bool bwd_read_layout() {
    return D == 128 && !kCausal;
}

template <int D, bool F16, bool kRead>
struct BwdCfg {
    static constexpr int kAtomElems = 64;                // 16-bit elements per 128-byte row
    static constexpr int kAtoms = D / kAtomElems;
    static constexpr int kAtomBytes = 128 * 128;         // 128 rows x 128 bytes
    static constexpr int kTileBytes = kAtoms * kAtomBytes;  // 128 rows x D
    static constexpr int kUmmaK = 16;
    static constexpr int kDSteps = D / kUmmaK;           // k-steps of S^T and dP^T (over d)
    static constexpr int kRowSteps = 128 / kUmmaK;       // k-steps over 128 query rows or keys
    // Q/dO stages: the stage of tile j is handed back only when tile j's dQ
    // reduction (staged in it) has been read, so deeper rings hide that
    // latency; d = 128 fits two stages, d = 64 four.
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr uint32_t kFmt = F16 ? 0u : 1u;
    // S^T = K Q^T and dP^T = V dO^T: M = 128 keys, N = 128 query rows, both K-major.
    static constexpr uint32_t kIdescS = instr_desc(kFmt, false, false, 128, 128);
    // dV += P^T dO and dK += dS^T Q: A from TMEM, B ([query rows x d]) MN-major.
    static constexpr uint32_t kIdescAcc = instr_desc(kFmt, false, true, 128, D);
    // dQ = dS K: A = dS (shared memory, stored keys x queries: MN-major),
    // B = K ([keys x d]) MN-major; M = 128 query rows.
    static constexpr uint32_t kIdescDQ = instr_desc(kFmt, true, true, 128, D);

    static constexpr int kThreads = kRead ? 512 : 384;
    static constexpr uint32_t kLaunchRegs = kRead ? 128 : 168;
    // register split (setmaxnreg): gradient warpgroups / warpgroup 2 / read-out warpgroup
    static constexpr uint32_t kGradRegs = kRead ? 160 : 208;
    static constexpr uint32_t kOtherRegs = kRead ? 96 : 88;
    static constexpr uint32_t kReadRegs = kRead ? 96 : 0;
    static_assert(2 * 128 * kGradRegs + 128 * kOtherRegs + 128 * kReadRegs == kThreads * kLaunchRegs,
                  "register split must equal the launch allocation");

    // shared-memory map (offsets from the 1024-aligned base)
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;                 // [kStages]
    static constexpr int kOffDO = kOffQ + kStages * kTileBytes;      // [kStages]
    static constexpr int kOffDS = kOffDO + kStages * kTileBytes;     // 128 x 128, two atoms
    static constexpr int kOffStats = kOffDS + 2 * kAtomBytes;        // [kStages] x 1 KB
    static constexpr int kTilesEnd = kOffStats + kStages * kBwdStatBytes;

    // barrier slots
    static constexpr int kBarKV = 0;
    // A stage is two halves with their own barriers: Q with the row
    // statistics, and dO.  Each half is handed back as soon as the dQ
    // reduction staged in it has read it.
    static constexpr int kBarFull = 1;                      // [kStages] Q + statistics landed
    static constexpr int kBarFullDO = kBarFull + kStages;   // [kStages] dO landed
    static constexpr int kBarEmpty = kBarFullDO + kStages;  // [kStages] Q half free
    static constexpr int kBarEmptyDO = kBarEmpty + kStages; // [kStages] dO half free
    static constexpr int kBarS = kBarEmptyDO + kStages;     // S^T computed
    static constexpr int kBarDP = kBarS + 1;           // dP^T computed
    static constexpr int kBarP = kBarDP + 1;           // P^T in TMEM (8 warp arrivals)
    static constexpr int kBarDS = kBarP + 1;           // dS^T in TMEM and dS in smem (8)
    static constexpr int kBarDQ = kBarDS + 1;          // dQ computed
    static constexpr int kBarDK = kBarDQ + 1;          // read-out layout: dK computed, the Q tile read
    static constexpr int kBarDQFree = kBarDK + 1;      // dQ read out (8; read-out layout 4)
    static constexpr int kBarAcc = kBarDQFree + 1;     // dK, dV final
    static constexpr int kBarDrain = kBarAcc + 1;
    static constexpr int kBarEpi = kBarDrain + 1;      // [2]
    // [kStages]: the tile's dQ is staged (8); read-out layout: its columns
    // [0, d/2), in the Q tile (4)
    static constexpr int kBarStaged = kBarEpi + 2;
    static constexpr int kBarStagedDO = kBarStaged + kStages;  // [kStages] read-out layout: [d/2, d), in the dO tile (4)
    static constexpr int kNumBars = kBarStagedDO + kStages;
    // barriers, TMEM slot and abort flag
    static constexpr int kCtrlBytes = kNumBars * 8 + 8;
    // The control block lives in whichever alignment gap holds it: below the
    // 1024-aligned base when the slack there is large enough, else after the
    // tiles, so the launch needs only the tiles plus 1 KB.
    static constexpr size_t kSmemBytes = static_cast<size_t>(kTilesEnd) + 1024;
    static_assert(kCtrlBytes <= 512, "control block must fit either gap");
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
    static_assert(256 + 2 * D <= static_cast<int>(kBwdTmemCols), "tensor memory budget exceeded");

    // tensor-memory columns
    static constexpr uint32_t kColS = 0;      // S^T; P^T of warpgroup w at [64w, 64w + 32)
    static constexpr uint32_t kColDP = 128;   // dP^T; dS^T of warpgroup w at [128 + 64w, 128 + 64w + 32)
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
    // dQ of a tile: its own columns when they fit (d = 64), else over the dP
    // columns (d = 128), which the next tile's dP^T may then only overwrite
    // once dQ has been read out
    static constexpr bool kDqOwnCols = 256 + 3 * D <= static_cast<int>(kBwdTmemCols);
    static constexpr uint32_t kColDQ = kDqOwnCols ? 256 + 2 * D : 128;
    // Issue order.  With dQ in its own columns, S^T(j+1) goes right after
    // dV(j) and the gradient warpgroups form P^T(j+1) while dK(j) and dQ(j)
    // run.  With dQ over the dP^T columns, dP^T(j+1) must wait for the
    // read-out of dQ(j) anyway: S^T(j+1) then follows dQ(j) and runs during
    // that read-out, and P^T(j+1) comes after it.
    static constexpr bool kEarlyS = kDqOwnCols;
};

// Bounded wait on an mbarrier phase (the forward kernel's policy): returns
// false when the CTA is aborting (if `honor_abort`) or when this wait gave up
// after kBwdWaitLimitNs, in which case it raises the CTA's abort flag, sets
// the sticky device error bits (waiting role in bits 8-15) and marks this
// launch's generation as aborted.
__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         const BwdParams& bp, unsigned int where,
                                         bool honor_abort = true) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if ((++spins & 31u) == 0u) {
            if (honor_abort && *abort_flag) return false;
            if (global_timer_ns() - t0 > kBwdWaitLimitNs) {
                *abort_flag = 1u;
                atomicOr(&bp.status->word, kDevErrTimeout | (where << 8));
                atomicExch(&bp.status->abort_gen, bp.gen);
                return false;
            }
        }
    }
}

// Bulk copy of `bytes` (a multiple of 16) from global memory into this CTA's
// shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D tiled reduction shared -> global: the box at (c0, c1, c2) is added
// element-wise (fp32) into the tensor; rows outside the tensor are skipped.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float bwd_u2f(uint32_t x) { return __uint_as_float(x); }

// 32 lanes x 16 consecutive fp32 columns of tensor memory, and the wait for
// them (the registers tied so that no use is scheduled before it).
__device__ __forceinline__ void bwd_tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void bwd_tmem_ld_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

template <int D, bool F16, bool kCausal>
__global__ void __launch_bounds__((BwdCfg<D, F16, bwd_read_layout<D, kCausal>()>::kThreads), 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                  const __grid_constant__ CUtensorMap map_dq, const BwdParams p) {
    constexpr bool kRead = bwd_read_layout<D, kCausal>();
    using C = BwdCfg<D, F16, kRead>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_u32 + pad;
    // control block: below the aligned base if the slack holds it, else after the tiles
    uint8_t* ctrl = (pad >= static_cast<uint32_t>(C::kCtrlBytes)) ? smem_raw : smem + C::kTilesEnd;
    const uint32_t ctrl_u32 = smem_u32(ctrl);

    const int warp = static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) % 32;
    // unit = b * H_kv + key/value head; kb = key block of the unit.  Causal:
    // key block 0 sees every query tile and later blocks fewer, so they go
    // heaviest first, by groups of units; otherwise blockIdx.x = unit *
    // n_kv_blocks + kb.
    int kb, unit;
    if (kCausal) {
        lpt_item(blockIdx.x, static_cast<int>(gridDim.x) / p.n_kv_blocks, p.n_kv_blocks, unit, kb);
    } else {
        kb = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.n_kv_blocks));
        unit = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.n_kv_blocks));
    }
    const int b = unit / p.H_kv;
    const int kvh = unit % p.H_kv;
    // Query tiles that see a key of this block: all, or under the causal mask
    // those holding a row i >= kb*128 - causal_offset (query i sees key j iff
    // j <= i + causal_offset).  The last query row sees every key, so at
    // least one tile remains.
    int qt_begin = 0;
    if (kCausal) {
        const long long first_i = static_cast<long long>(kb) * 128 - p.causal_offset;
        qt_begin = first_i <= 0 ? 0 : static_cast<int>(min(first_i / 128, static_cast<long long>(p.n_q_tiles)));
    }
    const int nqt = p.n_q_tiles - qt_begin;
    const int T = p.group * nqt;  // (query head, query tile) pairs swept by this CTA
    const bool has_work = T > 0;

    auto bar = [&](int i) -> uint32_t { return ctrl_u32 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + C::kNumBars * 8);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(ctrl + C::kNumBars * 8 + 4);

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarKV), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarFull + s), 1);
            mbar_init(bar(C::kBarFullDO + s), 1);
            mbar_init(bar(C::kBarEmpty + s), 1);
            mbar_init(bar(C::kBarEmptyDO + s), 1);
            mbar_init(bar(C::kBarStaged + s), kRead ? 4 : 8);
            mbar_init(bar(C::kBarStagedDO + s), 4);
        }
        mbar_init(bar(C::kBarS), 1);
        mbar_init(bar(C::kBarDP), 1);
        mbar_init(bar(C::kBarP), 8);  // one arrival per gradient warp
        mbar_init(bar(C::kBarDS), 8);
        mbar_init(bar(C::kBarDQ), 1);
        mbar_init(bar(C::kBarDK), 1);
        mbar_init(bar(C::kBarDQFree), kRead ? 4 : 8);
        mbar_init(bar(C::kBarAcc), 1);
        mbar_init(bar(C::kBarDrain), 1);
        mbar_init(bar(C::kBarEpi + 0), 128);
        mbar_init(bar(C::kBarEpi + 1), 128);
        // A CTA starting after another CTA of this launch timed out does no work.
        *abort_flag = (*reinterpret_cast<volatile unsigned int*>(&p.status->abort_gen) == p.gen) ? 1u : 0u;
        mbar_init_fence();
    }
    if (warp == kBwdLoadWarp && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        tma_prefetch_desc(&map_do);
        tma_prefetch_desc(&map_dq);
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0u;

    if (skip) {
        // nothing issued: go straight to the teardown
    } else if (kRead && warp >= kBwdReadWarp0) {
        // ------------------------------ dQ read-out warpgroup (read-out layout)
        // Tile j's dQ (query row t, all d columns): columns [d/2, d) into the
        // stage's dO tile once dQ(j) is computed (dV(j), the tile's last
        // reader, ran before it), then [0, d/2) into its Q tile once dK(j)
        // has read it; fp32 boxes of 32 columns with the 128-byte swizzle,
        // the layout the reducer's tensor reductions read.
        regs_decrease<C::kReadRegs>();
        const int wi = warp % 4;        // TMEM lane quarter this warp may access
        const int t = wi * 32 + lane;   // query row of the tile (= TMEM lane)
        const uint32_t tDQ = tmem + (static_cast<uint32_t>(wi * 32) << 16) + C::kColDQ;
        for (int it = 0; it < T; ++it) {
            const int s = it % C::kStages;
            bool got = bwd_wait(bar(C::kBarDQ), it & 1, abort_flag, p, 46);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            bool fine = true;
#pragma unroll
            for (int half = 1; half >= 0; --half) {
                if (half == 0) {
                    got = bwd_wait(bar(C::kBarDK), it & 1, abort_flag, p, 47);
                    fine = __all_sync(0xffffffffu, got);
                    if (!fine) break;
                }
                uint8_t* stg = smem + (half == 0 ? C::kOffQ : C::kOffDO) + s * C::kTileBytes;
#pragma unroll
                for (int k16 = 0; k16 < D / 32; ++k16) {  // 16 columns: half a box row
                    uint32_t v[16];
                    bwd_tmem_ld16(tDQ + static_cast<uint32_t>(half * (D / 2) + 16 * k16), v);
                    bwd_tmem_ld_wait16(v);
                    uint8_t* rowp = stg + (k16 / 2) * C::kAtomBytes + t * 128;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int ch = (k16 % 2) * 4 + c4;
                        *reinterpret_cast<uint4*>(rowp + ((ch ^ (t & 7)) << 4)) =
                            make_uint4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
                    }
                }
                if (half == 0) tc_fence_before();  // every load of dQ(j) precedes DQFree
                fence_proxy_async_smem();          // the staged rows are read by the TMA reductions
                __syncwarp();
                if (lane == 0) {
                    if (half == 0) mbar_arrive(bar(C::kBarDQFree));
                    mbar_arrive(bar((half == 0 ? C::kBarStaged : C::kBarStagedDO) + s));
                }
            }
            if (!fine) break;
        }
    } else if (warp >= 8) {
        regs_decrease<C::kOtherRegs>();
      if (!has_work) {
        // no query row sees this key block: the epilogue stores zeros
      } else if (warp == kBwdLoadWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();   // Q, dO, stats: read by every key block of the head
            const uint64_t once = policy_evict_first();  // K, V: read once
            mbar_arrive_expect_tx(bar(C::kBarKV), 2u * C::kTileBytes);
            for (int a = 0; a < C::kAtoms; ++a) {
                tma_load_3d(sbase + C::kOffK + a * C::kAtomBytes, &map_k, bar(C::kBarKV), a * C::kAtomElems,
                            kb * 128, unit, once);
                tma_load_3d(sbase + C::kOffV + a * C::kAtomBytes, &map_v, bar(C::kBarKV), a * C::kAtomElems,
                            kb * 128, unit, once);
            }
            int issued_q = 0, issued_do = 0;
            for (int it = 0; it < T; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = ((it / C::kStages) & 1) ^ 1;
                const int g = it / nqt;
                const int qt = qt_begin + it % nqt;
                const int bh = b * p.H + kvh * p.group + g;
                if (!bwd_wait(bar(C::kBarEmpty + s), ph, abort_flag, p, 31)) break;
                mbar_arrive_expect_tx(bar(C::kBarFull + s), C::kTileBytes + kBwdStatBytes);
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffQ + s * C::kTileBytes + a * C::kAtomBytes, &map_q,
                                bar(C::kBarFull + s), a * C::kAtomElems, qt * 128, bh, keep);
                bulk_load(sbase + C::kOffStats + s * kBwdStatBytes,
                          p.stats + (static_cast<size_t>(bh) * (p.Nq_pad / 128) + static_cast<size_t>(qt)) *
                                        kStatFloatsPerTile,
                          kBwdStatBytes, bar(C::kBarFull + s), keep);
                issued_q = it + 1;
                if (!bwd_wait(bar(C::kBarEmptyDO + s), ph, abort_flag, p, 31)) break;
                mbar_arrive_expect_tx(bar(C::kBarFullDO + s), C::kTileBytes);
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_3d(sbase + C::kOffDO + s * C::kTileBytes + a * C::kAtomBytes, &map_do,
                                bar(C::kBarFullDO + s), a * C::kAtomElems, qt * 128, bh, keep);
                issued_do = it + 1;
            }
            // Drain: every issued load has landed before the CTA may exit.
            bwd_wait(bar(C::kBarKV), 0, abort_flag, p, 32, false);
            for (int s = 0; s < C::kStages; ++s) {
                if (s < issued_q) {
                    const int last = s + ((issued_q - 1 - s) / C::kStages) * C::kStages;
                    bwd_wait(bar(C::kBarFull + s), (last / C::kStages) & 1, abort_flag, p, 32, false);
                }
                if (s < issued_do) {
                    const int last = s + ((issued_do - 1 - s) / C::kStages) * C::kStages;
                    bwd_wait(bar(C::kBarFullDO + s), (last / C::kStages) & 1, abort_flag, p, 32, false);
                }
            }
        }
      } else if (warp == kBwdReduceWarp) {
        // ------------------------------------------------------ dQ reducer
        // Adds each tile's staged dQ (warpgroup 0's columns in the stage's Q
        // tile, warpgroup 1's in its dO tile) into the fp32 accumulator and
        // hands the stage back to the producer once the reductions have read
        // it.  The gradient warpgroups never wait for the L2.
        // (Read-out layout: each half as soon as it is staged, the dO tile's
        // columns [d/2, d) first.)
        if (lane == 0) {
            for (int it = 0; it < T; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                const int qt = qt_begin + it % nqt;
                const int bh = b * p.H + kvh * p.group + it / nqt;
                if (!kRead && !bwd_wait(bar(C::kBarStaged + s), ph, abort_flag, p, 39)) break;
                bool got = true;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int w = kRead ? 1 - i : i;  // w = 0: columns [0, d/2) in the Q tile
                    if (kRead) {
                        got = bwd_wait(bar((w == 0 ? C::kBarStaged : C::kBarStagedDO) + s), ph, abort_flag, p, 39);
                        if (!got) break;
                    }
                    const uint32_t stg = sbase + (w == 0 ? C::kOffQ : C::kOffDO) + s * C::kTileBytes;
#pragma unroll
                    for (int h = 0; h < D / 64; ++h)
                        tma_reduce_add_3d(&map_dq, stg + h * C::kAtomBytes, w * (D / 2) + 32 * h, qt * 128, bh);
                    tma_store_commit();  // one group per half
                }
                if (!got) break;
                // the first-committed half has been read, then the other
                bulk_wait_read<1>();
                mbar_arrive(bar((kRead ? C::kBarEmptyDO : C::kBarEmpty) + s));
                bulk_wait_read<0>();
                mbar_arrive(bar((kRead ? C::kBarEmpty : C::kBarEmptyDO) + s));
            }
            bulk_wait_read<0>();  // nothing may still read shared memory at the exit
        }
      } else if (warp == kBwdMmaWarp) {
        // ------------------------------------------------ tensor-core issuer
        // Order per tile j: dP^T(j), dV(j) once P^T(j) is written, S^T(j+1)
        // right after (it overwrites P^T(j), which dV(j) has consumed: same
        // thread, the tensor core runs them in order), then dK(j) and dQ(j)
        // once dS(j) is written.  The gradient warpgroups compute P^T(j+1)
        // while dK(j) and dQ(j) run.
        if (lane == 0) {
            const uint32_t tS = tmem + C::kColS;
            const uint32_t tDP = tmem + C::kColDP;
            const uint32_t tDV = tmem + C::kColDV;
            const uint32_t tDK = tmem + C::kColDK;
            const uint32_t tDQ = tmem + C::kColDQ;
            const uint32_t sK = sbase + C::kOffK;
            const uint32_t sV = sbase + C::kOffV;
            const uint32_t sDS = sbase + C::kOffDS;
            // K-major operand [128 rows x D]: a k-step is 16 elements (32 bytes)
            auto kmaj = [&](uint32_t tile, int kk) {
                const uint32_t off = (kk * 32) / 128 * C::kAtomBytes + (kk * 32) % 128;
                return smem_desc_sw128(tile + off, 16, 1024);
            };
            // MN-major operand stored [rows x 128-byte rows]: a k-step is 16
            // rows (2048 bytes); 64-element column blocks kAtomBytes apart
            auto mnmaj = [&](uint32_t tile, int kk) {
                return smem_desc_sw128(tile + kk * C::kUmmaK * 128, C::kAtomBytes, 1024);
            };
            auto stage_q = [&](int j) { return sbase + C::kOffQ + (j % C::kStages) * C::kTileBytes; };
            auto stage_do = [&](int j) { return sbase + C::kOffDO + (j % C::kStages) * C::kTileBytes; };
            // S^T(j) = K Q_j^T
            auto issue_s = [&](int j) {
#pragma unroll
                for (int kk = 0; kk < C::kDSteps; ++kk)
                    mma_ss<false>(tS, kmaj(sK, kk), kmaj(stage_q(j), kk), C::kIdescS, kk > 0 ? 1u : 0u);
                tc_commit(bar(C::kBarS));
            };

            bool ok = bwd_wait(bar(C::kBarKV), 0, abort_flag, p, 33);
            if (ok) ok = bwd_wait(bar(C::kBarFull + 0), 0, abort_flag, p, 34);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int it = 0; ok && it < T; ++it) {
                const uint32_t sQ = stage_q(it);
                const uint32_t sDO = stage_do(it);
                // dP^T = V dO^T (d = 128: into the columns the previous dQ occupied)
                ok = bwd_wait(bar(C::kBarFullDO + it % C::kStages), (it / C::kStages) & 1, abort_flag, p, 34);
                if (!ok) break;
                if (!C::kDqOwnCols && it > 0) {
                    ok = bwd_wait(bar(C::kBarDQFree), (it - 1) & 1, abort_flag, p, 35);
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::kDSteps; ++kk)
                    mma_ss<false>(tDP, kmaj(sV, kk), kmaj(sDO, kk), C::kIdescS, kk > 0 ? 1u : 0u);
                tc_commit(bar(C::kBarDP));
                // dV += P^T dO: query rows 16kk.. of P^T sit in warpgroup kk/4's columns
                ok = bwd_wait(bar(C::kBarP), it & 1, abort_flag, p, 36);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::kRowSteps; ++kk)
                    mma_ts<false>(tDV, tS + (kk / 4) * 64 + (kk % 4) * 8, mnmaj(sDO, kk), C::kIdescAcc,
                                  (it > 0 || kk > 0) ? 1u : 0u);
                // the next tile's scores (early order)
                if (C::kEarlyS && it + 1 < T) {
                    ok = bwd_wait(bar(C::kBarFull + (it + 1) % C::kStages), ((it + 1) / C::kStages) & 1,
                                  abort_flag, p, 34);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
                // dK += dS^T Q (dS^T read K-major from the dS tile), then this
                // tile's dQ = dS K (the same tile read MN-major)
                ok = bwd_wait(bar(C::kBarDS), it & 1, abort_flag, p, 37);
                if (!ok) break;
                tc_fence_after();
                auto issue_dk = [&]() {
#pragma unroll
                    for (int kk = 0; kk < C::kRowSteps; ++kk)
                        mma_ss<false>(tDK, kmaj(sDS, kk), mnmaj(sQ, kk), C::kIdescAcc, (it > 0 || kk > 0) ? 1u : 0u);
                };
                auto issue_dq = [&]() {
#pragma unroll
                    for (int kk = 0; kk < C::kRowSteps; ++kk)
                        mma_ss<false>(tDQ, smem_desc_sw128(sDS + kk * C::kUmmaK * 128, C::kAtomBytes, 1024),
                                      mnmaj(sK, kk), C::kIdescDQ, kk > 0 ? 1u : 0u);
                    tc_commit(bar(C::kBarDQ));
                };
                if (kRead) {
                    // dQ first: the read-out stages its dO-tile half while dK runs
                    issue_dq();
                    issue_dk();
                    tc_commit(bar(C::kBarDK));
                } else {
                    issue_dk();
                    if (C::kDqOwnCols && it > 0) {  // the previous dQ has been read out
                        ok = bwd_wait(bar(C::kBarDQFree), (it - 1) & 1, abort_flag, p, 35);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    issue_dq();
                }
                // the next tile's scores (late order: they run during dQ's read-out)
                if (!C::kEarlyS && it + 1 < T) {
                    ok = bwd_wait(bar(C::kBarFull + (it + 1) % C::kStages), ((it + 1) / C::kStages) & 1,
                                  abort_flag, p, 34);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
            }
            if (ok) tc_commit(bar(C::kBarAcc));
            // Drain every tensor-core operation before tensor memory is released.
            tc_commit(bar(C::kBarDrain));
            bwd_wait(bar(C::kBarDrain), 0, abort_flag, p, 38, false);
        }
      }
    } else {
        // ----------------------------------------------- gradient warpgroups
        // Order per tile j: dS(j) once dP^T(j) is ready, then P^T(j+1) (its
        // scores were issued right after dV(j)), then the read-out of dQ(j).
        regs_increase<C::kGradRegs>();
        const int w = warp / 4;         // query columns [64w, 64w + 64) of each tile
        const int wi = warp % 4;        // TMEM lane quarter this warp may access
        const int t = wi * 32 + lane;   // key row of the block (= TMEM lane); query row for dQ
        const uint32_t lane_off = static_cast<uint32_t>(wi * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS + 64u * static_cast<uint32_t>(w);
        const uint32_t tDP = tmem + lane_off + C::kColDP + 64u * static_cast<uint32_t>(w);
        [[maybe_unused]] const uint32_t tDQ = tmem + lane_off + C::kColDQ + static_cast<uint32_t>(w * (D / 2));
        const long long key = static_cast<long long>(kb) * 128 + t;
        const bool key_valid = key < p.Nkv;  // rows past Nkv were zero-filled: weight 0
        const float c = p.scale_log2;
        bool ok = true;
        uint32_t x[2][32];  // P^T of the current tile in fp32: this key, 64 query columns

        // P^T(j) = 2^(S^T scale log2(e) - lse_i log2(e)) into x and, as 16-bit
        // pairs, over this warpgroup's first 32 S^T columns
        auto p_phase = [&](int j) -> bool {
            const int sj = j % C::kStages;
            const int qt = qt_begin + j % nqt;
            // the stage's statistics have landed, and S^T(j) is ready
            bool got = bwd_wait(bar(C::kBarFull + sj), (j / C::kStages) & 1, abort_flag, p, 40);
            if (got) got = bwd_wait(bar(C::kBarS), j & 1, abort_flag, p, 41);
            if (!__all_sync(0xffffffffu, got)) return false;
            tc_fence_after();
            tmem_ld32(tS, x[0]);
            tmem_ld32(tS + 32u, x[1]);
            tmem_ld_wait(x[0]);
            tmem_ld_wait(x[1]);
            // -lse log2(e) of this warpgroup's 64 query columns
            const float4* nl4 = reinterpret_cast<const float4*>(smem + C::kOffStats + sj * kBwdStatBytes) + 16 * w;
            // causal: query column q (index qt*128 + q) sees this key iff q >= thr
            int thr = 0;
            if (kCausal) {
                const long long v = key - p.causal_offset - static_cast<long long>(qt) * 128;
                thr = static_cast<int>(v < -1 ? -1 : (v > 129 ? 129 : v));
            }
            const uint64_t c2 = f2_pack(c, c);
            uint32_t pk[32];  // pair m: query columns 64w + 2m, 64w + 2m + 1
#pragma unroll
            for (int m4 = 0; m4 < 16; ++m4) {
                const float4 nl = nl4[m4];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int m = 2 * m4 + hh, h = m / 16, e = (m % 16) * 2;
                    float t0, t1;
                    f2_unpack(f2_fma(f2_pack(bwd_u2f(x[h][e]), bwd_u2f(x[h][e + 1])), c2,
                                     hh == 0 ? f2_pack(nl.x, nl.y) : f2_pack(nl.z, nl.w)),
                              t0, t1);
                    float p0 = ex2(t0), p1 = ex2(t1);
                    if (kCausal) {
                        const int q0 = 64 * w + 2 * m;
                        if (q0 < thr) p0 = 0.0f;
                        if (q0 + 1 < thr) p1 = 0.0f;
                    }
                    if (!key_valid) {
                        p0 = 0.0f;
                        p1 = 0.0f;
                    }
                    x[h][e] = __float_as_uint(p0);
                    x[h][e + 1] = __float_as_uint(p1);
                    pk[m] = pack_16x2<F16>(p0, p1);
                }
            }
            tmem_st32(tS, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarP));
            return true;
        };

        if (T > 0) ok = p_phase(0);
        for (int it = 0; ok && it < T; ++it) {
            const int s = it % C::kStages;

            // dS^T = P^T o (dP^T - D), as 16-bit pairs into row t of atom w of
            // the dS tile (free: the previous dK and dQ have completed)
            bool got = bwd_wait(bar(C::kBarDP), it & 1, abort_flag, p, 42);
            ok = __all_sync(0xffffffffu, got);
            if (!ok) break;
            tc_fence_after();
            const float4* d4 =
                reinterpret_cast<const float4*>(smem + C::kOffStats + s * kBwdStatBytes + kBwdStatBytes / 2) + 16 * w;
            const float* dcol = reinterpret_cast<const float*>(d4);
            uint32_t dpk[32];  // pair m: query columns 64w + 2m, 64w + 2m + 1
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t dp[32];
                tmem_ld32(tDP + 32u * h, dp);
                tmem_ld_wait(dp);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int m = h * 16 + e / 2;
                    const float d0 = bwd_u2f(x[h][e]) * (bwd_u2f(dp[e]) - dcol[2 * m]);
                    const float d1 = bwd_u2f(x[h][e + 1]) * (bwd_u2f(dp[e + 1]) - dcol[2 * m + 1]);
                    dpk[m] = pack_16x2<F16>(d0, d1);
                }
            }
            uint8_t* row_ptr = smem + C::kOffDS + w * C::kAtomBytes + t * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(row_ptr + ((ch ^ (t & 7)) << 4)) =
                    make_uint4(dpk[4 * ch], dpk[4 * ch + 1], dpk[4 * ch + 2], dpk[4 * ch + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarDS));

            // the next tile's P^T while dK and dQ of this tile run (early order)
            if (C::kEarlyS && it + 1 < T) {
                ok = p_phase(it + 1);
                if (!ok) break;
            }

            if constexpr (!kRead) {
                // (384-thread layout) this tile's dQ (query row t, columns
                // [w d/2, (w+1) d/2)): staged as fp32 boxes of 32 columns
                // (128-byte swizzle) in the stage's Q tile (w = 0) or dO tile
                // (w = 1), which the reducer adds into the accumulator
                got = bwd_wait(bar(C::kBarDQ), it & 1, abort_flag, p, 43);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) break;
                tc_fence_after();
                uint8_t* stg = smem + (w == 0 ? C::kOffQ : C::kOffDO) + s * C::kTileBytes;
                uint32_t v[D / 64][32];
#pragma unroll
                for (int h = 0; h < D / 64; ++h) tmem_ld32(tDQ + 32u * h, v[h]);
#pragma unroll
                for (int h = 0; h < D / 64; ++h) tmem_ld_wait(v[h]);
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    uint8_t* rowp = stg + h * C::kAtomBytes + t * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4*>(rowp + ((ch ^ (t & 7)) << 4)) =
                            make_uint4(v[h][4 * ch], v[h][4 * ch + 1], v[h][4 * ch + 2], v[h][4 * ch + 3]);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(C::kBarDQFree));    // its tensor-memory columns are free
                    mbar_arrive(bar(C::kBarStaged + s));  // the reducer may read the staged rows
                }
            }
            // the next tile's P^T (late order)
            if (!C::kEarlyS && it + 1 < T) {
                ok = p_phase(it + 1);
                if (!ok) break;
            }
        }

        // ------------------------------------------------------- epilogue
        // warpgroup 0: dV (staged in the V tile); warpgroup 1: scale * dK (in the K tile)
        if (ok && has_work) {
            const bool got = bwd_wait(bar(C::kBarAcc), 0, abort_flag, p, 44);
            ok = __all_sync(0xffffffffu, got);
        }
        uint8_t* stage = smem + (w == 0 ? C::kOffV : C::kOffK);
        if (ok) {
            tc_fence_after();
            const uint32_t tAcc = tmem + lane_off + 256u + (w == 0 ? 0u : static_cast<uint32_t>(D));
            const float mul = (w == 0) ? 1.0f : p.scale;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                if (has_work) {
                    tmem_ld32(tAcc + 32u * q, o);
                    tmem_ld_wait(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                // 32 values = half a swizzle row: chunks 4*(q%2) .. +3 of atom q/2
                uint8_t* rowp = stage + (q / 2) * C::kAtomBytes + t * 128;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int ch = (q % 2) * 4 + cc;
                    uint4 v4;
                    v4.x = pack_16x2<F16>(bwd_u2f(o[8 * cc + 0]) * mul, bwd_u2f(o[8 * cc + 1]) * mul);
                    v4.y = pack_16x2<F16>(bwd_u2f(o[8 * cc + 2]) * mul, bwd_u2f(o[8 * cc + 3]) * mul);
                    v4.z = pack_16x2<F16>(bwd_u2f(o[8 * cc + 4]) * mul, bwd_u2f(o[8 * cc + 5]) * mul);
                    v4.w = pack_16x2<F16>(bwd_u2f(o[8 * cc + 6]) * mul, bwd_u2f(o[8 * cc + 7]) * mul);
                    *reinterpret_cast<uint4*>(rowp + ((ch ^ (t & 7)) << 4)) = v4;
                }
            }
            fence_proxy_async_smem();
        }
        // Every thread of the warpgroup arrives exactly once, whatever happened.
        mbar_arrive(bar(C::kBarEpi + w));
        if (t == 0) {
            const bool all_in = bwd_wait(bar(C::kBarEpi + w), 0, abort_flag, p, 45);
            if (all_in && !*abort_flag) {
                const CUtensorMap* map = (w == 0) ? &map_dv : &map_dk;
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_store_3d(map, smem_u32(stage + a * C::kAtomBytes), a * C::kAtomElems, kb * 128, unit);
                tma_store_commit();
                tma_store_wait_read();
            }
        }
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kBwdTmemCols);
    }
}

template <int D, bool F16, bool kCausal>
cudaError_t launch_bwd_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                               const CUtensorMap& dq, const BwdParams& p, unsigned int grid,
                               cudaStream_t stream) {
    using C = BwdCfg<D, F16, bwd_read_layout<D, kCausal>()>;
    auto kern = fa_bwd_kernel<D, F16, kCausal>;
    // The register split relies on the compiled kernel holding exactly
    // C::kLaunchRegs per thread (a setmaxnreg.inc without the registers behind
    // it would never return); refuse to launch otherwise.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != static_cast<int>(C::kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(q, k, v, dout, dk, dv, dq, p);
    return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                       const CUtensorMap& dq, const BwdParams& p, unsigned int grid, cudaStream_t stream) {
    return p.causal ? launch_bwd_variant<D, F16, true>(q, k, v, dout, dk, dv, dq, p, grid, stream)
                    : launch_bwd_variant<D, F16, false>(q, k, v, dout, dk, dv, dq, p, grid, stream);
}

}  // namespace fa
