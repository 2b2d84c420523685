// C-ABI entry points of the attention library (declared in include/fa.h):
// host-side argument checks, TMA tensor-map encoding, kernel dispatch and
// the device error word.
//
// The boundary follows the fused kernel of "CUDA Flash Attention: Online
// Softmax with Shared Memory Tiling" (Kernel 2: Q, K, V, O, N, d and scale
// as arguments; Design decisions: size_t indexing, restrict-qualified
// non-aliasing outputs; Correctness Audit: launch errors surfaced, the head
// dimension checked instead of assumed), extended with batch, heads, dtype,
// the log-sum-exp output and a stream.
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_host.h"
#include "fa_internal.h"

// Set by the kernels when a bounded wait gives up (one per device).
__device__ fa::DevStatus g_fa_device_status;

namespace fa {
// An empty kernel with the forward kernel's launch shape, used only to ask
// the occupancy calculator about clusters (see device_shape); never launched.
__global__ void fa_cluster_shape_probe() {}
}  // namespace fa

namespace {
thread_local char g_last_error[512] = "";
}  // namespace

namespace fa {
namespace host {

void set_error(const char* what, int code, const char* text) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: error %d (%s)", what, code,
                  text ? text : "");
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

constexpr int kMaxDevices = 64;
std::mutex g_err_mutex;
std::atomic<unsigned int> g_generation{0};

// Identity of the current CUDA context, unique over the process's life (the
// driver's context id), or 0 when no context is current or the driver
// entry points cannot be reached.  A device reset destroys the context and
// the module's device symbols with it; the next context gets a new id.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

// Device address of a __device__ variable of this library on the current
// device, looked up once per device and context (cudaGetSymbolAddress, with
// that device current) and looked up again after a device reset.  *status
// gets FA_OK or FA_ERR_CUDA.
void* SymbolCache::address(const void* symbol, const char* what, int* status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxCachedDevices) {
        set_error("cudaGetDevice", static_cast<int>(e), cudaGetErrorString(e));
        *status = FA_ERR_CUDA;
        return nullptr;
    }
    unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (ptr[dev] == nullptr || ctx == 0 || ctx != ctx_id[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, symbol);
        if (e != cudaSuccess || p == nullptr) {
            set_error(what, static_cast<int>(e), cudaGetErrorString(e));
            *status = FA_ERR_CUDA;
            return nullptr;
        }
        ptr[dev] = p;
        ctx_id[dev] = current_context_id();  // the lookup made the context current if it was not
    }
    *status = FA_OK;
    return ptr[dev];
}

// Launch generation: never 0 (0 is the status word's initial abort_gen).
unsigned int next_generation() {
    unsigned int g = ++g_generation;
    if (g == 0) g = ++g_generation;
    return g;
}

// Device address of the status words on the current device.
fa::DevStatus* device_status_words(int* status) {
    static SymbolCache cache;
    return static_cast<fa::DevStatus*>(
        cache.address(&g_fa_device_status, "cudaGetSymbolAddress(status words)", status));
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Boxes are 128 x 1 rows x heads normally and Nq x group for packed grouped
// heads in the forward pass.
int encode_map(CUtensorMap* map, const void* base, int dtype, int64_t BH, int64_t N, int64_t d,
               uint32_t box_rows, uint32_t box_heads) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) {
        set_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)",
                  static_cast<int>(g_encode_err), cudaGetErrorString(g_encode_err));
        return FA_ERR_CUDA;
    }
    const cuuint64_t elem = dtype == FA_DTYPE_F32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem,
                                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * elem};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), box_rows, box_heads};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType type = dtype == FA_DTYPE_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : dtype == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = enc(map, type,
                     3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled", static_cast<int>(r), "tensor map rejected");
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace host
}  // namespace fa

using namespace fa::host;

namespace {
constexpr int64_t kInt32Max = 2147483647;

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported head dimension, dtype or size";
        case FA_ERR_ALIGNMENT: return "tensor base address not 16-byte aligned";
        case FA_ERR_CUDA: return "CUDA call failed";
        case FA_ERR_TIMEOUT: return "kernel timed out waiting on an internal barrier";
        default: return "unknown status";
    }
}

const char* fa_last_error_message(void) { return g_last_error; }

}  // extern "C"

namespace {

// Effective key partitions for a requested count: at most one per key tile,
// at most kMaxSplits, and no empty partition.
struct SplitPlan {
    int splits;
    int tiles_per_split;
    int n_kv_tiles;
};

// Grouped query heads whose Nq rows all fit one 128-row tile are packed: one
// CTA per key/value head serves its `group` query heads (a decode step reads
// each key/value tile once instead of once per query head).
bool packed_heads(int64_t H, int64_t H_kv, int64_t N_q) {
    const int64_t group = H / H_kv;
    return group > 1 && N_q * group <= 128;
}

// Decode steps: at most 32 query rows per key/value head (N_q x group) go to
// the decode kernel (16-bit inputs), one CTA per key/value head and key
// partition, keys on the tensor-memory lanes.
constexpr int64_t kDecodeMaxRows = 32;
bool decode_rows(int64_t H, int64_t H_kv, int64_t N_q) { return N_q * (H / H_kv) <= kDecodeMaxRows; }

// CTAs of one key partition: query blocks of 256 rows per head (per key/value
// head when packed or in the decode kernel; with group 1 and N_q <= 32 the
// two counts agree, so the count does not depend on the dtype).
int64_t ctas_per_partition(int64_t B, int64_t H, int64_t H_kv, int64_t N_q) {
    if (packed_heads(H, H_kv, N_q) || decode_rows(H, H_kv, N_q)) return B * H_kv;
    return B * H * ((N_q + 255) / 256);
}
constexpr int kMaxSplits = 32;  // the merge kernel holds one partition per lane

SplitPlan plan_splits(int64_t N_kv, int num_splits) {
    SplitPlan sp;
    sp.n_kv_tiles = static_cast<int>((N_kv + 127) / 128);
    int s = num_splits < 1 ? 1 : num_splits;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s > sp.n_kv_tiles) s = sp.n_kv_tiles;
    sp.tiles_per_split = (sp.n_kv_tiles + s - 1) / s;
    sp.splits = (sp.n_kv_tiles + sp.tiles_per_split - 1) / sp.tiles_per_split;
    return sp;
}

size_t workspace_bytes_for(int64_t B, int64_t H, int64_t N_q, int64_t d, const SplitPlan& sp) {
    if (sp.splits <= 1) return 0;
    const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(N_q);
    return static_cast<size_t>(sp.splits) * rows * (static_cast<size_t>(d) + 4) * sizeof(float);
}

// What the automatic plan needs to know about the current device: its SM
// count, and how many thread-block clusters of s CTAs (one CTA per SM, as
// every forward variant runs) can be resident at once.  The second depends
// on how the SMs are grouped on the chip (on a 152-SM GB300: 76 clusters of
// 2, 36 of 4, 15 of 8), so it is asked of the runtime.
constexpr int kMaxClusterSplits = 8;  // portable cluster size

struct DeviceShape {
    int sms = 0;                                  // 0: no device answered
    int max_clusters[kMaxClusterSplits + 1] = {};  // [s], s = 2 .. 8
};

DeviceShape query_device_shape(int dev) {
    DeviceShape ds;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return ds;
    ds.sms = n;
    const int smem = 160 * 1024;  // above half an SM's shared memory: one CTA per SM
    if (cudaFuncSetAttribute(fa::fa_cluster_shape_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return ds;
    }
    for (int cs = 2; cs <= kMaxClusterSplits; ++cs) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(cs));
        cfg.blockDim = dim3(384);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, fa::fa_cluster_shape_probe, &cfg) != cudaSuccess || c < 0) {
            cudaGetLastError();
            c = 0;  // unknown: no clusters of this size
        }
        ds.max_clusters[cs] = c;
    }
    return ds;
}

// The current device's shape (cached per device; sms = 0 when no device
// answers, which makes the automatic plan use one partition).
DeviceShape device_shape() {
    static DeviceShape cache[kMaxDevices];
    static bool known[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DeviceShape{};
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!known[dev]) {
        cache[dev] = query_device_shape(dev);
        known[dev] = cache[dev].sms > 0;
    }
    return cache[dev];
}

int device_sm_count() { return device_shape().sms; }

// The launches of one fa_fwd_ex call.  num_splits >= 1: one launch with that
// many key partitions (capped by plan_splits), their partial results in the
// caller's workspace, merged by a second kernel when more than one.
// num_splits == 0 (automatic), on a GPU of `sms` SMs, one CTA per SM:
//   * fewer query blocks than SMs: as many partitions as fill one wave
//     (the fa_fwd_ex_splits count).  When they fit one thread-block cluster
//     (at most 8, and every block's cluster resident at once) the
//     partitions of a query block form a cluster and merge through
//     distributed shared memory inside the same launch (no workspace, no
//     merge kernel); the cluster is then made as large as the device can
//     hold for this many blocks.  Otherwise (more partitions wanted,
//     workspace allowed) they go through the workspace and the merge kernel.
//   * several waves whose last one is at most half full (16-bit inputs,
//     unmasked, one query head per query block, at least kTailMinTiles key
//     tiles per block): the full waves' blocks run unsplit, and the blocks of
//     the last wave (the last in block order) run in a second launch, split
//     along the keys into clusters of at most 4 partitions merged in-cluster;
//   * otherwise one partition.
// allow_workspace = false (fa_fwd): only in-cluster merges.  Any workspace a
// plan uses stays below sms x 256 partial rows, which bounds
// fa_fwd_ex_workspace_size with num_splits == 0.
#ifndef FA_TAIL_MIN_TILES
#define FA_TAIL_MIN_TILES 16
#endif
// the tail launch pays off when a block sweeps at least this many key tiles
// (measured with the merge kernel: +10 % at 128 tiles, +1.2 % at 64, -1 % at
// 16; with the in-cluster merge +1 % at 16, b4h16_n2048 98.5 -> 97.4 us)
constexpr int kTailMinTiles = FA_TAIL_MIN_TILES;

struct LaunchPlan {
    SplitPlan sp;              // partitions of the (first) launch
    bool cluster = false;      // the first launch merges its partitions in-cluster
    int64_t tail_first = -1;   // >= 0: first query block of the tail launch (in-cluster merge)
    SplitPlan tail{};          // partitions of the tail launch
    size_t workspace = 0;      // bytes the plan writes
};

// Partitions of `items` query blocks that merge in-cluster: the largest count
// <= limit (and <= what the kernel's shared memory can merge for this dtype
// and head dimension) whose clusters can all be resident at once; splits = 1
// when none can.
SplitPlan cluster_plan(int64_t N_kv, int64_t items, int limit, const DeviceShape& dev, int dtype, int64_t d) {
    const int cap = fa::fwd_max_merge_parts(dtype & 0xFF, static_cast<int>(d));
    if (limit > cap) limit = cap;
    for (int s = limit < kMaxClusterSplits ? limit : kMaxClusterSplits; s >= 2; --s) {
        const SplitPlan sp = plan_splits(N_kv, s);
        if (sp.splits >= 2 && items <= dev.max_clusters[sp.splits]) return sp;
    }
    return plan_splits(N_kv, 1);
}

LaunchPlan make_launch_plan(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                            int dtype_arg, int num_splits, const DeviceShape& dev, bool allow_workspace) {
    LaunchPlan pl;
    if (num_splits >= 1) {
        pl.sp = plan_splits(N_kv, num_splits);
        pl.workspace = workspace_bytes_for(B, H, N_q, d, pl.sp);
        return pl;
    }
    pl.sp = plan_splits(N_kv, 1);
    const int sms = dev.sms;
    if (sms <= 0) return pl;
    const int dtype = dtype_arg & 0xFF;
    // the general kernel on unpacked query blocks merges in-cluster
    const bool cluster_ok = !packed_heads(H, H_kv, N_q) && !(dtype != FA_DTYPE_F32 && decode_rows(H, H_kv, N_q));
    const int64_t blocks = ctas_per_partition(B, H, H_kv, N_q);
    if (blocks < sms) {
        const int64_t want = sms / blocks;
        const SplitPlan full = plan_splits(N_kv, static_cast<int>(want > kMaxSplits ? kMaxSplits : want));
        if (full.splits < 2) return pl;
        if (cluster_ok && (full.splits <= fa::fwd_max_merge_parts(dtype, static_cast<int>(d)) || !allow_workspace)) {
            const SplitPlan cp = cluster_plan(N_kv, blocks, full.splits, dev, dtype, d);
            if (cp.splits >= 2) {
                pl.sp = cp;
                pl.cluster = true;
                return pl;
            }
        }
        if (allow_workspace) {
            pl.sp = full;
            pl.workspace = workspace_bytes_for(B, H, N_q, d, pl.sp);
        }
        return pl;
    }
    const bool eligible = cluster_ok && dtype != FA_DTYPE_F32 && !(dtype_arg & FA_FLAG_CAUSAL) &&
                          !packed_heads(H, H_kv, N_q);
    const int64_t frac = blocks % sms;  // blocks of the last wave
    if (!eligible || frac == 0 || 2 * frac > sms || pl.sp.n_kv_tiles < kTailMinTiles) return pl;
    const int64_t ts = sms / frac < 4 ? sms / frac : 4;
    const SplitPlan tail = cluster_plan(N_kv, frac, static_cast<int>(ts), dev, dtype, d);
    if (tail.splits < 2) return pl;
    pl.tail = tail;
    pl.tail_first = blocks - frac;
    return pl;
}

// Workspace bound of the automatic plan on the current device.
size_t auto_workspace_bound(int64_t B, int64_t H, int64_t N_q, int64_t d) {
    int sms = device_sm_count();
    if (sms <= 0) sms = 1024;  // no device to ask: a bound for any
    const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(N_q);
    size_t r = static_cast<size_t>(sms) * 256;
    if (r > rows * kMaxSplits) r = rows * kMaxSplits;
    return r * (static_cast<size_t>(d) + 4) * sizeof(float);
}

// Every host check of fa_fwd_ex except those on the workspace: pointers,
// sizes, dtype, alignment and overlaps of the tensors.
int validate_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                  float scale, int dtype_arg, int num_splits) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (num_splits < 0) return FA_ERR_INVALID_ARG;  // 0: automatic
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype_arg & ~(0xFF | FA_FLAG_CAUSAL)) return FA_ERR_INVALID_ARG;  // unknown flag
    const int dtype = dtype_arg & 0xFF;
    if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return FA_ERR_UNSUPPORTED;
    if (dtype != FA_DTYPE_F32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (dtype == FA_DTYPE_F32 && d != 64) return FA_ERR_UNSUPPORTED;
    // element counts and byte sizes must fit in int64 (d is 64 or 128 here)
    if (B > INT64_MAX / H) return FA_ERR_INVALID_ARG;
    const int64_t BH = B * H, BHkv = B * H_kv;
    if (BH > INT64_MAX / N_q || BH * N_q > INT64_MAX / (d * 4)) return FA_ERR_INVALID_ARG;
    if (BHkv > INT64_MAX / N_kv || BHkv * N_kv > INT64_MAX / (d * 4)) return FA_ERR_INVALID_ARG;
    // TMA coordinates are 32-bit; global strides below 2^40 bytes
    if (BH > kInt32Max || N_q > kInt32Max || N_kv > kInt32Max) return FA_ERR_UNSUPPORTED;
    const int64_t elem = dtype == FA_DTYPE_F32 ? 4 : 2;
    if (N_q * d * elem >= (int64_t(1) << 40) || N_kv * d * elem >= (int64_t(1) << 40))
        return FA_ERR_UNSUPPORTED;
    const SplitPlan sp = plan_splits(N_kv, num_splits);
    if (ctas_per_partition(B, H, H_kv, N_q) > kInt32Max / sp.splits) return FA_ERR_UNSUPPORTED;  // grid size
    const uintptr_t mask = 15;
    if ((reinterpret_cast<uintptr_t>(q) & mask) || (reinterpret_cast<uintptr_t>(k) & mask) ||
        (reinterpret_cast<uintptr_t>(v) & mask) || (reinterpret_cast<uintptr_t>(o) & mask))
        return FA_ERR_ALIGNMENT;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3)) return FA_ERR_ALIGNMENT;
    const size_t qbytes = static_cast<size_t>(BH * N_q * d * elem);
    const size_t kvbytes = static_cast<size_t>(BHkv * N_kv * d * elem);
    if (overlaps(o, qbytes, q, qbytes) || overlaps(o, qbytes, k, kvbytes) || overlaps(o, qbytes, v, kvbytes))
        return FA_ERR_INVALID_ARG;
    if (lse != nullptr) {
        const size_t lbytes = static_cast<size_t>(BH * N_q) * sizeof(float);
        if (overlaps(lse, lbytes, o, qbytes) || overlaps(lse, lbytes, q, qbytes) ||
            overlaps(lse, lbytes, k, kvbytes) || overlaps(lse, lbytes, v, kvbytes))
            return FA_ERR_INVALID_ARG;
    }
    return FA_OK;
}

// Workspace bytes the plan of these (valid) arguments writes on the current device.
size_t plan_workspace(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                      int dtype_arg, int num_splits) {
    return make_launch_plan(B, H, H_kv, N_q, N_kv, d, dtype_arg, num_splits, device_shape(), true).workspace;
}

// The workspace checks of fa_fwd_ex for a plan that writes `need` bytes.
int validate_workspace(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                       int dtype_arg, size_t need, const void* workspace, size_t workspace_bytes) {
    if (need == 0) return FA_OK;
    if (workspace == nullptr || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return FA_ERR_ALIGNMENT;
    const int64_t elem = (dtype_arg & 0xFF) == FA_DTYPE_F32 ? 4 : 2;
    const size_t qbytes = static_cast<size_t>(B * H * N_q * d * elem);
    const size_t kvbytes = static_cast<size_t>(B * H_kv * N_kv * d * elem);
    if (overlaps(workspace, need, o, qbytes) || overlaps(workspace, need, q, qbytes) ||
        overlaps(workspace, need, k, kvbytes) || overlaps(workspace, need, v, kvbytes) ||
        (lse != nullptr && overlaps(workspace, need, lse, static_cast<size_t>(B * H * N_q) * sizeof(float))))
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

int validate_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                float scale, int dtype_arg, int num_splits, const void* workspace,
                size_t workspace_bytes) {
    const int st = validate_args(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype_arg, num_splits);
    if (st != FA_OK) return st;
    const size_t need = plan_workspace(B, H, H_kv, N_q, N_kv, d, dtype_arg, num_splits);
    return validate_workspace(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, dtype_arg, need, workspace,
                              workspace_bytes);
}

// allow_workspace: the plan may put split partials in `workspace` (fa_fwd_ex);
// false for fa_fwd, which has none (its splits merge in-cluster).
int launch_ex(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
              int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale,
              int dtype_arg, int num_splits, void* workspace, void* stream, bool allow_workspace = true) {
    const int dtype = dtype_arg & 0xFF;
    const bool causal = (dtype_arg & FA_FLAG_CAUSAL) != 0;
    const int64_t BH = B * H;
    const LaunchPlan plan =
        make_launch_plan(B, H, H_kv, N_q, N_kv, d, dtype_arg, num_splits, device_shape(), allow_workspace);
    const SplitPlan sp = plan.sp;
    const bool pack = packed_heads(H, H_kv, N_q);
    const bool dec = dtype != FA_DTYPE_F32 && decode_rows(H, H_kv, N_q);
    const uint32_t qbox_rows = (pack || dec) ? static_cast<uint32_t>(N_q) : 128u;
    const uint32_t qbox_heads = (pack || dec) ? static_cast<uint32_t>(H / H_kv) : 1u;
    CUtensorMap mq, mk, mv, mo;
    int st;
    if ((st = encode_map(&mq, q, dtype, BH, N_q, d, qbox_rows, qbox_heads)) != FA_OK) return st;
    if ((st = encode_map(&mk, k, dtype, B * H_kv, N_kv, d)) != FA_OK) return st;
    if ((st = encode_map(&mv, v, dtype, B * H_kv, N_kv, d)) != FA_OK) return st;
    if ((st = encode_map(&mo, o, dtype, BH, N_q, d, qbox_rows, qbox_heads)) != FA_OK) return st;

    fa::FwdParams p{};
    p.status = device_status_words(&st);
    if (st != FA_OK) return st;
    p.gen = next_generation();
    p.Nq = static_cast<int>(N_q);
    p.Nkv = static_cast<int>(N_kv);
    p.n_kv_tiles = sp.n_kv_tiles;
    p.pack = pack ? 1 : 0;
    p.n_q_blocks = pack ? 1 : static_cast<int>((N_q + 255) / 256);
    p.H = static_cast<int>(H);
    p.H_kv = static_cast<int>(H_kv);
    p.group = static_cast<int>(H / H_kv);
    p.causal = causal ? 1 : 0;
    p.causal_offset = static_cast<int>(N_kv - N_q);
    p.splits = sp.splits;
    p.tiles_per_split = sp.tiles_per_split;
    p.scale_log2 = scale * 1.4426950408889634f;
    const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(N_q);
    p.part_row0 = 0;
    p.part_rows = static_cast<long long>(rows);
    p.cluster = plan.cluster ? 1 : 0;
    const bool via_workspace = sp.splits > 1 && !plan.cluster;
    if (via_workspace) {
        p.o_part = static_cast<float*>(workspace);
        p.ml_part = p.o_part + static_cast<size_t>(sp.splits) * rows * static_cast<size_t>(d);
        p.lse = nullptr;
    } else {
        p.lse = lse;
    }
    const int64_t blocks = ctas_per_partition(B, H, H_kv, N_q);
    // automatic plan with a tail launch: the first launch takes the full waves' blocks
    const int64_t first_blocks = plan.tail_first >= 0 ? plan.tail_first : blocks;
    const unsigned int grid = static_cast<unsigned int>(first_blocks * sp.splits);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    p.out = o;
    auto launch = [&](const fa::FwdParams& lp, unsigned int g) -> cudaError_t {
        if (dec && dtype == FA_DTYPE_BF16) return fa::launch_decode_bf16(static_cast<int>(d), mq, mk, mv, lp, g, s);
        if (dec) return fa::launch_decode_f16(static_cast<int>(d), mq, mk, mv, lp, g, s);
        if (dtype == FA_DTYPE_BF16 && d == 64) return fa::launch_fwd_bf16_d64(mq, mk, mv, mo, lp, g, s);
        if (dtype == FA_DTYPE_BF16) return fa::launch_fwd_bf16_d128(mq, mk, mv, mo, lp, g, s);
        if (dtype == FA_DTYPE_F16 && d == 64) return fa::launch_fwd_f16_d64(mq, mk, mv, mo, lp, g, s);
        if (dtype == FA_DTYPE_F16) return fa::launch_fwd_f16_d128(mq, mk, mv, mo, lp, g, s);
        return fa::launch_fwd_tf32_d64(mq, mk, mv, mo, lp, g, s);
    };
    cudaError_t e = launch(p, grid);
    if (e == cudaSuccess && via_workspace) {
        fa::MergeParams m{};
        m.o_part = p.o_part;
        m.ml_part = p.ml_part;
        m.o = o;
        m.lse = lse;
        m.rows = static_cast<long long>(rows);
        m.splits = sp.splits;
        e = fa::launch_merge(m, static_cast<int>(d), dtype, s);
    }
    if (e == cudaSuccess && plan.tail_first >= 0) {
        // the last wave's blocks, split along the keys into clusters that
        // merge their partitions in distributed shared memory
        fa::FwdParams t = p;
        t.gen = next_generation();
        t.item_offset = static_cast<int>(plan.tail_first);
        t.splits = plan.tail.splits;
        t.tiles_per_split = plan.tail.tiles_per_split;
        t.cluster = 1;
        t.o_part = nullptr;
        t.ml_part = nullptr;
        t.lse = lse;
        e = launch(t, static_cast<unsigned int>((blocks - plan.tail_first) * plan.tail.splits));
    }
    if (e != cudaSuccess) {
        set_error("fa_fwd launch", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_validate(const void* q, const void* k, const void* v, void* o, const float* lse,
                    int64_t B, int64_t H, int64_t N, int64_t d, float scale, int dtype) {
    return validate_args(q, k, v, o, lse, B, H, H, N, N, d, scale, dtype, 0);
}

// The automatic plan without a workspace: key partitions, where the device
// is underfilled, merge inside thread-block clusters.
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
           int64_t N, int64_t d, float scale, int dtype, void* stream) {
    const int st = validate_args(q, k, v, o, lse, B, H, H, N, N, d, scale, dtype, 0);
    if (st != FA_OK) return st;
    return launch_ex(q, k, v, o, lse, B, H, H, N, N, d, scale, dtype, 0, nullptr, stream, false);
}

int fa_fwd_launches(int64_t B, int64_t H, int64_t N, int64_t d, int dtype) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    const LaunchPlan pl = make_launch_plan(B, H, H, N, N, d, dtype, 0, device_shape(), false);
    return pl.tail_first >= 0 ? 2 : 1;
}

int fa_fwd_ex_validate(const void* q, const void* k, const void* v, void* o, const float* lse,
                       int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                       float scale, int dtype, int num_splits, const void* workspace,
                       size_t workspace_bytes) {
    return validate_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, num_splits,
                       workspace, workspace_bytes);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
              int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype,
              int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
    const int st = validate_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, num_splits,
                               workspace, workspace_bytes);
    if (st != FA_OK) return st;
    return launch_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, num_splits, workspace,
                     stream);
}

size_t fa_fwd_ex_workspace_size(int64_t B, int64_t H, int64_t N_q, int64_t N_kv, int64_t d,
                                int num_splits) {
    if (B < 1 || H < 1 || N_q < 1 || N_kv < 1 || d < 1 || num_splits < 0) return 0;
    if (num_splits == 0) return auto_workspace_bound(B, H, N_q, d);  // automatic: current device
    return workspace_bytes_for(B, H, N_q, d, plan_splits(N_kv, num_splits));
}

int fa_fwd_ex_launches(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, int dtype,
                       int num_splits) {
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || d < 1 || num_splits < 0) return 0;
    const LaunchPlan pl = make_launch_plan(B, H, H_kv, N_q, N_kv, d, dtype, num_splits,
                                           num_splits == 0 ? device_shape() : DeviceShape{}, true);
    const int first = (pl.sp.splits > 1 && !pl.cluster) ? 2 : 1;  // + the merge kernel
    return first + (pl.tail_first >= 0 ? 1 : 0);
}

int fa_fwd_ex_splits(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int num_sms) {
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || num_sms < 1) return 1;
    const int64_t ctas = ctas_per_partition(B, H, H_kv, N_q);
    if (ctas >= num_sms) return 1;
    const int64_t want = num_sms / ctas;  // fill about one wave
    return plan_splits(N_kv, static_cast<int>(want > kMaxSplits ? kMaxSplits : want)).splits;
}

int fa_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_error("cudaStreamSynchronize", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    fa::DevStatus st{};
    e = cudaMemcpyFromSymbol(&st, g_fa_device_status, sizeof(st));
    if (e != cudaSuccess) {
        set_error("cudaMemcpyFromSymbol", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    if (st.word == 0) return FA_OK;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_fa_device_status, &zero, sizeof(zero), offsetof(fa::DevStatus, word));
    if (e != cudaSuccess) {
        set_error("cudaMemcpyToSymbol", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    std::snprintf(g_last_error, sizeof(g_last_error), "device error word 0x%08x", st.word);
    return (st.word & fa::kDevErrTimeout) ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
}

int fa_selftest_barrier_timeout(void* stream) {
    int st = FA_OK;
    fa::FwdParams p{};
    p.status = device_status_words(&st);
    if (st != FA_OK) return st;
    p.gen = next_generation();
    cudaError_t e = fa::launch_selftest_wait(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_error("fa_selftest_barrier_timeout launch", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of fa_fwd_ex.
//
// Some callers cannot obtain device scratch memory for the split-KV partials:
// plugins inside inference engines that own the whole device memory pool,
// and per-step code that must not call cudaMalloc (it can synchronise the
// device and can fail at run time).  For them, the partials live in one
// fixed array of device memory that belongs to this library: every GPU that
// loads the library holds kStaticWorkspaceBytes until the process exits.
// All calls on a device share the array and it keeps the last call's
// contents; nothing in it needs to start at zero (every partial slot a call
// reads was written earlier by the same call).  Calls whose kernels overlap
// on the GPU (different streams, or host threads) race on the array and
// must be serialised by the caller.
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_fa_static_workspace[kStaticWorkspaceBytes];

// Device address of the static array on the current device, looked up with
// cudaGetSymbolAddress the first time a device (or a new context of it,
// after a device reset) uses it: host code cannot use the array's name as a
// device address.
void* static_workspace(int* status) {
    static SymbolCache cache;
    return cache.address(&g_fa_static_workspace, "cudaGetSymbolAddress(static workspace)", status);
}

}  // namespace

extern "C" {

size_t fa_fwd_ex_static_capacity(void) { return kStaticWorkspaceBytes; }

int fa_fwd_ex_static(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale,
                     int dtype, int num_splits, void* stream) {
    // The worst case of the request must fit the array, whatever the device.
    if (B >= 1 && H >= 1 && N_q >= 1 && N_kv >= 1 && d >= 1 && num_splits >= 0) {
        const size_t bound = fa_fwd_ex_workspace_size(B, H, N_q, N_kv, d, num_splits);
        if (bound > kStaticWorkspaceBytes) {
            std::snprintf(g_last_error, sizeof(g_last_error),
                          "fa_fwd_ex_static: the split partials need %zu bytes, more than the "
                          "%zu-byte static workspace; use fewer splits or fa_fwd_ex",
                          bound, kStaticWorkspaceBytes);
            return FA_ERR_UNSUPPORTED;
        }
    }
    // Every check that does not involve the workspace, before anything else.
    int st = validate_args(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, num_splits);
    if (st != FA_OK) return st;
    const size_t need = plan_workspace(B, H, H_kv, N_q, N_kv, d, dtype, num_splits);
    if (need > kStaticWorkspaceBytes) return FA_ERR_UNSUPPORTED;  // (the bound above covers it)
    void* ws = nullptr;
    if (need > 0) {
        ws = static_workspace(&st);
        if (st != FA_OK) return st;
        st = validate_workspace(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, dtype, need, ws,
                                kStaticWorkspaceBytes);
        if (st != FA_OK) return st;
    }
    return launch_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, num_splits, ws, stream);
}

}  // extern "C"
