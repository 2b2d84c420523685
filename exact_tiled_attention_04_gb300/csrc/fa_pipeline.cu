// fa_fwd_host: the forward pass on tensors in host memory, with the copies
// to and from the GPU overlapped with the computation (declared in
// include/fa.h).
//
// The work is cut into chunks of consecutive key/value heads (with their
// query heads), at most eight and each large enough to keep about 256 CTAs
// (one chunk for small problems).  In the flattened [B*H_kv] head order, a
// chunk's q, o and lse rows and its k, v rows are each one contiguous range,
// so each chunk is an ordinary fa_fwd_ex call on device copies of those
// ranges.  Three streams:
// copies in, the caller's stream for the kernels, copies out; chunk slots in
// the caller's workspace form a ring so chunk c+1 arrives while chunk c is
// computed and chunk c-1 leaves.  The caller's stream is made to wait for the
// last copy out, so completion on `stream` means the outputs are in host
// memory.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_host.h"

using namespace fa::host;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 3;             // chunks resident at once (in, compute, out)
constexpr int kMaxChunks = 8;         // chunks per call at most
constexpr int64_t kChunkCtas = 256;   // CTAs a chunk's launch should keep (1.7 waves of 152 SMs)

struct DeviceStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t loaded[kSlots] = {}, computed[kSlots] = {}, freed[kSlots] = {};
    bool ready = false;
};
DeviceStreams g_streams[kMaxDevices];
std::mutex g_streams_mutex[kMaxDevices];

int device_streams(DeviceStreams** out, int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_error("cudaGetDevice", static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    DeviceStreams& ds = g_streams[dev];
    if (!ds.ready) {
        e = cudaStreamCreateWithFlags(&ds.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ds.out, cudaStreamNonBlocking);
        for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&ds.loaded[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.computed[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.freed[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            set_error("stream/event creation", static_cast<int>(e), cudaGetErrorString(e));
            return FA_ERR_CUDA;
        }
        ds.ready = true;
    }
    *out = &ds;
    *dev_out = dev;
    return FA_OK;
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// The chunking of a problem: units (key/value heads, flattened over the
// batch) per chunk, and the bytes of one slot.
struct Plan {
    int64_t units = 0, per_chunk = 0, chunks = 0;
    size_t q_bytes = 0, kv_bytes = 0, lse_bytes = 0, split_bytes = 0;  // per chunk
    size_t slot_bytes = 0;
};

Plan make_plan(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, int dtype) {
    Plan pl;
    const int64_t group = H / H_kv;
    const size_t elem = (dtype & 0xFF) == FA_DTYPE_F32 ? 4 : 2;
    pl.units = B * H_kv;
    // as many chunks as keep each launch about kChunkCtas CTAs (a chunk that
    // underfills the GPU computes slower than the copies it would hide)
    const bool packed = group > 1 && N_q * group <= 128;
    const int64_t ctas_per_unit = packed ? 1 : group * ((N_q + 255) / 256);
    int64_t chunks = pl.units * ctas_per_unit / kChunkCtas;
    if (chunks > kMaxChunks) chunks = kMaxChunks;
    if (chunks > pl.units) chunks = pl.units;
    if (chunks < 1) chunks = 1;
    pl.per_chunk = (pl.units + chunks - 1) / chunks;
    pl.chunks = (pl.units + pl.per_chunk - 1) / pl.per_chunk;
    const size_t qh = static_cast<size_t>(pl.per_chunk * group);
    pl.q_bytes = qh * static_cast<size_t>(N_q) * static_cast<size_t>(d) * elem;
    pl.kv_bytes = static_cast<size_t>(pl.per_chunk) * static_cast<size_t>(N_kv) * static_cast<size_t>(d) * elem;
    pl.lse_bytes = qh * static_cast<size_t>(N_q) * sizeof(float);
    pl.split_bytes = fa_fwd_ex_workspace_size(1, static_cast<int64_t>(qh), N_q, N_kv, d, 1);
    pl.slot_bytes = 2 * align256(pl.q_bytes) + 2 * align256(pl.kv_bytes) + align256(pl.lse_bytes) +
                    align256(pl.split_bytes);
    return pl;
}

}  // namespace

extern "C" {

size_t fa_fwd_host_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d,
                                  int dtype) {
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || d < 1) return 0;
    if (B > INT64_MAX / H || B * H > INT64_MAX / N_q || B * H * N_q > INT64_MAX / (d * 4)) return 0;
    if (B * H_kv > INT64_MAX / N_kv || B * H_kv * N_kv > INT64_MAX / (d * 4)) return 0;
    const Plan pl = make_plan(B, H, H_kv, N_q, N_kv, d, dtype);
    return static_cast<size_t>(pl.chunks < kSlots ? pl.chunks : kSlots) * pl.slot_bytes;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
    // The argument checks of the device entry point, on the whole problem
    // (host pointers pass its alignment and overlap checks the same way).
    int st = fa_fwd_ex_validate(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, d, scale, dtype, 1, nullptr, 0);
    if (st != FA_OK) return st;
    if (workspace == nullptr) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
    const Plan pl = make_plan(B, H, H_kv, N_q, N_kv, d, dtype);
    const int slots = static_cast<int>(pl.chunks < kSlots ? pl.chunks : kSlots);
    if (workspace_bytes < static_cast<size_t>(slots) * pl.slot_bytes) return FA_ERR_INVALID_ARG;

    DeviceStreams* ds = nullptr;
    int dev = 0;
    if ((st = device_streams(&ds, &dev)) != FA_OK) return st;
    std::lock_guard<std::mutex> lock(g_streams_mutex[dev]);  // the internal streams are per device
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t group = H / H_kv;
    const size_t elem = (dtype & 0xFF) == FA_DTYPE_F32 ? 4 : 2;
    const size_t q_head = static_cast<size_t>(N_q) * static_cast<size_t>(d) * elem;
    const size_t kv_head = static_cast<size_t>(N_kv) * static_cast<size_t>(d) * elem;
    const size_t lse_head = static_cast<size_t>(N_q) * sizeof(float);
    auto fail = [&](const char* what, cudaError_t e) {
        set_error(what, static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    };

    // the inputs of the first chunk may only be written once earlier work on
    // the caller's stream that may read the workspace is done
    cudaError_t e = cudaEventRecord(ds->computed[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->in, ds->computed[0], 0);
    if (e != cudaSuccess) return fail("pipeline start", e);

    for (int64_t c = 0; c < pl.chunks; ++c) {
        const int slot = static_cast<int>(c % slots);
        const int64_t u0 = c * pl.per_chunk;
        const int64_t nu = (u0 + pl.per_chunk <= pl.units) ? pl.per_chunk : pl.units - u0;
        const int64_t hq0 = u0 * group, nq = nu * group;  // query heads of the chunk (flattened)
        uint8_t* base = static_cast<uint8_t*>(workspace) + static_cast<size_t>(slot) * pl.slot_bytes;
        uint8_t* dq = base;
        uint8_t* dout = dq + align256(pl.q_bytes);
        uint8_t* dk = dout + align256(pl.q_bytes);
        uint8_t* dv = dk + align256(pl.kv_bytes);
        float* dl = reinterpret_cast<float*>(dv + align256(pl.kv_bytes));
        uint8_t* dsplit = reinterpret_cast<uint8_t*>(dl) + align256(pl.lse_bytes);

        // copies in, once the slot's previous chunk has left
        if (c >= slots && (e = cudaStreamWaitEvent(ds->in, ds->freed[slot], 0)) != cudaSuccess)
            return fail("pipeline wait (slot)", e);
        const size_t qb = static_cast<size_t>(nq) * q_head, kvb = static_cast<size_t>(nu) * kv_head;
        if ((e = cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + static_cast<size_t>(hq0) * q_head, qb,
                                 cudaMemcpyHostToDevice, ds->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + static_cast<size_t>(u0) * kv_head, kvb,
                                 cudaMemcpyHostToDevice, ds->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + static_cast<size_t>(u0) * kv_head, kvb,
                                 cudaMemcpyHostToDevice, ds->in)) != cudaSuccess ||
            (e = cudaEventRecord(ds->loaded[slot], ds->in)) != cudaSuccess)
            return fail("pipeline copy in", e);

        // the chunk's forward pass on the caller's stream
        if ((e = cudaStreamWaitEvent(s, ds->loaded[slot], 0)) != cudaSuccess) return fail("pipeline wait (in)", e);
        st = fa_fwd_ex(dq, dk, dv, dout, lse != nullptr ? dl : nullptr, 1, nq, nu, N_q, N_kv, d, scale, dtype, 1,
                       pl.split_bytes ? dsplit : nullptr, pl.split_bytes, s);
        if (st != FA_OK) return st;
        if ((e = cudaEventRecord(ds->computed[slot], s)) != cudaSuccess) return fail("pipeline record", e);

        // copies out
        if ((e = cudaStreamWaitEvent(ds->out, ds->computed[slot], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(static_cast<uint8_t*>(o) + static_cast<size_t>(hq0) * q_head, dout, qb,
                                 cudaMemcpyDeviceToHost, ds->out)) != cudaSuccess)
            return fail("pipeline copy out", e);
        if (lse != nullptr &&
            (e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse) + static_cast<size_t>(hq0) * lse_head, dl,
                                 static_cast<size_t>(nq) * lse_head, cudaMemcpyDeviceToHost, ds->out)) !=
                cudaSuccess)
            return fail("pipeline copy out (lse)", e);
        if ((e = cudaEventRecord(ds->freed[slot], ds->out)) != cudaSuccess) return fail("pipeline record", e);
    }
    // completion on the caller's stream: every copy out has finished
    const int last = static_cast<int>((pl.chunks - 1) % slots);
    if ((e = cudaStreamWaitEvent(s, ds->freed[last], 0)) != cudaSuccess) return fail("pipeline end", e);
    return FA_OK;
}

}  // extern "C"
