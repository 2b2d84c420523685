// fa_fwd_host / fa_bwd_host: the forward and backward passes on tensors in
// host memory, with the copies to and from the GPU overlapped with the
// computation (declared in include/fa.h).
//
// The work is cut into chunks of consecutive key/value heads (with their
// query heads), at most sixteen and each large enough to keep about 128
// CTAs (one chunk for small problems), plus, for large problems, two
// smaller chunks at either end.  In the flattened [B*H_kv] head order, a
// chunk's q, o and lse rows and its k, v rows are each one contiguous range,
// so each chunk is an ordinary fa_fwd_ex call on device copies of those
// ranges (fa_bwd for the backward pass).  Four streams: copies in, two for
// the kernels (chunks alternate between them, so a chunk's CTAs start on
// the SMs the previous chunk's last CTAs leave idle), copies out; chunk
// slots in the caller's workspace form a ring so chunk c+1 arrives while
// chunk c is computed and chunk c-1 leaves.  All of them start after the
// work already queued on the caller's stream, and the caller's stream is
// made to wait for the last copy out, so completion on `stream` means the
// outputs are in host memory.
#include <cstddef>
#include <cstdint>
#include <functional>
#include <mutex>

#include "fa.h"
#include "fa_bwd_internal.h"
#include "fa_host.h"

using namespace fa::host;

namespace {

constexpr int kMaxDevices = 64;
// Chunks resident at once (being copied in, computed, copied out).  The
// backward pass's chunks take longer from their first copy in to their last
// copy out than their copies in alone, so a fourth slot keeps its copies in
// running (headline backward end to end 5.60 -> 5.19 ms); the forward pass
// measured no gain from it.
constexpr int kFwdSlots = 3;
constexpr int kBwdSlots = 4;
constexpr int kMaxSlots = 4;
// Chunks of about 128 CTAs, at most 16: the first upload and the last
// download are the only copies nothing overlaps, and smaller chunks shorten
// them (measured against 256 CTAs / 8 chunks: headline forward 2.450 ->
// 2.415 ms, backward 6.62 -> 6.45 ms).  With the kernels of consecutive
// chunks overlapping on two streams, 64-CTA chunks still lost (forward
// 2.42 -> 2.73 ms: more, smaller copies), and the ramp chunks at either
// end took the forward to 2.38 ms and the backward from 5.65 to 5.59 ms.
constexpr int kMaxChunks = 16;        // chunks per call at most
constexpr int64_t kChunkCtas = 128;   // CTAs a chunk's launch should keep

constexpr int kComputeStreams = 2;   // chunk kernels alternate between them

struct DeviceStreams {
    cudaStream_t in = nullptr, out = nullptr, comp[kComputeStreams] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t loaded[kMaxSlots] = {}, computed[kMaxSlots] = {}, freed[kMaxSlots] = {};
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
        for (int i = 0; i < kComputeStreams && e == cudaSuccess; ++i)
            e = cudaStreamCreateWithFlags(&ds.comp[i], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.start, cudaEventDisableTiming);
        for (int i = 0; i < kMaxSlots && e == cudaSuccess; ++i) {
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

// One chunk's work: copies in (host -> device), the kernels (enqueued by
// `compute` on the stream it is given), copies out (device -> host).
struct Copy {
    void* dst;
    const void* src;
    size_t bytes;
};
struct ChunkWork {
    Copy in[8];
    int n_in = 0;
    Copy out[4];
    int n_out = 0;
    std::function<int(cudaStream_t)> compute;
};

// Runs `chunks` chunks through `slots` workspace slots: chunk c's copies in
// wait for slot c % slots to be freed by chunk c - slots's copies out; its
// kernels run on compute stream c % 2 once its copies in are done.  The
// copies out run in chunk order on one stream and each waits for its
// chunk's kernels, so the caller's stream, which waits for the last copies
// out, completes after everything.
int run_pipeline(DeviceStreams* ds, cudaStream_t s, int64_t chunks, int slots,
                 const std::function<void(int64_t, int, ChunkWork&)>& make) {
    auto fail = [&](const char* what, cudaError_t e) {
        set_error(what, static_cast<int>(e), cudaGetErrorString(e));
        return FA_ERR_CUDA;
    };
    // the first copies in may only write the workspace once earlier work on
    // the caller's stream (which may still read it) is done; the kernels
    // likewise follow that work
    cudaError_t e = cudaEventRecord(ds->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->in, ds->start, 0);
    for (int i = 0; i < kComputeStreams && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(ds->comp[i], ds->start, 0);
    if (e != cudaSuccess) return fail("pipeline start", e);
    for (int64_t c = 0; c < chunks; ++c) {
        const int slot = static_cast<int>(c % slots);
        ChunkWork w;
        make(c, slot, w);
        if (c >= slots && (e = cudaStreamWaitEvent(ds->in, ds->freed[slot], 0)) != cudaSuccess)
            return fail("pipeline wait (slot)", e);
        for (int i = 0; i < w.n_in; ++i)
            if ((e = cudaMemcpyAsync(w.in[i].dst, w.in[i].src, w.in[i].bytes, cudaMemcpyHostToDevice, ds->in)) !=
                cudaSuccess)
                return fail("pipeline copy in", e);
        if ((e = cudaEventRecord(ds->loaded[slot], ds->in)) != cudaSuccess) return fail("pipeline record", e);
        cudaStream_t cs = ds->comp[c % kComputeStreams];
        if ((e = cudaStreamWaitEvent(cs, ds->loaded[slot], 0)) != cudaSuccess) return fail("pipeline wait (in)", e);
        const int st = w.compute(cs);
        if (st != FA_OK) return st;
        if ((e = cudaEventRecord(ds->computed[slot], cs)) != cudaSuccess) return fail("pipeline record", e);
        if ((e = cudaStreamWaitEvent(ds->out, ds->computed[slot], 0)) != cudaSuccess)
            return fail("pipeline wait (computed)", e);
        for (int i = 0; i < w.n_out; ++i)
            if ((e = cudaMemcpyAsync(w.out[i].dst, w.out[i].src, w.out[i].bytes, cudaMemcpyDeviceToHost,
                                     ds->out)) != cudaSuccess)
                return fail("pipeline copy out", e);
        if ((e = cudaEventRecord(ds->freed[slot], ds->out)) != cudaSuccess) return fail("pipeline record", e);
    }
    const int last = static_cast<int>((chunks - 1) % slots);
    if ((e = cudaStreamWaitEvent(s, ds->freed[last], 0)) != cudaSuccess) return fail("pipeline end", e);
    return FA_OK;
}

// Chunks of consecutive key/value heads (units) keeping about kChunkCtas
// CTAs each, at most kMaxChunks.
int64_t chunk_count(int64_t units, int64_t ctas_per_unit) {
    int64_t chunks = units * ctas_per_unit / kChunkCtas;
    if (chunks > kMaxChunks) chunks = kMaxChunks;
    if (chunks > units) chunks = units;
    return chunks < 1 ? 1 : chunks;
}

// The chunk boundaries: `per` units per chunk, except that, given enough
// units, the first two chunks ramp up (per/4, per/2 units) and the last two
// ramp down (per/2, per/4).  Nothing overlaps the first chunk's copies in
// or the last chunk's kernels and copies out; smaller chunks there shorten
// both.
struct ChunkGrid {
    int64_t units = 0, per = 1, count = 1;
    int64_t ramp[2] = {0, 0};  // sizes of the ramp chunks (0: no ramp)
    int64_t middle = 0;        // chunks of (at most) `per` units between the ramps

    void plan(int64_t units_, int64_t per_) {
        units = units_;
        per = per_ < 1 ? 1 : per_;
        ramp[0] = per / 4;
        ramp[1] = per / 2;
        if (ramp[0] < 1 || units < 2 * (ramp[0] + ramp[1]) + 2 * per) ramp[0] = ramp[1] = 0;
        const int64_t inner = units - 2 * (ramp[0] + ramp[1]);
        middle = (inner + per - 1) / per;
        count = middle + (ramp[0] ? 4 : 0);
    }
    // first unit and units of chunk c
    void at(int64_t c, int64_t& u0, int64_t& nu) const {
        if (!ramp[0]) {
            u0 = c * per;
            nu = (u0 + per <= units) ? per : units - u0;
            return;
        }
        const int64_t head = ramp[0] + ramp[1];
        if (c < 2) {
            u0 = c == 0 ? 0 : ramp[0];
            nu = ramp[c];
        } else if (c < 2 + middle) {
            u0 = head + (c - 2) * per;
            const int64_t end = units - head;
            nu = (u0 + per <= end) ? per : end - u0;
        } else {
            const int64_t k = c - 2 - middle;  // 0: per/2, 1: per/4
            u0 = units - head + (k == 0 ? 0 : ramp[1]);
            nu = ramp[1 - k];
        }
    }
};

// The forward chunking: units per chunk and the bytes of one slot
// (q, o, k, v, lse and split partials of a chunk).
struct Plan {
    int64_t units = 0, per_chunk = 0, chunks = 0;
    ChunkGrid grid;
    size_t q_bytes = 0, kv_bytes = 0, lse_bytes = 0, split_bytes = 0;  // per chunk
    size_t slot_bytes = 0;
};

Plan make_plan(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, int dtype) {
    Plan pl;
    const int64_t group = H / H_kv;
    const size_t elem = (dtype & 0xFF) == FA_DTYPE_F32 ? 4 : 2;
    pl.units = B * H_kv;
    // a chunk that underfills the GPU computes slower than the copies it would hide
    const bool packed = group > 1 && N_q * group <= 128;
    // causal: a chunk's launch lasts as long as its heaviest query block
    // whatever the chunk's size, so fewer, larger chunks (about 256 CTAs;
    // measured on the causal headline: 16 chunks 2.66 ms, 8 chunks 2.40 ms)
    const int64_t per_unit = packed ? 1 : group * ((N_q + 255) / 256);
    const int64_t chunks = chunk_count(pl.units, (dtype & FA_FLAG_CAUSAL) ? 2 * per_unit : per_unit);
    pl.grid.plan(pl.units, (pl.units + chunks - 1) / chunks);
    pl.per_chunk = pl.grid.per;
    pl.chunks = pl.grid.count;
    const size_t qh = static_cast<size_t>(pl.per_chunk * group);
    pl.q_bytes = qh * static_cast<size_t>(N_q) * static_cast<size_t>(d) * elem;
    pl.kv_bytes = static_cast<size_t>(pl.per_chunk) * static_cast<size_t>(N_kv) * static_cast<size_t>(d) * elem;
    pl.lse_bytes = qh * static_cast<size_t>(N_q) * sizeof(float);
    // a chunk's launch takes the library's automatic plan (key partitions
    // for the small ramp chunks, which alone underfill the GPU)
    pl.split_bytes = fa_fwd_ex_workspace_size(1, static_cast<int64_t>(qh), N_q, N_kv, d, 0);
    pl.slot_bytes = 2 * align256(pl.q_bytes) + 2 * align256(pl.kv_bytes) + align256(pl.lse_bytes) +
                    align256(pl.split_bytes);
    return pl;
}

// The backward chunking: slot = q, o, dO, dq, k, v, dk, dv, lse and the
// chunk's fa_bwd workspace.
struct BwdPlan {
    int64_t units = 0, per_chunk = 0, chunks = 0;
    ChunkGrid grid;
    size_t q_bytes = 0, kv_bytes = 0, lse_bytes = 0, ws_bytes = 0;
    size_t slot_bytes = 0;
};

BwdPlan make_bwd_plan(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d) {
    BwdPlan pl;
    const int64_t group = H / H_kv;
    pl.units = B * H_kv;
    const int64_t chunks = chunk_count(pl.units, (N_kv + 127) / 128);  // one CTA per 128 keys of a unit
    pl.grid.plan(pl.units, (pl.units + chunks - 1) / chunks);
    pl.per_chunk = pl.grid.per;
    pl.chunks = pl.grid.count;
    const size_t qh = static_cast<size_t>(pl.per_chunk * group);
    pl.q_bytes = qh * static_cast<size_t>(N_q) * static_cast<size_t>(d) * 2;
    pl.kv_bytes = static_cast<size_t>(pl.per_chunk) * static_cast<size_t>(N_kv) * static_cast<size_t>(d) * 2;
    pl.lse_bytes = qh * static_cast<size_t>(N_q) * sizeof(float);
    pl.ws_bytes = fa_bwd_workspace_size(1, static_cast<int64_t>(qh), N_q, d);
    pl.slot_bytes = 4 * align256(pl.q_bytes) + 4 * align256(pl.kv_bytes) + align256(pl.lse_bytes) +
                    align256(pl.ws_bytes);
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
    return static_cast<size_t>(pl.chunks < kFwdSlots ? pl.chunks : kFwdSlots) * pl.slot_bytes;
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
    const int slots = static_cast<int>(pl.chunks < kFwdSlots ? pl.chunks : kFwdSlots);
    const size_t ws_need = static_cast<size_t>(slots) * pl.slot_bytes;
    if (workspace_bytes < ws_need) return FA_ERR_INVALID_ARG;
    {
        // the workspace overlaps none of the host tensors
        const size_t el = (dtype & 0xFF) == FA_DTYPE_F32 ? 4 : 2;
        const size_t qb = static_cast<size_t>(B * H * N_q * d) * el;
        const size_t kvb = static_cast<size_t>(B * H_kv * N_kv * d) * el;
        const void* ptr[5] = {q, k, v, o, lse};
        const size_t len[5] = {qb, kvb, kvb, qb, lse ? static_cast<size_t>(B * H * N_q) * sizeof(float) : 0};
        for (int i = 0; i < 5; ++i)
            if (len[i] && overlaps(workspace, ws_need, ptr[i], len[i])) return FA_ERR_INVALID_ARG;
    }

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
    return run_pipeline(ds, s, pl.chunks, slots, [&](int64_t c, int slot, ChunkWork& w) {
        int64_t u0 = 0, nu = 0;
        pl.grid.at(c, u0, nu);
        const int64_t hq0 = u0 * group, nq = nu * group;  // query heads of the chunk (flattened)
        uint8_t* dq = static_cast<uint8_t*>(workspace) + static_cast<size_t>(slot) * pl.slot_bytes;
        uint8_t* dout = dq + align256(pl.q_bytes);
        uint8_t* dk = dout + align256(pl.q_bytes);
        uint8_t* dv = dk + align256(pl.kv_bytes);
        float* dl = reinterpret_cast<float*>(dv + align256(pl.kv_bytes));
        uint8_t* dsplit = reinterpret_cast<uint8_t*>(dl) + align256(pl.lse_bytes);
        const size_t qb = static_cast<size_t>(nq) * q_head, kvb = static_cast<size_t>(nu) * kv_head;
        w.in[w.n_in++] = {dq, static_cast<const uint8_t*>(q) + static_cast<size_t>(hq0) * q_head, qb};
        w.in[w.n_in++] = {dk, static_cast<const uint8_t*>(k) + static_cast<size_t>(u0) * kv_head, kvb};
        w.in[w.n_in++] = {dv, static_cast<const uint8_t*>(v) + static_cast<size_t>(u0) * kv_head, kvb};
        w.compute = [=](cudaStream_t cs) {
            return fa_fwd_ex(dq, dk, dv, dout, lse != nullptr ? dl : nullptr, 1, nq, nu, N_q, N_kv, d, scale, dtype,
                             0, pl.split_bytes ? dsplit : nullptr, pl.split_bytes, cs);
        };
        w.out[w.n_out++] = {static_cast<uint8_t*>(o) + static_cast<size_t>(hq0) * q_head, dout, qb};
        if (lse != nullptr)
            w.out[w.n_out++] = {reinterpret_cast<uint8_t*>(lse) + static_cast<size_t>(hq0) * lse_head, dl,
                                static_cast<size_t>(nq) * lse_head};
    });
}

size_t fa_bwd_host_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d) {
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_kv < 1 || (d != 64 && d != 128)) return 0;
    if (B > INT64_MAX / H || B * H > INT64_MAX / (N_q + 128) || B * H * (N_q + 128) > INT64_MAX / (d * 4)) return 0;
    if (B * H_kv > INT64_MAX / N_kv || B * H_kv * N_kv > INT64_MAX / (d * 4)) return 0;
    const BwdPlan pl = make_bwd_plan(B, H, H_kv, N_q, N_kv, d);
    return static_cast<size_t>(pl.chunks < kBwdSlots ? pl.chunks : kBwdSlots) * pl.slot_bytes;
}

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
                int64_t d, float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (workspace == nullptr) return FA_ERR_INVALID_ARG;
    // the tensor checks of fa_bwd on the whole problem (host pointers); the
    // device workspace is checked against this call's own size below
    int st = fa::validate_bwd_tensors(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N_q, N_kv, d, scale, dtype);
    if (st != FA_OK) return st;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
    const BwdPlan pl = make_bwd_plan(B, H, H_kv, N_q, N_kv, d);
    const int slots = static_cast<int>(pl.chunks < kBwdSlots ? pl.chunks : kBwdSlots);
    const size_t ws_need = static_cast<size_t>(slots) * pl.slot_bytes;
    if (workspace_bytes < ws_need) return FA_ERR_INVALID_ARG;
    {
        const void* ptr[9] = {q, k, v, o, dout, lse, dq, dk, dv};
        size_t len[9];
        fa::bwd_tensor_bytes(B, H, H_kv, N_q, N_kv, d, len);
        len[6] = len[0];
        len[7] = len[1];
        len[8] = len[2];
        for (int i = 0; i < 9; ++i)
            if (overlaps(workspace, ws_need, ptr[i], len[i])) return FA_ERR_INVALID_ARG;
    }

    DeviceStreams* ds = nullptr;
    int dev = 0;
    if ((st = device_streams(&ds, &dev)) != FA_OK) return st;
    std::lock_guard<std::mutex> lock(g_streams_mutex[dev]);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t group = H / H_kv;
    const size_t q_head = static_cast<size_t>(N_q) * static_cast<size_t>(d) * 2;
    const size_t kv_head = static_cast<size_t>(N_kv) * static_cast<size_t>(d) * 2;
    const size_t lse_head = static_cast<size_t>(N_q) * sizeof(float);
    return run_pipeline(ds, s, pl.chunks, slots, [&](int64_t c, int slot, ChunkWork& w) {
        int64_t u0 = 0, nu = 0;
        pl.grid.at(c, u0, nu);
        const int64_t hq0 = u0 * group, nq = nu * group;
        uint8_t* p0 = static_cast<uint8_t*>(workspace) + static_cast<size_t>(slot) * pl.slot_bytes;
        uint8_t* d_q = p0;
        uint8_t* d_o = d_q + align256(pl.q_bytes);
        uint8_t* d_do = d_o + align256(pl.q_bytes);
        uint8_t* d_dq = d_do + align256(pl.q_bytes);
        uint8_t* d_k = d_dq + align256(pl.q_bytes);
        uint8_t* d_v = d_k + align256(pl.kv_bytes);
        uint8_t* d_dk = d_v + align256(pl.kv_bytes);
        uint8_t* d_dv = d_dk + align256(pl.kv_bytes);
        float* d_l = reinterpret_cast<float*>(d_dv + align256(pl.kv_bytes));
        uint8_t* d_ws = reinterpret_cast<uint8_t*>(d_l) + align256(pl.lse_bytes);
        const size_t qb = static_cast<size_t>(nq) * q_head, kvb = static_cast<size_t>(nu) * kv_head;
        const size_t qoff = static_cast<size_t>(hq0) * q_head, kvoff = static_cast<size_t>(u0) * kv_head;
        w.in[w.n_in++] = {d_q, static_cast<const uint8_t*>(q) + qoff, qb};
        w.in[w.n_in++] = {d_o, static_cast<const uint8_t*>(o) + qoff, qb};
        w.in[w.n_in++] = {d_do, static_cast<const uint8_t*>(dout) + qoff, qb};
        w.in[w.n_in++] = {d_k, static_cast<const uint8_t*>(k) + kvoff, kvb};
        w.in[w.n_in++] = {d_v, static_cast<const uint8_t*>(v) + kvoff, kvb};
        w.in[w.n_in++] = {d_l, reinterpret_cast<const uint8_t*>(lse) + static_cast<size_t>(hq0) * lse_head,
                          static_cast<size_t>(nq) * lse_head};
        w.compute = [=](cudaStream_t cs) {
            return fa_bwd(d_q, d_k, d_v, d_o, d_do, d_l, d_dq, d_dk, d_dv, 1, nq, nu, N_q, N_kv, d, scale, dtype,
                          d_ws, pl.ws_bytes, cs);
        };
        w.out[w.n_out++] = {static_cast<uint8_t*>(dq) + qoff, d_dq, qb};
        w.out[w.n_out++] = {static_cast<uint8_t*>(dk) + kvoff, d_dk, kvb};
        w.out[w.n_out++] = {static_cast<uint8_t*>(dv) + kvoff, d_dv, kvb};
    });
}

}  // extern "C"
