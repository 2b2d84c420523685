// Host-side helpers shared by the forward (fa_api.cu) and backward
// (fa_bwd_api.cu) entry points.  Not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {
namespace host {

// Record the message fa_last_error_message returns on this thread.
void set_error(const char* what, int code, const char* text);

// Launch generation: a fresh nonzero number per launch (the device status
// word's abort_gen starts at 0).
unsigned int next_generation();

// Device address of the status words on the current device; *status gets
// FA_OK or FA_ERR_CUDA (with the error message set).
DevStatus* device_status_words(int* status);

// Per-device cache of one __device__ variable's address.  Entries are keyed
// on the device's current CUDA context, so a device reset (which unloads the
// module and may move the variable) is followed by a fresh lookup.
constexpr int kMaxCachedDevices = 64;
struct SymbolCache {
    void* ptr[kMaxCachedDevices] = {};
    unsigned long long ctx_id[kMaxCachedDevices] = {};
    // `symbol`: the address of the variable as host code names it.
    void* address(const void* symbol, const char* what, int* status);
};

// True when the byte ranges [a, a + na) and [b, b + nb) intersect.
bool overlaps(const void* a, size_t na, const void* b, size_t nb);

// 3-D tiled TMA map over a contiguous [BH, N, d] tensor of `dtype` (innermost
// dimension first), 128-byte swizzle, boxes of 128 bytes x box_rows rows x
// box_heads heads; rows past N read as zero and are not written.  Returns
// FA_OK or FA_ERR_CUDA.
int encode_map(CUtensorMap* map, const void* base, int dtype, int64_t BH, int64_t N, int64_t d,
               uint32_t box_rows = 128, uint32_t box_heads = 1);

}  // namespace host
}  // namespace fa
