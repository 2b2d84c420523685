/*
 * fa.h — fused exact-attention forward pass on GB300 (sm_103a), C ABI.
 *
 * The operation ("CUDA Flash Attention: Online Softmax with Shared Memory
 * Tiling", Problem Statement; "FlashAttention dissected", section "Algorithmic
 * core in pseudocode"): for every batch b, head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) * v_j
 *     lse[b,h,i] = log( sum_j exp(scale * q_i . k_j) )          (natural log)
 *
 * computed by one fused kernel that keeps a query tile on chip, sweeps the
 * key/value sequence tile by tile with the online-softmax update (running
 * maximum m, running denominator l, accumulator rescaled by exp(m_old - m_new);
 * "How Did I Write My First FlashAttention Kernel in CUDA?", pseudo-algorithm
 * steps 1-5) and never writes the N x N score matrix to memory.
 *
 * Every entry point is callable from C.  No torch type appears here.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* NULL pointer, size < 1, overflow, non-finite scale */
    FA_ERR_UNSUPPORTED = 2,  /* head dimension / dtype combination not built, size beyond TMA limits */
    FA_ERR_ALIGNMENT = 3,    /* a tensor base address is not 16-byte aligned */
    FA_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed (see fa_last_error_message) */
    FA_ERR_TIMEOUT = 5       /* a kernel gave up waiting on an internal barrier (device status) */
} fa_status_t;

/* Element type of q, k, v and o (the low 8 bits of every `dtype` argument). */
typedef enum {
    FA_DTYPE_F32 = 0,   /* fp32 in/out; the two contractions run on TF32 tensor cores */
    FA_DTYPE_BF16 = 1,  /* bf16 in/out; fp32 accumulation and softmax */
    FA_DTYPE_F16 = 2    /* fp16 in/out; fp32 accumulation and softmax */
} fa_dtype_t;

/*
 * Flags OR-ed into a `dtype` argument.
 *
 * FA_FLAG_CAUSAL: autoregressive attention, query i sees only the keys
 * j <= i + (N_kv - N_q) (N_q = N_kv: the usual lower-triangular mask; the
 * last query always sees every key, as a decode step against a key cache
 * does).  A query that sees no key (N_q > N_kv) gets O = 0 and lse = -inf.
 * Causal masking is not on the pages; this is the conventional reading.
 */
#define FA_FLAG_CAUSAL 0x100

/*
 * fa_fwd — enqueue the attention forward pass on `stream`.
 *
 *   q, k, v : device pointers, contiguous row-major [B, H, N, d] of `dtype`
 *             (read only; they may alias one another).
 *   o       : device pointer, [B, H, N, d] of `dtype`, written in full.
 *   lse     : device pointer, fp32 [B, H, N], natural-log units; may be NULL,
 *             which skips the store.
 *   B, H, N : batch, heads, sequence length (queries = keys = N), each >= 1.
 *   d       : head dimension: 64 or 128 for bf16 and fp16, 64 for fp32.
 *   scale   : finite score scale (1/sqrt(d) for the pages' attention).
 *   dtype   : an fa_dtype_t value, optionally OR FA_FLAG_CAUSAL.
 *   stream  : a cudaStream_t (NULL = the legacy default stream) on the
 *             current device; all pointers must be on that device.
 *
 * Ownership: the caller owns every buffer; the library allocates and frees
 * nothing on the device.  o and lse must not overlap the inputs or each other.
 *
 * Work distribution (no workspace is needed): one CTA per 256 query rows of
 * one (b, h).  When those CTAs underfill the GPU (fewer than one per SM),
 * or the last of several waves is at most half full (16-bit inputs, no
 * causal mask, N >= 4096), the affected query blocks split their keys into
 * 2 to 8 partitions that run as one thread-block cluster and combine their
 * partial results in distributed shared memory with the online-softmax
 * rescaling ("FlashAttention dissected", sections "The mathematical
 * breakthrough: Tiling and Online Softmax" and "Interaction with the KV
 * cache during inference"); see fa_fwd_launches.  This is fa_fwd_ex's
 * automatic plan (num_splits = 0) restricted to merges inside a cluster.
 *
 * Errors: argument checks run on the host before any CUDA call and return
 * FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_ALIGNMENT without side
 * effects.  A failed launch returns FA_ERR_CUDA.  The call is asynchronous:
 * FA_OK means the kernels were enqueued; a kernel that aborted on a barrier
 * timeout is reported by fa_device_status().  There is no CPU fallback.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int64_t B, int64_t H, int64_t N, int64_t d, float scale, int dtype,
           void* stream);

/*
 * Kernel launches fa_fwd enqueues for these sizes on the current device: 1,
 * or 2 when the last wave's query blocks run split in a second launch; 0 for
 * invalid sizes.  The SM count and cluster occupancy of the current device
 * are the CUDA queries here (without a device the plan is one launch).
 */
int fa_fwd_launches(int64_t B, int64_t H, int64_t N, int64_t d, int dtype);

/*
 * fa_fwd_validate — the host-side argument checks of fa_fwd, alone.  Returns
 * the status fa_fwd would return before touching CUDA.  Makes no CUDA call,
 * so it also runs on machines without a GPU.
 */
int fa_fwd_validate(const void* q, const void* k, const void* v, void* o,
                    const float* lse, int64_t B, int64_t H, int64_t N,
                    int64_t d, float scale, int dtype);

/*
 * fa_fwd_ex — the general form: decode shapes, grouped-query heads and
 * key-range partitions ("split-KV").
 *
 *   q, o    : [B, H, N_q, d] of `dtype`;   k, v : [B, H_kv, N_kv, d];
 *   lse     : fp32 [B, H, N_q] or NULL.
 *   H_kv    : key/value heads, dividing H; query head h reads key/value
 *             head h / (H / H_kv) (grouped-query attention; H_kv = H is
 *             ordinary multi-head attention).
 *   N_q, N_kv: query rows and key/value rows per head (N_q = 1 is a decode
 *             step against a cache of N_kv keys, the FlashDecoding case of
 *             "FlashAttention dissected", section "Interaction with the KV
 *             cache during inference").
 *   num_splits: >= 1 key-range partitions per query block.  1 runs the fused
 *             kernel alone.  More partitions sweep disjoint key ranges in
 *             separate CTAs, which then fill the GPU when B * H * N_q is
 *             small; their partial results go to `workspace` and a second
 *             kernel merges them with the online-softmax rescaling.  The
 *             count is capped at 32 and at one partition per 128 keys.
 *             0 chooses automatically for the current device (one CTA per
 *             SM): a launch with fewer query blocks than SMs gets the
 *             fa_fwd_ex_splits count, merged inside thread-block clusters
 *             (distributed shared memory, no workspace, no merge kernel)
 *             when at most 8 partitions are wanted and every query block's
 *             cluster fits on the device at once, else through the
 *             workspace and the merge kernel; a launch of several waves
 *             whose last wave is at most half full (16-bit inputs,
 *             unmasked, query heads not packed, N_kv >= 4096) runs the full
 *             waves unsplit and the last wave's query blocks in a second
 *             launch, split along the keys (up to 4 partitions) into
 *             clusters that merge in-cluster; otherwise one partition.
 *   workspace, workspace_bytes: device scratch owned by the caller, 16-byte
 *             aligned, at least fa_fwd_ex_workspace_size(...) bytes; may be
 *             NULL when that size is 0.  Contents on entry do not matter.
 *
 * Same ownership, validation and error behaviour as fa_fwd; the workspace
 * must not overlap any tensor.  Every kernel of the call (one to three, see
 * fa_fwd_ex_launches) is enqueued on `stream`.
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
              int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
              int64_t d, float scale, int dtype, int num_splits,
              void* workspace, size_t workspace_bytes, void* stream);

/* Host-side argument checks of fa_fwd_ex alone (no CUDA call, except the
 * SM-count query of the current device when num_splits = 0). */
int fa_fwd_ex_validate(const void* q, const void* k, const void* v, void* o,
                       const float* lse, int64_t B, int64_t H, int64_t H_kv,
                       int64_t N_q, int64_t N_kv, int64_t d, float scale,
                       int dtype, int num_splits, const void* workspace,
                       size_t workspace_bytes);

/*
 * Workspace bytes fa_fwd_ex needs for `num_splits` (after the same capping):
 * splits * B * H * N_q * (d + 4) * 4, or 0 when one partition remains.
 * Pure host computation; 0 for invalid sizes.  num_splits = 0 (automatic):
 * a bound for every plan on the current device, min(SMs * 256,
 * 32 * B * H * N_q) * (d + 4) * 4 (SMs taken as 1024 when no device answers;
 * the SM count is the one CUDA query here).
 */
size_t fa_fwd_ex_workspace_size(int64_t B, int64_t H, int64_t N_q, int64_t N_kv,
                                int64_t d, int num_splits);

/*
 * A partition count that fills about one wave of `num_sms` SMs: 1 when the
 * CTAs of one partition already fill the GPU, else num_sms / that count
 * (capped as above).  A partition has B * H * ceil(N_q / 256) CTAs, or
 * B * H_kv when the grouped query heads are packed (H_kv < H and
 * N_q * H / H_kv <= 128: one CTA serves all query heads of a key/value head,
 * e.g. for decode steps).  Pure host computation; 1 for invalid sizes.
 */
int fa_fwd_ex_splits(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
                     int num_sms);

/*
 * Kernel launches fa_fwd_ex enqueues for these arguments: 1 (one key
 * partition, or partitions merged in-cluster), 2 (partitions and their
 * merge kernel, or num_splits = 0 with a split tail: the full waves, then
 * the tail's clusters), 3 (partitions through the workspace, their merge and
 * a tail launch; not produced by the current plan); 0 for invalid sizes.  For num_splits = 0 the plan is the current device's (the
 * SM-count query is the one CUDA call here).
 */
int fa_fwd_ex_launches(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
                       int64_t d, int dtype, int num_splits);

/*
 * fa_fwd_ex_static — fa_fwd_ex for callers that cannot allocate device
 * memory (plugins of engines that own the whole device memory pool, or
 * per-step code that must not call cudaMalloc, which can synchronise the
 * device and can fail at run time).  Same arguments and results as
 * fa_fwd_ex without the workspace: the split partials go to one static
 * device array of fa_fwd_ex_static_capacity() bytes (32 MiB) that the library
 * holds on every GPU that loads it, until the process exits.  The library
 * allocates nothing.
 *
 *   - Sizes whose partials exceed the capacity return FA_ERR_UNSUPPORTED
 *     (fa_fwd_ex_workspace_size() gives the bytes a call needs).
 *   - The first call on a device (and the first after a device reset)
 *     looks up the array's device address (cudaGetSymbolAddress) with that
 *     device current; make that first call before any stream capture.
 *   - Plans that merge their partitions inside thread-block clusters (see
 *     fa_fwd_ex, num_splits = 0) do not touch the array.
 *   - Every call on a device shares the array, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose kernels
 *     may overlap on the GPU race on it: serialise them.
 *
 * The pages have no counterpart of this entry point.
 */
int fa_fwd_ex_static(const void* q, const void* k, const void* v, void* o,
                     float* lse, int64_t B, int64_t H, int64_t H_kv,
                     int64_t N_q, int64_t N_kv, int64_t d, float scale,
                     int dtype, int num_splits, void* stream);

/* Bytes of the static array fa_fwd_ex_static uses, per device. */
size_t fa_fwd_ex_static_capacity(void);

/*
 * fa_fwd_host — fa_fwd_ex on tensors in HOST memory: the inputs are copied
 * to the GPU, the forward pass runs, and o and lse are copied back, with the
 * copies of one chunk of key/value heads overlapped with the computation of
 * the previous one (three streams: the caller's `stream` for the kernels and
 * two the library creates once per device).  Same arguments, layouts, dtypes,
 * flags and checks as fa_fwd_ex with num_splits = 1, except:
 *   q, k, v, o, lse : host memory; pinned (page-locked) memory is needed
 *                     for the copies to overlap (pageable memory works but
 *                     serialises them).
 *   workspace       : caller-owned DEVICE memory of at least
 *                     fa_fwd_host_workspace_size(...) bytes, 256-byte
 *                     aligned (three chunk slots of q, k, v, o, lse).
 * Completion: when `stream` reaches the point after this call, o and lse
 * hold the results in host memory.  Calls on one device share the two
 * internal streams (a mutex serialises their enqueueing).  Returns as
 * fa_fwd_ex; FA_ERR_INVALID_ARG for a missing or short workspace,
 * FA_ERR_ALIGNMENT for a workspace not 256-byte aligned.
 * The pages have no counterpart of this entry point; it is the host-to-host
 * form of the forward pass that end-to-end measurements call.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
                int64_t d, float scale, int dtype, void* workspace,
                size_t workspace_bytes, void* stream);

/* Device workspace bytes fa_fwd_host needs (0 for invalid sizes). */
size_t fa_fwd_host_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t N_q,
                                  int64_t N_kv, int64_t d, int dtype);

/*
 * fa_bwd — gradients of exact attention for an upstream gradient dO:
 *
 *   P = softmax(scale Q K^T) (recomputed from q, k and the saved lse),
 *   dV = P^T dO,  dS = P o (dO V^T - D),  D_i = dO_i . O_i,
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 * "FlashAttention dissected", section "Memory complexity: from O(N^2) to
 * O(N)": the backward pass recomputes the attention blocks from Q, K, V and
 * the saved softmax statistics instead of storing the N x N matrix; the
 * gradient is the exact one of the forward definition (the pages give no
 * formula; this is the chain rule through O = P V and the softmax formula of
 * the same page).  The causal mask and grouped heads are those of fa_fwd_ex.
 *
 * Layout (contiguous, row-major, dtype = the inputs' dtype):
 *   q, o, dout, dq : [B, H, N_q, d]      k, v, dk, dv : [B, H_kv, N_kv, d]
 *   lse            : fp32 [B, H, N_q], natural log, as fa_fwd / fa_fwd_ex
 *                    return it (a row with no visible key: -inf)
 *   o and lse must be the forward outputs for the same q, k, v, scale and
 *   mask; dk and dv sum over the H / H_kv query heads sharing a key/value
 *   head.
 * dtype: FA_DTYPE_BF16 or FA_DTYPE_F16, optionally | FA_FLAG_CAUSAL;
 *   FA_DTYPE_F32 returns FA_ERR_UNSUPPORTED.  d: 64 or 128.
 * workspace: caller-owned device memory of at least
 *   fa_bwd_workspace_size(B, H, N_q, d) bytes, 16-byte aligned (fp32 row
 *   statistics and the fp32 dQ accumulator; nothing needs to be zeroed).
 * Ownership and errors: as fa_fwd_ex.  Every pointer must be non-NULL and
 *   16-byte aligned (lse 4-byte); dq, dk, dv and the workspace must not
 *   overlap any input or one another (inputs may alias one another).
 *   Validation failures return before any CUDA call.  Three kernels are
 *   enqueued on `stream`; the call does not wait for them.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o,
           const void* dout, const float* lse, void* dq, void* dk, void* dv,
           int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
           int64_t d, float scale, int dtype, void* workspace,
           size_t workspace_bytes, void* stream);

/* The argument checks of fa_bwd alone; never touches the GPU. */
int fa_bwd_validate(const void* q, const void* k, const void* v, const void* o,
                    const void* dout, const float* lse, void* dq, void* dk,
                    void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t N_q,
                    int64_t N_kv, int64_t d, float scale, int dtype,
                    const void* workspace, size_t workspace_bytes);

/*
 * fa_bwd_host — fa_bwd on tensors in HOST memory (q, k, v, o, dout, lse in;
 * dq, dk, dv out), with the copies of one chunk of key/value heads
 * overlapped with the computation of the previous one, as fa_fwd_host does
 * (it shares that entry point's two internal streams).  Same arguments,
 * layouts, dtypes, flags and checks as fa_bwd, except: the tensors are host
 * memory (pinned for the copies to overlap), and `workspace` is device
 * memory of at least fa_bwd_host_workspace_size(...) bytes, 256-byte
 * aligned.  Completion on `stream` means dq, dk, dv are in host memory.
 * The pages have no counterpart of this entry point.
 */
int fa_bwd_host(const void* q, const void* k, const void* v, const void* o,
                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv,
                int64_t d, float scale, int dtype, void* workspace,
                size_t workspace_bytes, void* stream);

/* Device workspace bytes fa_bwd_host needs (0 for invalid sizes). */
size_t fa_bwd_host_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t N_q,
                                  int64_t N_kv, int64_t d);

/* Workspace bytes fa_bwd needs (0 for invalid sizes):
   8 * B * H * ceil(N_q / 128) * 128 (rounded up to 256) + 4 * B * H * N_q * d. */
size_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N_q, int64_t d);

/*
 * fa_device_status — synchronise `stream`, then read and clear the device
 * error word the kernels set when a bounded wait gives up.  Returns FA_OK,
 * FA_ERR_TIMEOUT, or FA_ERR_CUDA if the synchronisation itself failed.
 * A launch that timed out leaves its outputs incomplete (the CTAs of that
 * launch stop early); later launches run normally whether or not the word
 * has been read.
 *
 * Source: "CUDA Flash Attention: Online Softmax with Shared Memory Tiling",
 * Correctness Audit (13-Category Checklist), row "Async error surfacing"
 * (the fused kernel's launch errors are checked with cudaGetLastError).  The
 * page surfaces launch errors only; this call extends the same rule to
 * errors a kernel detects while it runs, which an asynchronous launch cannot
 * return.
 */
int fa_device_status(void* stream);

/*
 * fa_selftest_barrier_timeout — enqueue on `stream` a one-CTA kernel that
 * waits, with the forward kernel's bounded barrier wait (about 1 s), on a
 * barrier phase that nothing completes.  The wait gives up, the kernel exits
 * normally and fa_device_status(stream) then returns FA_ERR_TIMEOUT (once).
 * It exercises the failure-reporting path without faulting or hanging the
 * GPU; the context stays usable.  Returns FA_OK or FA_ERR_CUDA (launch).
 */
int fa_selftest_barrier_timeout(void* stream);

/*
 * Static English text for a status code; never NULL.
 *
 * Source: "CUDA Flash Attention: Online Softmax with Shared Memory Tiling",
 * Correctness Audit (13-Category Checklist), rows "Async error surfacing"
 * (cudaGetLastError after the launch) and "Latent coupling bugs" (the head
 * dimension is checked, assert(d==64), instead of assumed).  Here those
 * checks return status codes instead of aborting, and this call names them.
 */
const char* fa_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* fa_last_error_message(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
