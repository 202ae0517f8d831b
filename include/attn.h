/*
 * attn.h -- C ABI of libattn: grouped-query causal prefill attention,
 * single-query decode attention with an optional sliding window, and the
 * K/V cache append, on one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers to fp32 data unless stated.  The
 *    caller owns every buffer (inputs, outputs, caches, workspaces); the
 *    library never allocates, frees or retains caller memory.
 *  - Host-resident step buffers.  The decode entry points and kv_append also
 *    accept their small per-step buffers -- q, out, k_new, v_new, rope_cos,
 *    rope_sin, k_src, v_src -- in page-locked host memory that the device
 *    addresses directly (cudaHostAlloc / cudaMallocHost under unified
 *    addressing, or cudaHostRegister with cudaHostRegisterMapped).  The
 *    kernels then read and write those bytes over the CPU-GPU link in the
 *    call itself, with no separate copy (a decode call whose inputs are
 *    host-resident first copies them into its workspace with one small
 *    kernel, so that every CTA then reads them from HBM).  Caches, workspaces and every
 *    prefill buffer must be device memory (they are moved with TMA and bulk
 *    copies).  Pageable host memory is not supported anywhere.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).  Results are ready when the
 *    stream reaches the call.  No call synchronises the host except
 *    attn_get_device_status.
 *  - Kernels launch as programmatic dependents of the kernel before them on
 *    the stream: they may become resident while it drains, but no call reads
 *    an input or writes an output before every kernel enqueued earlier on
 *    the stream has completed (the decode kernel only warms L2 with cache
 *    rows meanwhile).  Stream order is therefore unchanged for the caller,
 *    including for inputs that the previous kernel writes.  (The guarantee
 *    reaches past the previous kernel as long as every earlier kernel that
 *    was itself launched as a programmatic dependent waits for its own
 *    predecessor before completing, as all of this library's kernels do.)
 *  - Pointers and row strides must be 16-byte aligned (4 fp32 elements): the
 *    kernels move rows with 128-bit loads and TMA tiles.
 *  - A call with a rejected argument launches nothing and returns
 *    ATTN_ERR_INVALID_ARG or ATTN_ERR_UNSUPPORTED.  ATTN_ERR_CUDA means a
 *    launch failed; attn_last_error_string() then names the CUDA error.
 *  - Overlapping an output with any input is undefined.
 *
 * Citations name the web page and the item on it that defines the operation.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null pointer, inconsistent sizes, misalignment */
    ATTN_ERR_UNSUPPORTED = 2, /* valid, but outside the compiled kernel set */
    ATTN_ERR_CUDA = 3,        /* a CUDA launch or query failed */
    ATTN_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
    ATTN_ERR_RANGE = 5        /* an input overflowed the fp16 operand range */
} attn_status_t;

typedef enum {
    /* Exact mode: fp32 CUDA-core arithmetic throughout (any head_dim in
     * {32, 64, 128}). */
    ATTN_PREC_FP32 = 0,
    /* Tensor-core mode: Q, K, V rounded to fp16 (round-to-nearest, 10-bit
     * mantissa as in TF32; K and V by a pre-pass into the workspace, Q
     * inside the kernel), P rounded to fp16, tcgen05 MMAs with fp32
     * accumulation, fp32 softmax statistics and fp32 output.  head_dim in
     * {64, 128}; |q|, |k|, |v| must stay below 65504 (a larger input sets
     * ATTN_ERR_RANGE in the device status). */
    ATTN_PREC_FP16 = 1,
    /* As ATTN_PREC_FP16 with bf16 operands (8-bit mantissa): wider range,
     * larger rounding error. */
    ATTN_PREC_BF16 = 2,
    /* Tensor-core mode with TF32 operands: tcgen05 kind::tf32 MMAs read fp32
     * data and use its top 19 bits (fp32's exponent, a 10-bit mantissa).  Q
     * is rounded to nearest TF32 inside the kernel; K and V by a pre-pass
     * into the workspace (V also transposed); P is written as fp32; fp32
     * accumulation, softmax statistics and output.  No input range limit
     * beyond fp32's own; half the 16-bit tensor rate.  head_dim in {64, 128}. */
    ATTN_PREC_TF32 = 3
} attn_precision_t;

/*
 * attn_prefill_causal -- fused causal grouped-query attention over M tokens.
 *
 * Defined by "aprender-gpu 0.32.0 -- src/kernels/attention/flash/
 * prefill_fused.rs": module doc (Algorithm 1-3: GQA map, causal j <= i,
 * online softmax, normalise) and `build_ptx` (parameters q_ptr, k_ptr, v_ptr,
 * o_ptr, m, q_stride, kv_stride, num_q_heads; scale 1/sqrt(head_dim)).
 *
 *   q : [m, q_stride]  fp32; query head h is columns [h*head_dim, (h+1)*head_dim)
 *   k : [m, kv_stride] fp32; KV head g is columns [g*head_dim, (g+1)*head_dim)
 *   v : [m, kv_stride] fp32; same layout as k
 *   o : [m, q_stride]  fp32 output; only the head columns are written
 *   kv head of query head h = h / (num_q_heads / num_kv_heads)
 *   O[i,h,:] = sum_{j<=i} softmax_j(scale * Q[i,h,:].K[j,g,:]) V[j,g,:]
 *
 *   scale      : > 0, or 0 for the default 1/sqrt(head_dim)
 *   precision  : an attn_precision_t
 *   workspace  : device scratch of at least attn_prefill_workspace_size()
 *                bytes (may be NULL when that size is 0); the call owns it
 *                until the stream passes the call.  256-byte aligned.
 * Validation: num_kv_heads > 0 and divides num_q_heads; head_dim % 32 == 0
 * (the page's constructor assertion); q_stride >= num_q_heads*head_dim;
 * kv_stride >= num_kv_heads*head_dim; strides % 4 == 0.  m == 0 is a no-op.
 * ATTN_ERR_UNSUPPORTED: head_dim outside {32, 64, 128} (FP32) or
 * {64, 128} (FP16/BF16/TF32).
 */
attn_status_t attn_prefill_causal(const float* q, const float* k, const float* v, float* o,
                                  uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                  uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                  float scale, attn_precision_t precision, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Bytes of device workspace attn_prefill_causal needs for these sizes
 * (0 for ATTN_PREC_FP32): the rounded K and V (fp16/bf16, or TF32-rounded
 * fp32 with V transposed), plus per-chunk partials when the call splits its
 * key walk (small problems).  Depends only on the arguments and on the
 * current device's SM count. */
size_t attn_prefill_workspace_size(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                   uint32_t head_dim, attn_precision_t precision);

/*
 * attn_decode -- single-query grouped-query attention against a K/V cache.
 *
 * Defined by "soft3/glia/run/backend/honeycrisp/kernels/attention.rs":
 * module doc (inputs, per-head formula, sliding window) and the decode
 * kernel `kmain` (window_start, the -1e4 score of masked positions, online
 * softmax, normalisation), Params {total_seq, window, scale}.
 *
 *   q       : [num_heads, head_dim] fp32
 *   k_cache : [kv_heads, max_seq, head_dim] fp32; rows [0, total_seq) valid
 *   v_cache : same shape as k_cache
 *   out     : [num_heads, head_dim] fp32
 *   kv head of query head h = h / (num_heads / kv_heads)
 *   window_start = (window > 0 && total_seq > window) ? total_seq - window : 0
 *   score_s = scale * q[h].K[g,s], replaced by -1e4 for s < window_start
 *   out[h] = sum_s softmax(score)_s V[g,s]
 * Positions below window_start keep their -1e4 score exactly: the kernels
 * skip reading them and add their (normally zero) weight back in the
 * combine step, reading their V rows only when that weight is not zero.
 *
 *   scale     : > 0, or 0 for the default 1/sqrt(head_dim)
 *   window    : 0 = no window
 *   workspace : device scratch of at least attn_decode_workspace_size()
 *               bytes, 256-byte aligned; owned by the call until the stream
 *               passes it.
 * Validation: total_seq in [1, max_seq] (total_seq == 0 has no softmax);
 * kv_heads > 0 and divides num_heads; head_dim % 32 == 0.
 * ATTN_ERR_UNSUPPORTED: head_dim outside {32, 64, 128}.
 */
attn_status_t attn_decode(const float* q, const float* k_cache, const float* v_cache,
                          float* out, uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                          uint32_t max_seq, uint32_t total_seq, uint32_t window, float scale,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_decode needs.  Depends on the arguments and on the
 * SM count of the current device (152 is assumed when no device is
 * visible).  Its contents need no initialisation.  Calls that overlap on the
 * GPU need separate workspaces. */
size_t attn_decode_workspace_size(uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                                  uint32_t total_seq, uint32_t window);

/*
 * attn_decode_append -- append one K/V row (optionally rotated) and decode,
 * in one launch.
 *
 * Defined by "soft3/glia/run/backend/honeycrisp/kernels/attention.rs",
 * FUSED_ROPE_KV_ATTN_TEMPLATE: the new key is rotated with rotate-half RoPE
 * (element d pairs with d + head_dim/2: x'[d] = x[d]cos[d] - x[d+h]sin[d],
 * x'[d+h] = x[d]sin[d] + x[d+h]cos[d], h = head_dim/2) and written to
 * k_cache[g, position]; v_new is copied to v_cache[g, position]; the query is
 * rotated the same way; then the decode of attn_decode runs over
 * [0, total_seq) with the window, seeing the appended row.
 *
 *   k_new, v_new        : [kv_heads, head_dim] fp32
 *   rope_cos, rope_sin  : [head_dim/2] fp32 tables for this position, or both
 *                         NULL for no rotation (plain append + decode)
 *   position            : row written; < max_seq (normally total_seq - 1)
 * Other arguments, workspace rules and validation as attn_decode.
 */
attn_status_t attn_decode_append(const float* q, const float* k_new, const float* v_new,
                                 const float* rope_cos, const float* rope_sin, float* k_cache,
                                 float* v_cache, float* out, uint32_t num_heads,
                                 uint32_t kv_heads, uint32_t head_dim, uint32_t max_seq,
                                 uint32_t total_seq, uint32_t position, uint32_t window,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * attn_decode_noalloc -- attn_decode without a caller workspace.  The pages
 * have no counterpart: this entry point exists for callers that cannot
 * allocate device memory or pass a workspace (an engine that owns every free
 * byte of HBM in its own pools, a plugin interface that hands over only
 * input and output pointers, a loop where allocation is not allowed).
 *
 * Same arguments, results and validation as attn_decode, minus the
 * workspace.  Its workspace (the per-chunk partials) is a fixed 4 MiB
 * device array inside libattn (resident on every GPU that loads the library, until exit); sizes
 * whose attn_decode_workspace_size() exceeds 4 MiB are rejected with
 * ATTN_ERR_UNSUPPORTED and a message in attn_last_error_string().  The call
 * allocates nothing.  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  All calls on a device share the array:
 * calls that overlap on the GPU race and corrupt each other's output.
 */
attn_status_t attn_decode_noalloc(const float* q, const float* k_cache, const float* v_cache,
                                  float* out, uint32_t num_heads, uint32_t kv_heads,
                                  uint32_t head_dim, uint32_t max_seq, uint32_t total_seq,
                                  uint32_t window, float scale, void* stream);

/*
 * kv_append -- write one new K row and one new V row into the caches.
 *
 * Defined by "soft3/glia/run/backend/honeycrisp/kernels/attention.rs",
 * KV_APPEND_BOTH_TEMPLATE (and KV_APPEND_TEMPLATE for a single cache):
 *   k_cache[g, position, :] = k_src[g, :],  v_cache[g, position, :] = v_src[g, :]
 *
 *   k_src, v_src     : [kv_heads, head_dim] fp32
 *   k_cache, v_cache : [kv_heads, max_seq, head_dim] fp32
 * v_src and v_cache may both be NULL to append to the K cache only.
 * Validation: position < max_seq; head_dim % 4 == 0 (16-byte rows).
 */
attn_status_t kv_append(const float* k_src, const float* v_src, float* k_cache, float* v_cache,
                        uint32_t kv_heads, uint32_t head_dim, uint32_t max_seq,
                        uint32_t position, void* stream);

/* Text for a status code (static storage). */
const char* attn_status_string(attn_status_t status);

/* Text of the last CUDA error seen by a call on this host thread ("" if
 * none). */
const char* attn_last_error_string(void);

/*
 * Synchronises the current device, then reads and clears the device-side
 * status word that kernels set when a bounded wait gave up
 * (ATTN_ERR_TIMEOUT) or an fp16 conversion overflowed (ATTN_ERR_RANGE).
 * Returns ATTN_OK when neither happened since the last read.
 */
attn_status_t attn_get_device_status(void);

/*
 * Failure-detection self-test: launches one CTA that waits on an mbarrier
 * nothing will ever complete, with a wait limit of `limit_us` microseconds,
 * so the bounded-wait path fires.  Returns ATTN_ERR_TIMEOUT (read back through
 * the same device status word) when the wait gave up and the kernel returned
 * cleanly, another status otherwise.  Synchronises the device.
 */
attn_status_t attn_selftest_wait_timeout(uint32_t limit_us);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_H_ */
