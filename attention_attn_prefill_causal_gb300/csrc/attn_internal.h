// attn_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public C ABI).
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

// Device status word bits (set by kernels with atomicOr).
enum : unsigned int {
    kStatusTimeout = 1u,  // a bounded mbarrier wait gave up
    kStatusRange = 2u,    // an fp32 -> fp16 conversion overflowed
};

// Address of the device status word on the current device.
unsigned int* device_status_ptr();

// Number of SMs of the current device (152 when no device is visible).
int device_sm_count();

// Record a CUDA error for attn_last_error_string() and map it to a status.
attn_status_t record_cuda_error(cudaError_t err);

// Set the text attn_last_error_string() returns on this host thread.
void set_last_error(const char* msg);

// Raise Kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (any host thread may call it; devices past the
// cached range set it on every call).
template <auto Kernel>
cudaError_t ensure_dynamic_smem(int bytes) {
    static std::atomic<bool> done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < 64;
    if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
    return e;
}

// ---------------------------------------------------------------- decode
struct DecodePlan {
    uint32_t window_start;
    uint32_t rows_live;
    uint32_t heads_per_pass;  // query heads per CTA (1, 2, 4, 6 or 8)
    uint32_t n_hgroups;       // query-head groups per KV head
    uint32_t chunk;           // live rows per CTA
    uint32_t rows_per_warp;   // rows per warp: ceil(chunk / warps per CTA)
    uint32_t n_splits;        // CTAs (row chunks) per KV head group
    size_t part_o_floats;
    size_t part_ml_floats;
    size_t stage_floats;      // copies of q, k_new, v_new and the RoPE tables
    size_t workspace_bytes;
};
DecodePlan make_decode_plan(uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                            uint32_t total_seq, uint32_t window, int sm_count);

// One decode call; k_new == nullptr means no append (plain decode).
struct DecodeCall {
    const float* q;
    const float* k_cache;
    const float* v_cache;
    float* k_cache_w;
    float* v_cache_w;
    const float* k_new;
    const float* v_new;
    const float* rope_cos;
    const float* rope_sin;
    float* out;
    uint32_t num_heads, kv_heads, head_dim, max_seq, total_seq, position;
    float scale;
    // Some step input (q, k_new, v_new, RoPE tables) is in page-locked host
    // memory: copy them into the workspace once, so that the decode CTAs
    // read them from HBM instead of each reading them over the host link.
    bool stage_inputs;
};

// Validation of the decode arguments other than the workspace (null and
// misaligned pointers, head counts, head_dim, total_seq, scale).
attn_status_t check_decode_args(const float* q, const float* k_cache, const float* v_cache,
                                const float* out, uint32_t num_heads, uint32_t kv_heads,
                                uint32_t head_dim, uint32_t max_seq, uint32_t total_seq,
                                float scale);

cudaError_t launch_decode(const DecodeCall& call, const DecodePlan& plan, void* workspace,
                          cudaStream_t stream);

cudaError_t launch_kv_append(const float* k_src, const float* v_src, float* k_cache,
                             float* v_cache, uint32_t kv_heads, uint32_t head_dim,
                             uint32_t max_seq, uint32_t position, cudaStream_t stream);

// ---------------------------------------------------------------- prefill
cudaError_t launch_prefill_fp32(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, cudaStream_t stream);

// 16-bit tensor-core prefill (prefill_tc.cu): the single-tile kernel, or the
// pair kernel below for grids of at least two waves of query-tile pairs.
size_t prefill_tc_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                  uint32_t head_dim);

// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
cudaError_t launch_prefill_tc(const float* q, const float* k, const float* v, float* o,
                              uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                              uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                              float scale, bool bf16, void* workspace, unsigned int* status,
                              uint64_t wait_limit_ns, cudaStream_t stream);

// The 16-bit kernel over query-tile pairs (prefill_tc_pair.cu), which
// launch_prefill_tc takes for grids of at least two waves of pairs.
bool prefill_use_pairs(uint32_t m, uint32_t num_q_heads, int sm_count);
size_t prefill_pair_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                    uint32_t head_dim);
cudaError_t launch_prefill_pair(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, bool bf16, void* workspace, unsigned int* status,
                                uint64_t wait_limit_ns, cudaStream_t stream);

size_t prefill_tf32_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                    uint32_t head_dim);

// TF32 tensor-core prefill (the single-tile kernel in prefill_tc.cu);
// cudaErrorNotSupported as launch_prefill_tc.
cudaError_t launch_prefill_tf32(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, void* workspace, unsigned int* status,
                                uint64_t wait_limit_ns, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(unsigned int* status, uint64_t limit_ns);

}  // namespace attn
