// attn_api.cu -- the C ABI of libattn (declared in include/attn.h): argument
// validation, dispatch to the kernels, workspace sizing, status reporting.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

__device__ unsigned int g_status_word;  // kStatus* bits, cleared by attn_get_device_status

thread_local char t_last_error[256] = "";
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // bounded device waits give up after 2 s

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True for page-locked host memory the device addresses directly.
bool in_host_memory(const void* p) {
    if (!p) return false;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a pointer CUDA knows: not staged
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

uint64_t wait_limit_ns() {
    static uint64_t v = []() -> uint64_t {
        const char* e = std::getenv("ATTN_WAIT_LIMIT_US");
        if (e && *e) {
            const unsigned long long us = std::strtoull(e, nullptr, 10);
            if (us > 0) return (uint64_t)us * 1000ull;
        }
        return kDefaultWaitNs;
    }();
    return v;
}

float resolve_scale(float scale, uint32_t head_dim) {
    return scale == 0.f ? 1.0f / std::sqrt((float)head_dim) : scale;
}

}  // namespace

unsigned int* device_status_ptr() {
    static unsigned int* ptrs[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned int*>(p);
    }
    return ptrs[dev];
}

int device_sm_count() {
    static std::atomic<int> cached[64];  // 0 = not queried yet
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        if (dev >= 0 && dev < 64 && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) {
            if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
            return n;
        }
    }
    cudaGetLastError();  // no device visible: clear the sticky query error
    return 152;
}

attn_status_t record_cuda_error(cudaError_t err) {
    if (err == cudaSuccess) return ATTN_OK;
    std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s", cudaGetErrorName(err),
                  cudaGetErrorString(err));
    return ATTN_ERR_CUDA;
}

void set_last_error(const char* msg) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s", msg);
}

// Validation of the decode arguments other than the workspace, shared by
// every decode entry point.
attn_status_t check_decode_args(const float* q, const float* k_cache, const float* v_cache,
                                const float* out, uint32_t num_heads, uint32_t kv_heads,
                                uint32_t head_dim, uint32_t max_seq, uint32_t total_seq,
                                float scale) {
    if (!q || !k_cache || !v_cache || !out) return ATTN_ERR_INVALID_ARG;
    if (num_heads == 0 || kv_heads == 0 || num_heads % kv_heads != 0) return ATTN_ERR_INVALID_ARG;
    if (head_dim == 0 || head_dim % 32 != 0) return ATTN_ERR_INVALID_ARG;
    if (total_seq == 0 || total_seq > max_seq) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return ATTN_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 32 && head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "device wait timed out";
        case ATTN_ERR_RANGE: return "input outside the fp16 operand range";
    }
    return "unknown status";
}

const char* attn_last_error_string(void) { return t_last_error; }

size_t attn_prefill_workspace_size(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                   uint32_t head_dim, attn_precision_t precision) {
    if (precision == ATTN_PREC_FP32) return 0;
    if (precision == ATTN_PREC_TF32)
        return prefill_tf32_workspace_bytes(m, num_q_heads, num_kv_heads, head_dim);
    return prefill_tc_workspace_bytes(m, num_q_heads, num_kv_heads, head_dim);
}

attn_status_t attn_prefill_causal(const float* q, const float* k, const float* v, float* o,
                                  uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                  uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                  float scale, attn_precision_t precision, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (num_q_heads == 0 || num_kv_heads == 0 || num_q_heads % num_kv_heads != 0)
        return ATTN_ERR_INVALID_ARG;
    if (head_dim == 0 || head_dim % 32 != 0) return ATTN_ERR_INVALID_ARG;
    if ((uint64_t)q_stride < (uint64_t)num_q_heads * head_dim ||
        (uint64_t)kv_stride < (uint64_t)num_kv_heads * head_dim)
        return ATTN_ERR_INVALID_ARG;
    if (q_stride % 4 != 0 || kv_stride % 4 != 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (precision != ATTN_PREC_FP32 && precision != ATTN_PREC_FP16 &&
        precision != ATTN_PREC_BF16 && precision != ATTN_PREC_TF32)
        return ATTN_ERR_INVALID_ARG;
    if (m == 0) return ATTN_OK;
    const float sc = resolve_scale(scale, head_dim);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (precision == ATTN_PREC_FP32) {
        if (head_dim != 32 && head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
        return record_cuda_error(launch_prefill_fp32(q, k, v, o, m, num_q_heads, num_kv_heads,
                                                     head_dim, q_stride, kv_stride, sc, st));
    }
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    // TMA tiles address rows with 32-bit coordinates.
    if (m > 0x7fffffffu) return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_prefill_workspace_size(m, num_q_heads, num_kv_heads, head_dim,
                                                    precision);
    if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
    unsigned int* status = device_status_ptr();
    if (!status) return record_cuda_error(cudaGetLastError());
    const cudaError_t e =
        precision == ATTN_PREC_TF32
            ? launch_prefill_tf32(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                  kv_stride, sc, workspace, status, wait_limit_ns(), st)
            : launch_prefill_tc(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                kv_stride, sc, precision == ATTN_PREC_BF16, workspace, status,
                                wait_limit_ns(), st);
    if (e == cudaErrorNotSupported) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "cuTensorMapEncodeTiled unavailable or rejected the operand layout");
        return ATTN_ERR_UNSUPPORTED;
    }
    return record_cuda_error(e);
}

size_t attn_decode_workspace_size(uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                                  uint32_t total_seq, uint32_t window) {
    if (kv_heads == 0 || total_seq == 0) return 0;
    return make_decode_plan(num_heads, kv_heads, head_dim, total_seq, window, device_sm_count())
        .workspace_bytes;
}


// Shared validation of the decode entry points; fills the plan.
static attn_status_t check_decode(const float* q, const float* k_cache, const float* v_cache,
                                  const float* out, uint32_t num_heads, uint32_t kv_heads,
                                  uint32_t head_dim, uint32_t max_seq, uint32_t total_seq,
                                  uint32_t window, float scale, const void* workspace,
                                  size_t workspace_bytes, DecodePlan* plan) {
    const attn_status_t st = check_decode_args(q, k_cache, v_cache, out, num_heads, kv_heads,
                                               head_dim, max_seq, total_seq, scale);
    if (st != ATTN_OK) return st;
    *plan = make_decode_plan(num_heads, kv_heads, head_dim, total_seq, window, device_sm_count());
    if (!workspace || workspace_bytes < plan->workspace_bytes) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

attn_status_t attn_decode(const float* q, const float* k_cache, const float* v_cache,
                          float* out, uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                          uint32_t max_seq, uint32_t total_seq, uint32_t window, float scale,
                          void* workspace, size_t workspace_bytes, void* stream) {
    DecodePlan plan;
    const attn_status_t st = check_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim,
                                          max_seq, total_seq, window, scale, workspace,
                                          workspace_bytes, &plan);
    if (st != ATTN_OK) return st;
    DecodeCall c{};
    c.q = q;
    c.k_cache = k_cache;
    c.v_cache = v_cache;
    c.out = out;
    c.num_heads = num_heads;
    c.kv_heads = kv_heads;
    c.head_dim = head_dim;
    c.max_seq = max_seq;
    c.total_seq = total_seq;
    c.scale = resolve_scale(scale, head_dim);
    c.stage_inputs = in_host_memory(q);
    return record_cuda_error(
        launch_decode(c, plan, workspace, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_decode_append(const float* q, const float* k_new, const float* v_new,
                                 const float* rope_cos, const float* rope_sin, float* k_cache,
                                 float* v_cache, float* out, uint32_t num_heads,
                                 uint32_t kv_heads, uint32_t head_dim, uint32_t max_seq,
                                 uint32_t total_seq, uint32_t position, uint32_t window,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    if (!k_new || !v_new) return ATTN_ERR_INVALID_ARG;
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return ATTN_ERR_INVALID_ARG;
    if (position >= max_seq) return ATTN_ERR_INVALID_ARG;
    DecodePlan plan;
    const attn_status_t st = check_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim,
                                          max_seq, total_seq, window, scale, workspace,
                                          workspace_bytes, &plan);
    if (st != ATTN_OK) return st;
    DecodeCall c{};
    c.q = q;
    c.k_cache = k_cache;
    c.v_cache = v_cache;
    c.k_cache_w = k_cache;
    c.v_cache_w = v_cache;
    c.k_new = k_new;
    c.v_new = v_new;
    c.rope_cos = rope_cos;
    c.rope_sin = rope_sin;
    c.out = out;
    c.num_heads = num_heads;
    c.kv_heads = kv_heads;
    c.head_dim = head_dim;
    c.max_seq = max_seq;
    c.total_seq = total_seq;
    c.position = position;
    c.scale = resolve_scale(scale, head_dim);
    c.stage_inputs = in_host_memory(q) || in_host_memory(k_new) || in_host_memory(v_new) ||
                     in_host_memory(rope_cos) || in_host_memory(rope_sin);
    return record_cuda_error(
        launch_decode(c, plan, workspace, static_cast<cudaStream_t>(stream)));
}

attn_status_t kv_append(const float* k_src, const float* v_src, float* k_cache, float* v_cache,
                        uint32_t kv_heads, uint32_t head_dim, uint32_t max_seq,
                        uint32_t position, void* stream) {
    if (!k_src || !k_cache) return ATTN_ERR_INVALID_ARG;
    if ((v_src == nullptr) != (v_cache == nullptr)) return ATTN_ERR_INVALID_ARG;
    if (kv_heads == 0 || head_dim == 0 || head_dim % 4 != 0) return ATTN_ERR_INVALID_ARG;
    if (position >= max_seq) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_src) || !aligned16(k_cache) || (v_src && !aligned16(v_src)) ||
        (v_cache && !aligned16(v_cache)))
        return ATTN_ERR_INVALID_ARG;
    return record_cuda_error(launch_kv_append(k_src, v_src, k_cache, v_cache, kv_heads, head_dim,
                                              max_seq, position,
                                              static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_get_device_status(void) {
    unsigned int* p = device_status_ptr();
    if (!p) return record_cuda_error(cudaGetLastError());
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return record_cuda_error(e);
    unsigned int word = 0;
    e = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return record_cuda_error(e);
    const unsigned int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (word & kStatusTimeout) return ATTN_ERR_TIMEOUT;
    if (word & kStatusRange) return ATTN_ERR_RANGE;
    return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(uint32_t limit_us) {
    if (limit_us == 0 || limit_us > 1000000u) return ATTN_ERR_INVALID_ARG;
    attn_status_t before = attn_get_device_status();  // clear older bits
    if (before == ATTN_ERR_CUDA) return before;
    unsigned int* p = device_status_ptr();
    if (!p) return record_cuda_error(cudaGetLastError());
    cudaError_t e = launch_wait_timeout_selftest(p, (uint64_t)limit_us * 1000ull);
    if (e != cudaSuccess) return record_cuda_error(e);
    return attn_get_device_status();
}

}  // extern "C"
