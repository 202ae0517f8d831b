// decode.cu -- single-query grouped-query decode attention against a
// [kv_heads, max_seq, head_dim] K/V cache, split along the sequence
// (flash-decoding), plus the K/V cache append.
//
// Operation ("soft3/glia/run/backend/honeycrisp/kernels/attention.rs",
// module doc and decode kernel `kmain`): for query head h with KV head
// g = h / (num_heads / kv_heads), score_s = scale * q[h].K[g,s] for
// s < total_seq, replaced by -1e4 below window_start; out[h] is the
// softmax-weighted sum of V[g,s].
//
// GB300 design (the page runs one 32-lane SIMD-group per head over the whole
// sequence, which leaves most of a 152-SM GPU idle):
//  * split kernel: one CTA per (sequence chunk, KV head, group of <= 8 query
//    heads).  Each K/V row is streamed from HBM once with 128-bit loads and
//    scored against every query head of its GQA group, so the cache is read
//    once rather than once per query head.  A warp owns one row at a time
//    (lane l holds elements [l*V, l*V+V) of the row), reduces the dot
//    products with warp shuffles and keeps a running max / sum / output per
//    head (online softmax in base 2).  The warps of a CTA merge their states
//    and write one partial (m, l, O) per (query head, split).
//  * combine kernel: merges the partials of each query head with a
//    log-sum-exp and normalises.  Positions below window_start are never
//    read by the split kernel; their score is -1e4 exactly as on the page,
//    and the combine adds their weight exp(-1e4 - max) back in.  That weight
//    is zero in fp32 unless every live score is below about -9896, in which
//    case the combine reads the masked V rows and adds them exactly.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kDecodeThreads = 256;            // 8 warps
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kRowsPerStep = 4;                // K/V rows a warp loads per step
constexpr int kMaxHeadsPerPass = 8;            // query heads per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaskScore = -1.0e4f;          // the page's replaced score

template <int VEC>
struct Vec;
template <>
struct Vec<1> {
    using T = float;
    __device__ static T ld(const float* p) { return __ldcs(p); }
    __device__ static T ldq(const float* p) { return *p; }
    __device__ static float get(const T& v, int i) { return v; }
};
template <>
struct Vec<2> {
    using T = float2;
    __device__ static T ld(const float* p) { return __ldcs(reinterpret_cast<const float2*>(p)); }
    __device__ static T ldq(const float* p) { return *reinterpret_cast<const float2*>(p); }
    __device__ static float get(const T& v, int i) { return i == 0 ? v.x : v.y; }
};
template <>
struct Vec<4> {
    using T = float4;
    __device__ static T ld(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
    __device__ static T ldq(const float* p) { return *reinterpret_cast<const float4*>(p); }
    __device__ static float get(const T& v, int i) {
        return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
    }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Split kernel.  grid = (n_splits, kv_heads, n_hgroups), block = 256.
// part_o  : [num_heads, n_splits, D]  unnormalised partial outputs
// part_ml : [num_heads, n_splits, 2]  (running max in log2 units, sum)
template <int D>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_split_kernel(const float* __restrict__ q, const float* __restrict__ k_cache,
                    const float* __restrict__ v_cache, float* __restrict__ part_o,
                    float* __restrict__ part_ml, uint32_t heads_per_kv, uint32_t max_seq,
                    uint32_t window_start, uint32_t total_seq, uint32_t chunk,
                    uint32_t n_splits, float scale_log2) {
    constexpr int V = D / 32;
    using VT = typename Vec<V>::T;
    __shared__ float sm_m[kDecodeWarps][kMaxHeadsPerPass];
    __shared__ float sm_l[kDecodeWarps][kMaxHeadsPerPass];
    __shared__ float sm_o[kDecodeWarps][kMaxHeadsPerPass][D];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t split = blockIdx.x, kvh = blockIdx.y;
    const uint32_t hg0 = blockIdx.z * kMaxHeadsPerPass;
    const int ng = (int)min((uint32_t)kMaxHeadsPerPass, heads_per_kv - hg0);
    const uint32_t h0 = kvh * heads_per_kv + hg0;  // first query head of this CTA
    const uint32_t r0 = window_start + split * chunk;
    const uint32_t r1 = min(r0 + chunk, total_seq);

    float qr[kMaxHeadsPerPass][V];
#pragma unroll
    for (int g = 0; g < kMaxHeadsPerPass; ++g) {
        if (g < ng) {
            VT t = Vec<V>::ldq(q + (size_t)(h0 + g) * D + lane * V);
#pragma unroll
            for (int e = 0; e < V; ++e) qr[g][e] = Vec<V>::get(t, e) * scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) qr[g][e] = 0.f;
        }
    }
    float m[kMaxHeadsPerPass], l[kMaxHeadsPerPass], o[kMaxHeadsPerPass][V];
#pragma unroll
    for (int g = 0; g < kMaxHeadsPerPass; ++g) {
        m[g] = -CUDART_INF_F;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) o[g][e] = 0.f;
    }

    const float* kb = k_cache + (size_t)kvh * max_seq * D + lane * V;
    const float* vb = v_cache + (size_t)kvh * max_seq * D + lane * V;
    for (uint32_t base = r0 + warp * kRowsPerStep; base < r1;
         base += kDecodeWarps * kRowsPerStep) {
        VT kr[kRowsPerStep], vr[kRowsPerStep];
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
            const uint32_t r = base + u;
            if (r < r1) {
                kr[u] = Vec<V>::ld(kb + (size_t)r * D);
                vr[u] = Vec<V>::ld(vb + (size_t)r * D);
            } else {
                kr[u] = VT{};
                vr[u] = VT{};
            }
        }
#pragma unroll
        for (int g = 0; g < kMaxHeadsPerPass; ++g) {
            if (g >= ng) continue;
            float s[kRowsPerStep];
            float mx = m[g];
#pragma unroll
            for (int u = 0; u < kRowsPerStep; ++u) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < V; ++e) d = fmaf(qr[g][e], Vec<V>::get(kr[u], e), d);
                d = warp_sum(d);
                s[u] = (base + u < r1) ? d : -CUDART_INF_F;
                mx = fmaxf(mx, s[u]);
            }
            const float corr = exp2f(m[g] - mx);  // m = -inf on the first step -> 0
            float lsum = l[g] * corr;
#pragma unroll
            for (int e = 0; e < V; ++e) o[g][e] *= corr;
#pragma unroll
            for (int u = 0; u < kRowsPerStep; ++u) {
                const float p = exp2f(s[u] - mx);
                lsum += p;
                if (base + u < r1) {
#pragma unroll
                    for (int e = 0; e < V; ++e) o[g][e] = fmaf(p, Vec<V>::get(vr[u], e), o[g][e]);
                }
            }
            l[g] = lsum;
            m[g] = mx;
        }
    }

    // Merge the warps' states.
#pragma unroll
    for (int g = 0; g < kMaxHeadsPerPass; ++g) {
        if (g >= ng) continue;
        if (lane == 0) {
            sm_m[warp][g] = m[g];
            sm_l[warp][g] = l[g];
        }
#pragma unroll
        for (int e = 0; e < V; ++e) sm_o[warp][g][lane * V + e] = o[g][e];
    }
    __syncthreads();
    for (int t = threadIdx.x; t < ng * D; t += kDecodeThreads) {
        const int g = t / D, d = t % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sm_m[w][g]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            const float f = exp2f(sm_m[w][g] - M);  // warps without rows: m = -inf -> 0
            L = fmaf(sm_l[w][g], f, L);
            O = fmaf(sm_o[w][g][d], f, O);
        }
        const size_t pidx = (size_t)(h0 + g) * n_splits + split;
        part_o[pidx * D + d] = O;
        if (d == 0) {
            part_ml[pidx * 2 + 0] = M;
            part_ml[pidx * 2 + 1] = L;
        }
    }
}

// Combine kernel.  grid = (num_heads, D / 32), block = 256: lane = element of
// the 32-wide slice, warps stride over the splits.
template <int D>
__global__ void __launch_bounds__(kDecodeThreads)
decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                      const float* __restrict__ v_cache, float* __restrict__ out,
                      uint32_t heads_per_kv, uint32_t max_seq, uint32_t window_start,
                      uint32_t n_splits) {
    __shared__ float red_m[kDecodeWarps];
    __shared__ float red_l[kDecodeWarps];
    __shared__ float red_o[kDecodeWarps][32];
    __shared__ float s_mask_v[kDecodeWarps][32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t h = blockIdx.x;
    const uint32_t d = blockIdx.y * 32 + lane;
    const float* pml = part_ml + (size_t)h * n_splits * 2;
    const float* po = part_o + (size_t)h * n_splits * D;

    float mloc = -CUDART_INF_F;
    for (uint32_t c = warp; c < n_splits; c += kDecodeWarps) mloc = fmaxf(mloc, pml[2 * c]);
    if (lane == 0) red_m[warp] = mloc;
    __syncthreads();
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, red_m[w]);

    float L = 0.f, O = 0.f;
    for (uint32_t c = warp; c < n_splits; c += kDecodeWarps) {
        const float f = exp2f(pml[2 * c] - M);
        L = fmaf(pml[2 * c + 1], f, L);
        O = fmaf(po[(size_t)c * D + d], f, O);
    }
    if (lane == 0) red_l[warp] = L;
    red_o[warp][lane] = O;

    // Masked positions s < window_start carry the score -1e4 (log2 units:
    // -1e4 * log2 e).  Their weight relative to the live maximum is usually
    // exactly zero in fp32; only otherwise are their V rows read.
    const float mask_l2 = kMaskScore * kLog2e;
    const bool need_mask = window_start > 0 && !(M >= mask_l2 + 150.f);
    float vsum = 0.f;
    if (need_mask) {
        const uint32_t kvh = h / heads_per_kv;
        const float* vb = v_cache + (size_t)kvh * max_seq * D + d;
        for (uint32_t s = warp; s < window_start; s += kDecodeWarps) vsum += vb[(size_t)s * D];
    }
    s_mask_v[warp][lane] = vsum;
    __syncthreads();
    if (warp == 0) {
        float Lt = 0.f, Ot = 0.f, Vm = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            Lt += red_l[w];
            Ot += red_o[w][lane];
            Vm += s_mask_v[w][lane];
        }
        if (need_mask) {
            const float Mt = fmaxf(M, mask_l2);
            const float fl = exp2f(M - Mt), fm = exp2f(mask_l2 - Mt);
            Lt = Lt * fl + (float)window_start * fm;
            Ot = Ot * fl + Vm * fm;
        }
        out[(size_t)h * D + d] = Ot / Lt;
    }
}

__global__ void kv_append_kernel(const float4* __restrict__ k_src, const float4* __restrict__ v_src,
                                 float4* __restrict__ k_cache, float4* __restrict__ v_cache,
                                 uint32_t kv_heads, uint32_t d4, uint32_t max_seq,
                                 uint32_t position) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= kv_heads * d4) return;
    const uint32_t g = i / d4, e = i % d4;
    const size_t dst = ((size_t)g * max_seq + position) * d4 + e;
    k_cache[dst] = k_src[i];
    if (v_cache) v_cache[dst] = v_src[i];
}

template <int D>
cudaError_t launch_decode_d(const float* q, const float* k_cache, const float* v_cache,
                            float* out, uint32_t num_heads, uint32_t kv_heads, uint32_t max_seq,
                            uint32_t total_seq, const DecodePlan& plan, float scale,
                            float* part_o, float* part_ml, cudaStream_t stream) {
    const uint32_t G = num_heads / kv_heads;
    dim3 g1(plan.n_splits, kv_heads, plan.n_hgroups);
    decode_split_kernel<D><<<g1, kDecodeThreads, 0, stream>>>(
        q, k_cache, v_cache, part_o, part_ml, G, max_seq, plan.window_start, total_seq,
        plan.chunk, plan.n_splits, scale * kLog2e);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2(num_heads, D / 32);
    decode_combine_kernel<D><<<g2, kDecodeThreads, 0, stream>>>(
        part_o, part_ml, v_cache, out, G, max_seq, plan.window_start, plan.n_splits);
    return cudaGetLastError();
}

}  // namespace

DecodePlan make_decode_plan(uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                            uint32_t total_seq, uint32_t window, int sm_count) {
    DecodePlan p{};
    p.window_start = (window > 0 && total_seq > window) ? total_seq - window : 0;
    p.rows_live = total_seq - p.window_start;
    const uint32_t G = kv_heads ? num_heads / kv_heads : 1;
    p.n_hgroups = (G + kMaxHeadsPerPass - 1) / kMaxHeadsPerPass;
    const uint32_t step = kDecodeWarps * kRowsPerStep;  // rows of one CTA-wide step
    const uint32_t target_ctas = 2u * (uint32_t)std::max(sm_count, 1);
    const uint32_t per_head = std::max(1u, target_ctas / std::max(1u, kv_heads * p.n_hgroups));
    uint32_t chunk = (p.rows_live + per_head - 1) / per_head;
    chunk = std::max(step, (chunk + step - 1) / step * step);
    p.chunk = chunk;
    p.n_splits = p.rows_live ? (p.rows_live + chunk - 1) / chunk : 0;
    p.part_o_floats = (size_t)num_heads * p.n_splits * head_dim;
    p.part_ml_floats = (size_t)num_heads * p.n_splits * 2;
    const size_t a = (p.part_o_floats * 4 + 255) / 256 * 256;
    p.workspace_bytes = a + (p.part_ml_floats * 4 + 255) / 256 * 256;
    return p;
}

cudaError_t launch_decode(const float* q, const float* k_cache, const float* v_cache,
                          float* out, uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                          uint32_t max_seq, uint32_t total_seq, const DecodePlan& plan,
                          float scale, float* part_o, float* part_ml, cudaStream_t stream) {
    switch (head_dim) {
        case 32:
            return launch_decode_d<32>(q, k_cache, v_cache, out, num_heads, kv_heads, max_seq,
                                       total_seq, plan, scale, part_o, part_ml, stream);
        case 64:
            return launch_decode_d<64>(q, k_cache, v_cache, out, num_heads, kv_heads, max_seq,
                                       total_seq, plan, scale, part_o, part_ml, stream);
        case 128:
            return launch_decode_d<128>(q, k_cache, v_cache, out, num_heads, kv_heads, max_seq,
                                        total_seq, plan, scale, part_o, part_ml, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_kv_append(const float* k_src, const float* v_src, float* k_cache,
                             float* v_cache, uint32_t kv_heads, uint32_t head_dim,
                             uint32_t max_seq, uint32_t position, cudaStream_t stream) {
    const uint32_t d4 = head_dim / 4;
    const uint32_t n = kv_heads * d4;
    const uint32_t threads = 256, blocks = (n + threads - 1) / threads;
    kv_append_kernel<<<blocks, threads, 0, stream>>>(
        reinterpret_cast<const float4*>(k_src), reinterpret_cast<const float4*>(v_src),
        reinterpret_cast<float4*>(k_cache), reinterpret_cast<float4*>(v_cache), kv_heads, d4,
        max_seq, position);
    return cudaGetLastError();
}

}  // namespace attn

// ---------------------------------------------------------------------------
// attn_decode_noalloc: decode with a fixed, library-owned scratch buffer.
//
// Some callers cannot hand this library a workspace and must not see it call
// cudaMalloc: an engine that has already carved all of device memory into
// its own pools (a KV-cache pool that owns every free byte), a plugin
// interface that passes only input and output pointers, or a latency-bound
// loop that forbids allocation and the implicit synchronisation it can bring.
// For them the split partials live in one file-scope device array of
// kNoAllocScratchBytes.  Every GPU that loads this library keeps that array
// resident until the process exits.  The array is shared by every call on a
// device and keeps the last call's contents; the decode kernels overwrite
// every partial they later read, so nothing in it has to start at zero.  Two
// calls that overlap on the GPU (different streams, or graphs replayed
// concurrently) race on the array and corrupt each other's results.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[kNoAllocScratchBytes];
}  // namespace

namespace attn {
// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static cudaError_t noalloc_scratch_address(void** out) {
    static void* addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}
}  // namespace attn

extern "C" attn_status_t attn_decode_noalloc(const float* q, const float* k_cache,
                                             const float* v_cache, float* out,
                                             uint32_t num_heads, uint32_t kv_heads,
                                             uint32_t head_dim, uint32_t max_seq,
                                             uint32_t total_seq, uint32_t window, float scale,
                                             void* stream) {
    const size_t need = attn_decode_workspace_size(num_heads, kv_heads, head_dim, total_seq, window);
    if (need > kNoAllocScratchBytes) {
        char msg[160];
        std::snprintf(msg, sizeof(msg),
                      "attn_decode_noalloc: these sizes need %zu bytes of scratch, more than the "
                      "fixed %zu-byte buffer",
                      need, kNoAllocScratchBytes);
        attn::set_last_error(msg);
        return ATTN_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    const cudaError_t e = attn::noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return attn::record_cuda_error(e);
    return attn_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim, max_seq,
                       total_seq, window, scale, scratch, kNoAllocScratchBytes, stream);
}
