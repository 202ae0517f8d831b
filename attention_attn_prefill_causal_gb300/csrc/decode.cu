// decode.cu -- single-query grouped-query decode attention against a
// [kv_heads, max_seq, head_dim] K/V cache, the K/V cache append, and the
// fused (RoPE +) append + decode.
//
// Operation ("soft3/glia/run/backend/honeycrisp/kernels/attention.rs",
// module doc and decode kernel `kmain`): for query head h with KV head
// g = h / (num_heads / kv_heads), score_s = scale * q[h].K[g,s] for
// s < total_seq, replaced by -1e4 below window_start; out[h] is the
// softmax-weighted sum of V[g,s].  The fused form follows the page's
// FUSED_ROPE_KV_ATTN_TEMPLATE: rotate k_new (rotate-half pairs (d, d+D/2)
// with per-pair cos/sin tables) into k_cache[g, position], copy v_new into
// v_cache[g, position], rotate q, then decode.
//
// GB300 design.  The page walks the whole sequence with one 32-lane group
// per head; a 4096-row cache is then a few microseconds of work for a
// handful of SMs.  Here one launch covers every SM:
//  * CTA = (sequence chunk, KV head, group of GP in {1,2,4,6,8} query
//    heads), eight warps, each warp a contiguous run of rows.  Each K/V row
//    is read from HBM once for every query head of its GQA group, with
//    128-bit loads issued before any arithmetic (lane l holds elements
//    [l*V, l*V+V)).
//  * A warp takes 4 rows per step, i.e. 4*GP (row, head) dot products.  Each
//    lane forms its partial sums of all of them, and a reduce-scatter over
//    the warp (at most 31 shuffles) leaves lane j holding the full score of
//    pair j, ordered head-major (j = 4 * head + row) so that a head's four
//    rows sit in adjacent lanes.  The online softmax (base 2) then costs one
//    exponential per lane; the weights reach every lane through shared
//    memory, as (p, p) pairs for the packed P.V update of the lane's slice of
//    head_dim.  The next step's keys are fetched as soon as the dot products
//    are formed, its values after the P.V update.
//  * The warps' states merge in shared memory and each CTA writes one
//    partial (max, sum, unnormalised output) per query head to the
//    workspace; with a single chunk per KV head the CTA writes the
//    normalised output itself.
//  * A combine kernel, launched as a programmatic dependent of the decode
//    kernel (its launch overlaps the decode grid; it waits on that grid's
//    completion in hardware), merges the partials of each query head with a
//    log-sum-exp and normalises.
//  * Consecutive calls overlap: each decode launch is a programmatic
//    dependent of the kernel before it on the stream, and its CTAs prefetch
//    their first step's K/V rows into L2 while that kernel drains, then wait
//    for it before reading anything.  A warp that walks more than one step
//    keeps a bulk L2 prefetch one step ahead of its register loads (the ROLL
//    build); prefetching a whole long range at once would overfill L2.
//  * q, k_new, v_new, the RoPE tables and out are read and written with
//    plain loads and stores, so they may also sit in page-locked host memory
//    (read over the CPU-GPU link inside the call).
//  * Positions below window_start are never read; their score is -1e4
//    exactly as on the page, and the final merge adds their weight
//    exp(-1e4 - max) back.  That weight is zero in fp32 unless every live
//    score is below about -9896, in which case the final merge reads the
//    masked V rows and adds them exactly.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

// Launch shape (compile-time so that variants can be built and compared).
#ifndef ATTN_DECODE_WARPS
#define ATTN_DECODE_WARPS 8
#endif
#ifndef ATTN_DECODE_WARPS_PER_SM
#define ATTN_DECODE_WARPS_PER_SM 16
#endif
constexpr int kWarps = ATTN_DECODE_WARPS;                 // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kWarpsPerSm = ATTN_DECODE_WARPS_PER_SM;     // occupancy the plan aims for
constexpr int kMinBlocks = kWarpsPerSm / kWarps > 0 ? kWarpsPerSm / kWarps : 1;
constexpr int kRowsPerStep = 4;  // K/V rows a warp holds per step
// L2 prefetch lead: a warp asks L2 for the K/V rows this many rows ahead of
// the step it computes (one bulk prefetch per step, no registers or shared
// memory).  Measured on long caches: one step ahead streams at the copy
// rate; leads of 8 rows and more lose 5-40%, and an unbounded prefetch of
// the whole range (more than L2 holds) evicts rows before they are read.
#ifndef ATTN_DECODE_PREFETCH_LEAD
#define ATTN_DECODE_PREFETCH_LEAD 4
#endif
constexpr uint32_t kPrefetchLead = ATTN_DECODE_PREFETCH_LEAD;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaskScore = -1.0e4f;  // the page's replaced score
constexpr uint32_t kNoRow = 0xffffffffu;

struct DecodeArgs {
    const float* q;
    const float* k_cache;
    const float* v_cache;
    float* k_cache_w;        // append target (fused call only)
    float* v_cache_w;
    const float* k_new;      // [kv_heads, D] (fused call only)
    const float* v_new;
    const float* rope_cos;   // [D/2] or null
    const float* rope_sin;
    float* out;              // [num_heads, D]
    float* part_o;           // [num_heads, n_splits, D]
    float* part_ml;          // [num_heads, n_splits, 2]
    uint32_t heads_per_kv;
    uint32_t n_hgroups;
    uint32_t max_seq;
    uint32_t window_start;
    uint32_t total_seq;
    uint32_t chunk;          // live rows per CTA
    uint32_t rows_per_warp;  // ceil(chunk / kWarps)
    uint32_t n_splits;
    uint32_t position;       // appended row, or kNoRow
    float scale_log2;
};

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned start, size a
// multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int V>
__device__ __forceinline__ void load_slice(float (&x)[V], const float* p) {
    if constexpr (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (V == 2) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = *p;
    }
}

// Streaming (evict-first) load of a cache slice: each K/V byte is used once.
template <int V>
__device__ __forceinline__ void load_slice_stream(float (&x)[V], const float* p) {
    if constexpr (V == 4) {
        const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (V == 2) {
        const float2 t = __ldcs(reinterpret_cast<const float2*>(p));
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = __ldcs(p);
    }
}

template <int V>
__device__ __forceinline__ void store_slice(float* p, const float (&x)[V]) {
    if constexpr (V == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (V == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    } else {
        *p = x[0];
    }
}

// Rotate-half RoPE on the lane's slice: element d pairs with d +- D/2, which
// sits in lane l ^ 16 at the same slot.
template <int V>
__device__ __forceinline__ void rope_slice(float (&x)[V], const float* cosv, const float* sinv,
                                           int lane) {
    constexpr int kHalfLanes = 16;
    float partner[V];
#pragma unroll
    for (int e = 0; e < V; ++e) partner[e] = __shfl_xor_sync(0xffffffffu, x[e], kHalfLanes);
    const bool low = lane < kHalfLanes;
    const int base = (low ? lane : lane - kHalfLanes) * V;
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const float c = cosv[base + e], s = sinv[base + e];
        x[e] = low ? (x[e] * c - partner[e] * s) : (partner[e] * s + x[e] * c);
    }
}

// Reduce-scatter of NV values (NV a power of two, 4..32) over the 32 lanes of
// a warp: on return v[0] of lane l holds the warp-wide sum of value
// l & (NV - 1).  Lane bits above NV first exchange every value (butterfly);
// then each stage with offset o keeps the half of the remaining values
// selected by lane bit o and adds the partner's copy of that half.
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
    static_assert(NV >= 4 && NV <= 32 && (NV & (NV - 1)) == 0, "NV must be a power of two");
#pragma unroll
    for (int o = 16; o >= NV; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
#pragma unroll
    for (int o = NV / 2; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float keep = upper ? v[i + o] : v[i];
            const float send = upper ? v[i] : v[i + o];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Merged (max, sum, output) of one (head, element), plus the positions below
// window_start whose score is -1e4; returns the normalised output.  A row
// appended by this call (position, value vnew) is taken from vnew, not from
// the cache it is being written to.
__device__ __forceinline__ float finish(float M, float L, float O, uint32_t window_start,
                                        const float* vcol, uint32_t D, uint32_t position,
                                        float vnew) {
    const float mask_l2 = kMaskScore * kLog2e;
    if (window_start > 0 && !(M >= mask_l2 + 150.f)) {
        float vs = 0.f;
        for (uint32_t s = 0; s < window_start; ++s)
            vs += (s == position) ? vnew : vcol[(size_t)s * D];
        const float Mt = fmaxf(M, mask_l2);
        const float fl = exp2f(M - Mt), fm = exp2f(mask_l2 - Mt);
        L = L * fl + (float)window_start * fm;
        O = O * fl + vs * fm;
    }
    return O / L;
}

// ROLL: keep the L2 prefetch running ahead inside the step loop.  Launched
// only when a warp walks more than kPrefetchLead rows: the extra code costs
// the 128-register builds a spill, which a one-step walk should not pay.
template <int D, int GP, bool ROLL>
__global__ void __launch_bounds__(kThreads, kMinBlocks) decode_kernel(const DecodeArgs a) {
    constexpr int V = D / 32;    // elements of a row per lane
    constexpr int U = kRowsPerStep;
    constexpr int NV = U * GP;   // (row, head) pairs per warp step, head-major: j = g * U + u
    constexpr int NR = (NV & (NV - 1)) == 0 ? NV : 32;  // reduced width (a power of two)
    // Scaled (and rotated) queries.  With GP >= 2 they are stored head-pair
    // interleaved, sq[g/2][d][g%2], so one 64-bit read gives element d of two
    // heads for a packed (fp32x2) multiply-add.
    __shared__ __align__(16) float sq[GP * D];
    __shared__ __align__(16) float2 pbuf[kWarps][32];  // (p, p) per pair
    __shared__ __align__(16) float2 cbuf[kWarps][GP];  // (corr, corr) per head
    __shared__ float wm[kWarps][GP], wl[kWarps][GP];
    __shared__ __align__(16) float wo[kWarps][GP][D];
    __shared__ __align__(16) float s_knew[D], s_vnew[D];  // the appended row (fused call)

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t split = blockIdx.x;
    const uint32_t kvh = blockIdx.y / a.n_hgroups, hg = blockIdx.y % a.n_hgroups;
    const int ng = (int)min((uint32_t)GP, a.heads_per_kv - hg * GP);
    const uint32_t h0 = kvh * a.heads_per_kv + hg * GP;
    const uint32_t chunk = a.chunk;
    const uint32_t c0 = a.window_start + split * chunk;
    const uint32_t c1 = min(c0 + chunk, a.total_seq);
    const uint32_t r0 = min(c0 + warp * a.rows_per_warp, c1);  // this warp's rows
    const uint32_t r1 = min(r0 + a.rows_per_warp, c1);
    const bool has_new = a.position != kNoRow;
    const size_t kv_base = (size_t)kvh * a.max_seq * D;

    // The launch is a programmatic dependent of the previous kernel on the
    // stream, so this CTA may start while that kernel drains.  Until the
    // grid dependency resolves it only warms L2 with its first K/V rows (a bulk
    // prefetch reads memory without using it, and L2 is coherent, so a row
    // written by the previous kernel is still read fresh below); every read
    // of data and every write waits for the previous kernel's completion.
    if (lane == 0 && r1 > r0 && kPrefetchLead > 0) {
        const uint32_t bytes = min(r1 - r0, kPrefetchLead) * (uint32_t)D * 4u;
        bulk_prefetch_l2(a.k_cache + kv_base + (size_t)r0 * D, bytes);
        bulk_prefetch_l2(a.v_cache + kv_base + (size_t)r0 * D, bytes);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Issue the first step's K/V loads before anything else.
    float kx[U][V], vx[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t row = r0 + u;
#pragma unroll
        for (int e = 0; e < V; ++e) kx[u][e] = vx[u][e] = 0.f;  // rows past r1 stay finite
        if (row < r1) {
            load_slice_stream<V>(kx[u], a.k_cache + kv_base + (size_t)row * D + lane * V);
            load_slice_stream<V>(vx[u], a.v_cache + kv_base + (size_t)row * D + lane * V);
        }
    }

    // The appended row: written once per KV head (split 0, first head group)
    // and substituted from k_new / v_new wherever it is read in this call.
    const bool own_new = has_new && a.position >= r0 && a.position < r1;
    if (has_new && warp == kWarps - 1) {
        float knew[V], vnew[V];
        load_slice<V>(knew, a.k_new + (size_t)kvh * D + lane * V);
        load_slice<V>(vnew, a.v_new + (size_t)kvh * D + lane * V);
        if (a.rope_cos) rope_slice<V>(knew, a.rope_cos, a.rope_sin, lane);
        store_slice<V>(&s_knew[lane * V], knew);
        store_slice<V>(&s_vnew[lane * V], vnew);
        if (split == 0 && hg == 0) {
            const size_t dst = kv_base + (size_t)a.position * D + lane * V;
            store_slice<V>(a.k_cache_w + dst, knew);
            store_slice<V>(a.v_cache_w + dst, vnew);
        }
    }

    for (int g = warp; g < GP; g += kWarps) {
        float qv[V];
        if (g < ng) {
            load_slice<V>(qv, a.q + (size_t)(h0 + g) * D + lane * V);
            if (a.rope_cos) rope_slice<V>(qv, a.rope_cos, a.rope_sin, lane);
#pragma unroll
            for (int e = 0; e < V; ++e) qv[e] *= a.scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) qv[e] = 0.f;
        }
        if constexpr (GP >= 2) {
#pragma unroll
            for (int e = 0; e < V; ++e)
                sq[((g / 2) * D + lane * V + e) * 2 + (g % 2)] = qv[e];
        } else {
            store_slice<V>(&sq[lane * V], qv);
        }
    }
    __syncthreads();

    // Lane l owns the score of pair j = l (head g = j / U, row u = j % U) when
    // l < NV; the U lanes of a head hold its running max and sum.
    const int my_u = lane % U, my_g = lane / U;
    const bool my_live_head = lane < NV && my_g < ng;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    float o[GP][V];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) o[g][e] = 0.f;

    for (uint32_t base = r0; base < r1; base += U) {
        // Keep the L2 prefetch kPrefetchLead rows ahead of this step.
        if (ROLL && base + kPrefetchLead < r1) {
            if (lane == 0) {
                const uint32_t pf = base + kPrefetchLead;
                const uint32_t bytes = min(r1 - pf, (uint32_t)U) * (uint32_t)D * 4u;
                bulk_prefetch_l2(a.k_cache + kv_base + (size_t)pf * D, bytes);
                bulk_prefetch_l2(a.v_cache + kv_base + (size_t)pf * D, bytes);
            }
            __syncwarp();
        }
        if (own_new) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (base + u == a.position) {
                    load_slice<V>(kx[u], &s_knew[lane * V]);
                    load_slice<V>(vx[u], &s_vnew[lane * V]);
                }
        }
        // ---- scores: partial dot products of the lane's slice
        float part[NV];
        if constexpr (GP >= 2) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float2 kd[V];  // (k, k): one key element against two heads
#pragma unroll
                for (int e = 0; e < V; ++e) kd[e] = make_float2(kx[u][e], kx[u][e]);
#pragma unroll
                for (int hp = 0; hp < GP / 2; ++hp) {
                    float2 acc = make_float2(0.f, 0.f);
                    {
                        const float2* qp = reinterpret_cast<const float2*>(sq) + hp * D + lane * V;
#pragma unroll
                        for (int e = 0; e < V; ++e) acc = __ffma2_rn(qp[e], kd[e], acc);
                    }
                    part[(2 * hp) * U + u] = acc.x;
                    part[(2 * hp + 1) * U + u] = acc.y;
                }
            }
        } else {
            float qv[V];
            load_slice<V>(qv, &sq[lane * V]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < V; ++e) d = fmaf(qv[e], kx[u][e], d);
                part[u] = d;
            }
        }
        // GP = 6 gives 24 pairs: reduce them as 32 with zeros in the tail.
        float red[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) red[i] = i < NV ? part[i] : 0.f;
        float s = reduce_scatter<NR>(red, lane);
        // The keys of this step are consumed: fetch the next step's keys now.
        const uint32_t nb = base + U;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (nb + u < r1)
                load_slice_stream<V>(kx[u], a.k_cache + kv_base + (size_t)(nb + u) * D + lane * V);

        // ---- online softmax: one exponential per lane
        if (base + my_u >= r1 || !my_live_head) s = -CUDART_INF_F;
        float mx = s;
#pragma unroll
        for (int off = 1; off < U; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m_run, mx);
        const bool any = m_new != -CUDART_INF_F;
        const float corr = any ? ex2(m_run - m_new) : 1.f;
        const float p = any ? ex2(s - m_new) : 0.f;
        float psum = p;
#pragma unroll
        for (int off = 1; off < U; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_run = l_run * corr + psum;
        m_run = m_new;
        if (lane < NV) pbuf[warp][lane] = make_float2(p, p);
        if (lane < NV && my_u == 0) cbuf[warp][my_g] = make_float2(corr, corr);
        __syncwarp();

        // ---- O = O * corr + P V on the lane's slice (packed pairs of elements)
        if constexpr (V >= 2) {
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float2 c2 = cbuf[warp][g];
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    const float2 r = __fmul2_rn(make_float2(o[g][e], o[g][e + 1]), c2);
                    o[g][e] = r.x;
                    o[g][e + 1] = r.y;
                }
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float2 pd = pbuf[warp][g * U + u];
#pragma unroll
                    for (int e = 0; e < V; e += 2) {
                        const float2 r = __ffma2_rn(pd, make_float2(vx[u][e], vx[u][e + 1]),
                                                    make_float2(o[g][e], o[g][e + 1]));
                        o[g][e] = r.x;
                        o[g][e + 1] = r.y;
                    }
                }
            }
        } else {
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float c = cbuf[warp][g].x;
                o[g][0] *= c;
#pragma unroll
                for (int u = 0; u < U; ++u) o[g][0] = fmaf(pbuf[warp][g * U + u].x, vx[u][0], o[g][0]);
            }
        }
        __syncwarp();  // pbuf / cbuf are rewritten by the next step
        // The values of this step are consumed: fetch the next step's values.
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (nb + u < r1)
                load_slice_stream<V>(vx[u], a.v_cache + kv_base + (size_t)(nb + u) * D + lane * V);
    }

    // ----------------------------------------------------------- merge the warps
    if (lane < NV && my_u == 0) {
        wm[warp][my_g] = m_run;
        wl[warp][my_g] = l_run;
    }
#pragma unroll
    for (int g = 0; g < GP; ++g) store_slice<V>(&wo[warp][g][lane * V], o[g]);
    __syncthreads();
    // The combine kernel may start launching now; it waits for this whole grid.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // one thread per (head, 4 elements): this CTA's partial (max, sum, output)
    for (int t = threadIdx.x; t < ng * (D / 4); t += kThreads) {
        const int g = t / (D / 4), d = (t % (D / 4)) * 4;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][g]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = ex2(wm[w][g] - M);
                const float4 x = *reinterpret_cast<const float4*>(&wo[w][g][d]);
                L = fmaf(wl[w][g], f, L);
                O.x = fmaf(x.x, f, O.x);
                O.y = fmaf(x.y, f, O.y);
                O.z = fmaf(x.z, f, O.z);
                O.w = fmaf(x.w, f, O.w);
            }
        }
        const uint32_t h = h0 + g;
        if (a.n_splits == 1) {
            // A single chunk holds every live row: normalise here, no combine.
            const float* vcol = a.v_cache + kv_base + d;
            const float* vn = has_new ? a.v_new + (size_t)kvh * D + d : nullptr;
            float r[4] = {O.x, O.y, O.z, O.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                a.out[(size_t)h * D + d + e] =
                    finish(M, L, r[e], a.window_start, vcol + e, D, a.position, vn ? vn[e] : 0.f);
        } else {
            const size_t pidx = (size_t)h * a.n_splits + split;
            *reinterpret_cast<float4*>(&a.part_o[pidx * D + d]) = O;
            if (d == 0) *reinterpret_cast<float2*>(&a.part_ml[2 * pidx]) = make_float2(M, L);
        }
    }
}

struct CombineArgs {
    const float* part_o;
    const float* part_ml;
    const float* v_cache;
    const float* v_new;
    float* out;
    uint32_t heads_per_kv;
    uint32_t max_seq;
    uint32_t window_start;
    uint32_t n_splits;
    uint32_t position;
};

// Combine kernel: one CTA per (query head, 32 elements of head_dim); lane =
// element, warp w takes the partials w, w + 16, ... in batches whose loads
// are all issued before they are used (one round trip for up to 256).  Launched as a programmatic dependent of
// the decode kernel: it starts early and waits for that grid's results.
template <int D>
__global__ void __launch_bounds__(512) decode_combine_kernel(const CombineArgs a) {
    constexpr int kCW = 16;     // warps
    constexpr int kBatch = 16;  // partials per warp per batch (256 per round trip)
    __shared__ float sm_m[kCW], sm_l[kCW];
    __shared__ float sm_o[kCW][32];
    // The next call's decode kernel may start now (it only prefetches until
    // this grid completes).
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t h = blockIdx.x;
    const uint32_t d = blockIdx.y * 32 + lane;
    const float* pml = a.part_ml + (size_t)h * a.n_splits * 2;
    const float* po = a.part_o + (size_t)h * a.n_splits * D + d;
    float M = -CUDART_INF_F, L = 0.f, O = 0.f;
    for (uint32_t c0 = warp; c0 < a.n_splits; c0 += kCW * kBatch) {
        float pm[kBatch], pl[kBatch], pv[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t c = c0 + i * kCW;
            const bool ok = c < a.n_splits;
            const float2 ml = ok ? __ldcg(reinterpret_cast<const float2*>(pml) + c)
                                 : make_float2(-CUDART_INF_F, 0.f);
            pm[i] = ml.x;
            pl[i] = ml.y;
            pv[i] = ok ? __ldcg(po + (size_t)c * D) : 0.f;
        }
        float Mb = M;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) Mb = fmaxf(Mb, pm[i]);
        if (Mb == -CUDART_INF_F) continue;
        const float fo = ex2(M - Mb);  // M = -inf -> 0
        L *= fo;
        O *= fo;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const float f = ex2(pm[i] - Mb);
            L = fmaf(pl[i], f, L);
            O = fmaf(pv[i], f, O);
        }
        M = Mb;
    }
    if (lane == 0) {
        sm_m[warp] = M;
        sm_l[warp] = L;
    }
    sm_o[warp][lane] = O;
    __syncthreads();
    if (warp == 0) {
        float Mt = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kCW; ++w) Mt = fmaxf(Mt, sm_m[w]);
        float Lt = 0.f, Ot = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) {
            const float f = sm_m[w] == -CUDART_INF_F ? 0.f : ex2(sm_m[w] - Mt);
            Lt = fmaf(sm_l[w], f, Lt);
            Ot = fmaf(sm_o[w][lane], f, Ot);
        }
        const uint32_t kvh = h / a.heads_per_kv;
        const float* vcol = a.v_cache + (size_t)kvh * a.max_seq * D + d;
        const float vn = a.v_new ? a.v_new[(size_t)kvh * D + d] : 0.f;
        a.out[(size_t)h * D + d] = finish(Mt, Lt, Ot, a.window_start, vcol, D, a.position, vn);
    }
}

// Copies a decode step's small inputs (q, k_new, v_new: float4 counts n_q,
// n_kv, n_kv; the RoPE tables: n_half floats each, read as floats since the
// caller's tables need only 4-byte alignment) into the workspace, when
// some of them sit in page-locked host memory: one CTA reads them over the
// host link once, and the decode CTAs then read the copies from HBM.  A
// programmatic dependent of the kernel before it; the decode kernel is one of
// it (it may start its L2 prefetch of the cache at once and waits for this
// grid before reading any input).
__global__ void __launch_bounds__(512) stage_step_inputs_kernel(
    const float4* __restrict__ q, const float4* __restrict__ k_new,
    const float4* __restrict__ v_new, const float* __restrict__ rope_cos,
    const float* __restrict__ rope_sin, float4* __restrict__ dst, uint32_t n_q, uint32_t n_kv,
    uint32_t n_half) {
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // One flat index over q, k_new, v_new (float4s): every load of a thread is
    // issued before any store, so the copy costs one host-link round trip
    // for up to 4 x 512 float4s (32 KB).
    const uint32_t n_kv_all = k_new ? n_kv : 0u;
    const uint32_t total = n_q + 2 * n_kv_all;
    constexpr int kPer = 4;
    float4 x[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const uint32_t i = threadIdx.x + u * blockDim.x;
        if (i < n_q) x[u] = q[i];
        else if (i < n_q + n_kv_all) x[u] = k_new[i - n_q];
        else if (i < total) x[u] = v_new[i - n_q - n_kv_all];
    }
    float cs = 0.f, sn = 0.f;
    const bool rope_here = rope_cos && threadIdx.x < n_half;
    if (rope_here) {
        cs = rope_cos[threadIdx.x];
        sn = rope_sin[threadIdx.x];
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const uint32_t i = threadIdx.x + u * blockDim.x;
        if (i < total) dst[i] = x[u];
    }
    // the rest, should the inputs exceed one pass (more than 32 KB)
    for (uint32_t i = threadIdx.x + kPer * blockDim.x; i < total; i += blockDim.x) {
        if (i < n_q) dst[i] = q[i];
        else if (i < n_q + n_kv_all) dst[i] = k_new[i - n_q];
        else dst[i] = v_new[i - n_q - n_kv_all];
    }
    float* dc = reinterpret_cast<float*>(dst + n_q + 2 * n_kv);
    if (rope_here) {
        dc[threadIdx.x] = cs;
        dc[n_half + threadIdx.x] = sn;
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

template <int D, int GP>
cudaError_t launch_gp(const DecodeArgs& a, const DecodePlan& plan, uint32_t kv_heads,
                      uint32_t num_heads, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t dcfg = {};
    dcfg.gridDim = dim3(plan.n_splits, kv_heads * plan.n_hgroups, 1);
    dcfg.blockDim = dim3(kThreads, 1, 1);
    dcfg.stream = stream;
    dcfg.attrs = attr;
    dcfg.numAttrs = 1;
    const bool roll = kPrefetchLead > 0 && plan.rows_per_warp > kPrefetchLead;
    cudaError_t e = cudaLaunchKernelEx(&dcfg, roll ? decode_kernel<D, GP, true>
                                                   : decode_kernel<D, GP, false>, a);
    if (e != cudaSuccess || plan.n_splits == 1) return e;
    CombineArgs c{};
    c.part_o = a.part_o;
    c.part_ml = a.part_ml;
    c.v_cache = a.v_cache;
    c.v_new = a.position != kNoRow ? a.v_new : nullptr;
    c.out = a.out;
    c.heads_per_kv = a.heads_per_kv;
    c.max_seq = a.max_seq;
    c.window_start = a.window_start;
    c.n_splits = a.n_splits;
    c.position = a.position;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_heads, D / 32, 1);
    cfg.blockDim = dim3(512, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, c);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const DecodePlan& plan, uint32_t kv_heads,
                     uint32_t num_heads, cudaStream_t stream) {
    switch (plan.heads_per_pass) {
        case 1: return launch_gp<D, 1>(a, plan, kv_heads, num_heads, stream);
        case 2: return launch_gp<D, 2>(a, plan, kv_heads, num_heads, stream);
        case 4: return launch_gp<D, 4>(a, plan, kv_heads, num_heads, stream);
        case 6: return launch_gp<D, 6>(a, plan, kv_heads, num_heads, stream);
        default: return launch_gp<D, 8>(a, plan, kv_heads, num_heads, stream);
    }
}

}  // namespace

DecodePlan make_decode_plan(uint32_t num_heads, uint32_t kv_heads, uint32_t head_dim,
                            uint32_t total_seq, uint32_t window, int sm_count) {
    DecodePlan p{};
    p.window_start = (window > 0 && total_seq > window) ? total_seq - window : 0;
    p.rows_live = total_seq - p.window_start;
    const uint32_t G = kv_heads ? num_heads / kv_heads : 1;
    // Query heads per CTA: the width in {1, 2, 4, 6, 8} with the fewest head
    // groups (each group reads the K/V rows again), then the fewest idle
    // head slots.
    p.heads_per_pass = 1;
    {
        uint32_t best_groups = ~0u, best_idle = ~0u;
        for (uint32_t w : {1u, 2u, 4u, 6u, 8u}) {
            const uint32_t groups = (G + w - 1) / w, idle = groups * w - G;
            if (groups < best_groups || (groups == best_groups && idle < best_idle)) {
                best_groups = groups;
                best_idle = idle;
                p.heads_per_pass = w;
            }
        }
    }
    p.n_hgroups = (G + p.heads_per_pass - 1) / p.heads_per_pass;
    // kWarpsPerSm / kWarps CTAs on every SM: split the live rows of every KV
    // head group into that many equal chunks (the last warp step of a warp
    // may be partial; its missing rows are masked).
    const uint32_t target_ctas =
        (uint32_t)kMinBlocks * (uint32_t)std::max(sm_count, 1);
    const uint32_t groups = std::max(1u, kv_heads * p.n_hgroups);
    const uint32_t ctas_per_group = std::max(1u, target_ctas / groups);
    const uint32_t chunk = std::max(1u, (p.rows_live + ctas_per_group - 1) / ctas_per_group);
    p.chunk = chunk;
    p.rows_per_warp = (chunk + kWarps - 1) / kWarps;
    p.n_splits = p.rows_live ? (p.rows_live + chunk - 1) / chunk : 0;
    p.part_o_floats = (size_t)num_heads * p.n_splits * head_dim;
    p.part_ml_floats = (size_t)num_heads * p.n_splits * 2;
    p.stage_floats = (size_t)(num_heads + 2 * kv_heads + 1) * head_dim;
    p.workspace_bytes = (p.part_o_floats * 4 + 255) / 256 * 256 +
                        (p.part_ml_floats * 4 + 255) / 256 * 256 +
                        (p.stage_floats * 4 + 255) / 256 * 256;
    return p;
}

cudaError_t launch_decode(const DecodeCall& c, const DecodePlan& plan, void* workspace,
                          cudaStream_t stream) {
    DecodeArgs a{};
    a.q = c.q;
    a.k_cache = c.k_cache;
    a.v_cache = c.v_cache;
    a.k_cache_w = c.k_cache_w;
    a.v_cache_w = c.v_cache_w;
    a.k_new = c.k_new;
    a.v_new = c.v_new;
    a.rope_cos = c.rope_cos;
    a.rope_sin = c.rope_sin;
    a.out = c.out;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + (plan.part_o_floats * 4 + 255) / 256 * 256);
    a.heads_per_kv = c.num_heads / c.kv_heads;
    a.n_hgroups = plan.n_hgroups;
    a.max_seq = c.max_seq;
    a.window_start = plan.window_start;
    a.total_seq = c.total_seq;
    a.chunk = plan.chunk;
    a.rows_per_warp = plan.rows_per_warp;
    a.n_splits = plan.n_splits;
    a.position = c.k_new ? c.position : kNoRow;
    a.scale_log2 = c.scale * kLog2e;
    if (c.stage_inputs) {
        // Stage the step inputs into the workspace (after the partials), then
        // point the decode at the copies.
        float* st = reinterpret_cast<float*>(ws + (plan.part_o_floats * 4 + 255) / 256 * 256 +
                                             (plan.part_ml_floats * 4 + 255) / 256 * 256);
        const uint32_t n_q = c.num_heads * c.head_dim / 4, n_kv = c.kv_heads * c.head_dim / 4;
        const uint32_t n_half = c.head_dim / 2;  // cos and sin: head_dim/2 floats each
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(512, 1, 1);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(
            &cfg, stage_step_inputs_kernel, reinterpret_cast<const float4*>(c.q),
            reinterpret_cast<const float4*>(c.k_new), reinterpret_cast<const float4*>(c.v_new),
            c.rope_cos, c.rope_sin, reinterpret_cast<float4*>(st), n_q, n_kv, n_half);
        if (e != cudaSuccess) return e;
        a.q = st;
        float* sk = st + (size_t)n_q * 4;
        float* sv = sk + (size_t)n_kv * 4;
        float* sc = sv + (size_t)n_kv * 4;
        if (c.k_new) {
            a.k_new = sk;
            a.v_new = sv;
        }
        if (c.rope_cos) {
            a.rope_cos = sc;
            a.rope_sin = sc + n_half;
        }
    }
    switch (c.head_dim) {
        case 32: return launch_d<32>(a, plan, c.kv_heads, c.num_heads, stream);
        case 64: return launch_d<64>(a, plan, c.kv_heads, c.num_heads, stream);
        case 128: return launch_d<128>(a, plan, c.kv_heads, c.num_heads, stream);
        default: return cudaErrorInvalidValue;
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
// For them the decode workspace (the per-chunk partial results, and copies
// of host-resident step inputs) lives in one
// file-scope device array of kNoAllocScratchBytes.  Every GPU that loads
// this library keeps that array resident until the process exits.  The array
// is shared by every call on a device and keeps the last call's contents;
// every partial a call reads was written earlier in that same call, so
// nothing in the array has to start at zero.  Two calls that overlap on the
// GPU (different streams, or graphs replayed concurrently) race on the array
// and corrupt each other's results.
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
    // The arguments are checked as attn_decode checks them before the
    // scratch size is: a malformed call reports INVALID_ARG whatever its sizes.
    const attn_status_t st = attn::check_decode_args(q, k_cache, v_cache, out, num_heads,
                                                     kv_heads, head_dim, max_seq, total_seq,
                                                     scale);
    if (st != ATTN_OK) return st;
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
