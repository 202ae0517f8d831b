// prefill_fp32.cu -- exact-mode causal grouped-query prefill on CUDA cores,
// fp32 throughout.
//
// Operation ("aprender-gpu 0.32.0 -- prefill_fused.rs", module doc,
// Algorithm 1-3): query head h reads KV head h / heads_per_kv; row i attends
// to keys j <= i with scores scale * Q[i].K[j], an online softmax (running
// max, correction, p = exp(s - max)), O = O * corr + p V[j], and O / l at the
// end.  Q/O rows use q_stride, K/V rows use kv_stride (packed layout).
//
// The page runs one warp per query head, walking all M rows serially and
// reading K/V through L2.  Here a CTA takes a block of query rows of one
// head (64, 32 or 16 rows: the largest size that still gives every SM
// several blocks) and walks 64-key tiles staged in shared memory, so each
// K/V row is read from global memory once per block instead of once per row:
//  * tiles arrive by asynchronous 16-byte copies (cp.async), K and V in
//    separate groups: the scores wait for K only, so V lands during them;
//  * a warp owns 8, 4 or 2 query rows and scores all of them at once, each
//    lane taking keys lane and lane + 32 of the tile (dot products over
//    head_dim from shared memory: two 128-bit K reads per lane feed every
//    row, the Q reads are broadcasts);
//  * per row, the tile's max and sum come from warp shuffles; the online
//    softmax runs in base 2 (scores pre-multiplied by log2 e, as the page
//    does before ex2);
//  * for PV each warp writes its weights to shared memory over the K tile
//    (free once every warp's dot products are done); each lane owns
//    head_dim/32 output elements and reads four keys' weights of a row with
//    one broadcast 128-bit load, stopping at the warp's last attended key.
// The grid runs heads fastest and query blocks longest causal extent first,
// so the longest walks of every head start in the first wave.
// Causal masking is the loop bound plus a per-key test on the diagonal tile.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kBN = 64;           // keys per tile
constexpr int kThreads = 256;     // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int kBM>
struct Smem {
    static constexpr int kPitch = D + 4;  // pad: 128-bit reads across rows hit distinct banks
    // The weights of a tile ([kBM][kBN] floats) are staged over the K tile
    // once every warp's dot products are done, when they fit there; else
    // (head_dim 32 with 64-row blocks) in an array of their own.
    static constexpr bool kPInK = kBN * kPitch >= kBM * kBN;
    float q[kBM][kPitch];
    float k[kBN][kPitch];
    float v[kBN][D];
    float p[kPInK ? 4 : kBM * kBN];
};

// Asynchronous 16-byte copies of `rows` rows of D floats (from column col0 of
// rows row0, row0 + 1, ... of a matrix with row pitch `stride`) into shared
// memory with row pitch PITCH floats.  Rows at or past m are zero-filled: the
// copy reads 0 source bytes, from row 0 so that the address stays valid.
template <int D, int PITCH>
__device__ __forceinline__ void copy_rows_async(float* dst, const float* __restrict__ src,
                                                uint32_t row0, uint32_t m, uint32_t stride,
                                                uint32_t col0, int rows) {
    constexpr int C4 = D / 4;
#pragma unroll 4
    for (int t = threadIdx.x; t < rows * C4; t += kThreads) {
        const int r = t / C4, c = (t % C4) * 4;
        const bool live = row0 + r < m;
        const float* g = src + (size_t)(live ? row0 + r : 0u) * stride + col0 + c;
        const uint32_t sa = (uint32_t)__cvta_generic_to_shared(dst + r * PITCH + c);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                     :: "r"(sa), "l"(g), "r"(live ? 16u : 0u) : "memory");
    }
}
__device__ __forceinline__ void copies_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void copies_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// kBM query rows per CTA (64 for large problems; 32 or 16 when fewer blocks
// would leave the longest causal walks alone on a few SMs).  Grid: x = query
// head, y (+ z * gridDim.y) = query block counted from the last.
template <int D, int kBM>
__global__ void __launch_bounds__(kThreads, 2)
prefill_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                    const float* __restrict__ v, float* __restrict__ o, uint32_t m,
                    uint32_t heads_per_kv, uint32_t q_stride, uint32_t kv_stride,
                    float scale_log2) {
    constexpr int VEC = D / 32;  // output elements per lane
    constexpr int kRowsPerWarp = kBM / kWarps;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem<D, kBM>& sm = *reinterpret_cast<Smem<D, kBM>*>(smem_raw);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t nqb = (m + kBM - 1) / kBM;
    const uint32_t qb_rev = blockIdx.z * gridDim.y + blockIdx.y;
    if (qb_rev >= nqb) return;                 // past the last block (z overhang)
    const uint32_t qb = nqb - 1 - qb_rev;      // longest causal extent first
    const uint32_t h = blockIdx.x;
    const uint32_t kvh = h / heads_per_kv;
    const uint32_t q0 = qb * kBM;

    // Launched as a programmatic dependent of the previous kernel on the
    // stream: the CTA may be resident before that kernel finishes, so every
    // global read and write comes after the grid dependency resolves.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    copy_rows_async<D, D + 4>(&sm.q[0][0], q, q0, m, q_stride, h * D, kBM);
    copies_commit();

    float mrow[kRowsPerWarp], lrow[kRowsPerWarp], acc[kRowsPerWarp][VEC];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        mrow[r] = -CUDART_INF_F;
        lrow[r] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[r][e] = 0.f;
    }
    const int wr0 = warp * kRowsPerWarp;        // first local row of this warp
    const uint32_t wrow_last = q0 + wr0 + kRowsPerWarp - 1;
    const uint32_t last_row = min(q0 + kBM, m) - 1;
    const uint32_t n_tiles = last_row / kBN + 1;

    // This warp's weights for the current tile, [kRowsPerWarp][kBN], staged
    // over the K tile once every warp has finished its dot products (or in
    // their own array when the K tile is too small).
    float* const sp = (Smem<D, kBM>::kPInK ? &sm.k[0][0] : &sm.p[0]) + wr0 * kBN;
    for (uint32_t t = 0; t < n_tiles; ++t) {
        const uint32_t k0 = t * kBN;
        __syncthreads();  // the previous tile's P.V no longer reads K (P) or V
        copy_rows_async<D, D + 4>(&sm.k[0][0], k, k0, m, kv_stride, kvh * D, kBN);
        copies_commit();
        copy_rows_async<D, D>(&sm.v[0][0], v, k0, m, kv_stride, kvh * D, kBN);
        copies_commit();
        copies_wait<1>();  // Q and this tile's K have landed (V may still be in flight)
        __syncthreads();
        const bool active = k0 <= wrow_last;  // some key of the tile is attended by the warp
        // ---- scores: lane holds keys kA = k0 + lane and kB = k0 + 32 + lane
        // against every row of the warp (each K read feeds kRowsPerWarp rows).
        float sA[kRowsPerWarp], sB[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) sA[r] = sB[r] = 0.f;
        if (active) {
#pragma unroll 4
            for (int d4 = 0; d4 < D / 4; ++d4) {
                const float4 ka = *reinterpret_cast<const float4*>(&sm.k[lane][d4 * 4]);
                const float4 kb = *reinterpret_cast<const float4*>(&sm.k[32 + lane][d4 * 4]);
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    const float4 qq = *reinterpret_cast<const float4*>(&sm.q[wr0 + r][d4 * 4]);
                    sA[r] = fmaf(qq.x, ka.x, sA[r]);
                    sA[r] = fmaf(qq.y, ka.y, sA[r]);
                    sA[r] = fmaf(qq.z, ka.z, sA[r]);
                    sA[r] = fmaf(qq.w, ka.w, sA[r]);
                    sB[r] = fmaf(qq.x, kb.x, sB[r]);
                    sB[r] = fmaf(qq.y, kb.y, sB[r]);
                    sB[r] = fmaf(qq.z, kb.z, sB[r]);
                    sB[r] = fmaf(qq.w, kb.w, sB[r]);
                }
            }
            // ---- online softmax per row over the tile's 64 keys (base 2)
            const uint32_t keyA = k0 + lane, keyB = k0 + 32 + lane;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const uint32_t row = q0 + wr0 + r;
                const float a = keyA <= row ? sA[r] * scale_log2 : -CUDART_INF_F;
                const float b = keyB <= row ? sB[r] * scale_log2 : -CUDART_INF_F;
                float mx = fmaxf(a, b);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(mrow[r], mx);
                float pa = 0.f, pb = 0.f, corr = 1.f;
                if (m_new != -CUDART_INF_F) {  // some key attended so far
                    corr = exp2f(mrow[r] - m_new);
                    pa = exp2f(a - m_new);
                    pb = exp2f(b - m_new);
                }
                float ps = pa + pb;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                lrow[r] = fmaf(lrow[r], corr, ps);
                mrow[r] = m_new;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[r][e] *= corr;
                sA[r] = pa;  // the weights, kept for the P.V update
                sB[r] = pb;
            }
        }
        copies_wait<0>();  // this tile's V has landed
        __syncthreads();  // every warp's dot products are done (the K tile is free); V is visible
        if (!active) continue;
        // ---- O += P V.  The weights go to shared memory (row r, key j at
        // sp[r * kBN + j]); each lane then reads four keys' weights of a row
        // with one broadcast load and its VEC elements of the four V rows.
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            sp[r * kBN + lane] = sA[r];
            sp[r * kBN + 32 + lane] = sB[r];
        }
        __syncwarp();
        // keys past the warp's last row have weight 0: stop at the last attended one
        const int jn = (int)min((uint32_t)kBN, wrow_last - k0 + 1);
#pragma unroll 2
        for (int j = 0; j < jn; j += 4) {
            float vv[4][VEC];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float* vrow = &sm.v[j + u][lane * VEC];
                if constexpr (VEC == 4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(vrow);
                    vv[u][0] = t4.x; vv[u][1] = t4.y; vv[u][2] = t4.z; vv[u][3] = t4.w;
                } else if constexpr (VEC == 2) {
                    const float2 t2 = *reinterpret_cast<const float2*>(vrow);
                    vv[u][0] = t2.x; vv[u][1] = t2.y;
                } else {
                    vv[u][0] = vrow[0];
                }
            }
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const float4 p4 = *reinterpret_cast<const float4*>(&sp[r * kBN + j]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float a = acc[r][e];
                    a = fmaf(p4.x, vv[0][e], a);
                    a = fmaf(p4.y, vv[1][e], a);
                    a = fmaf(p4.z, vv[2][e], a);
                    a = fmaf(p4.w, vv[3][e], a);
                    acc[r][e] = a;
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const uint32_t row = q0 + wr0 + r;
        if (row >= m) continue;
        float* dst = o + (size_t)row * q_stride + h * D + lane * VEC;
        const float inv_l = 1.0f / lrow[r];
        if constexpr (VEC == 4) {
            *reinterpret_cast<float4*>(dst) =
                make_float4(acc[r][0] * inv_l, acc[r][1] * inv_l, acc[r][2] * inv_l, acc[r][3] * inv_l);
        } else if constexpr (VEC == 2) {
            *reinterpret_cast<float2*>(dst) = make_float2(acc[r][0] * inv_l, acc[r][1] * inv_l);
        } else {
            dst[0] = acc[r][0] * inv_l;
        }
    }
}

template <int D, int BM>
cudaError_t launch_bm(const float* q, const float* k, const float* v, float* o, uint32_t m,
                      uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t q_stride,
                      uint32_t kv_stride, float scale, cudaStream_t stream) {
    const int smem = (int)sizeof(Smem<D, BM>);
    const cudaError_t e = ensure_dynamic_smem<prefill_fp32_kernel<D, BM>>(smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const uint32_t nqb = (m + BM - 1) / BM;
    const uint32_t gy = nqb < 65535u ? nqb : 65535u;
    cfg.gridDim = dim3(num_q_heads, gy, (nqb + gy - 1) / gy);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_fp32_kernel<D, BM>, q, k, v, o, m,
                              num_q_heads / num_kv_heads, q_stride, kv_stride, scale * kLog2e);
}

template <int D>
cudaError_t launch_d(const float* q, const float* k, const float* v, float* o, uint32_t m,
                     uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t q_stride,
                     uint32_t kv_stride, float scale, cudaStream_t stream) {
    // The largest block that still gives the SMs several blocks each: 64
    // rows from four 64-row blocks per SM, 32 rows from one, else 16 rows.
    // Larger blocks read each K/V tile for more rows; smaller ones shorten
    // the longest causal walk, which bounds the call when blocks are few.
    const uint64_t blocks64 = (uint64_t)((m + 63) / 64) * num_q_heads;
    const uint64_t sms = (uint64_t)device_sm_count();
    if (blocks64 >= 4 * sms)
        return launch_bm<D, 64>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                scale, stream);
    if (blocks64 >= sms)
        return launch_bm<D, 32>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                scale, stream);
    return launch_bm<D, 16>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride, scale,
                            stream);
}

}  // namespace

cudaError_t launch_prefill_fp32(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, cudaStream_t stream) {
    switch (head_dim) {
        case 32:
            return launch_d<32>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                scale, stream);
        case 64:
            return launch_d<64>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                scale, stream);
        case 128:
            return launch_d<128>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                 scale, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace attn
