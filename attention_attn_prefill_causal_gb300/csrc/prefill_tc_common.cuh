// prefill_tc_common.cuh -- pieces shared by the two tensor-core prefill
// kernels (the single-tile kernel in prefill_tc.cu, the query-tile-pair
// kernel in prefill_tc_pair.cu): the split of small problems' key walks into
// chunks, the combine kernel that merges the chunks' partial results, the
// 16-bit rounding pre-pass and the TMA tensor map encoding.
//
// Operation ("aprender-gpu 0.32.0 -- prefill_fused.rs", module doc,
// Algorithm 1-3): causal grouped-query attention with an online softmax.  A
// chunk's partial is the online-softmax state (row max m, row sum l,
// unnormalised O) over its keys; the merge is the same online update applied
// to whole blocks: M = max m_c, O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

namespace attn {
namespace {

constexpr int kBM = 128;            // query rows per tile (TMEM lanes)
constexpr int kNQ = 2;              // query tiles per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint64_t kDrainWaitNs = 100000000ull;  // 100 ms: copies/MMAs in flight finish in us

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Split-KV scheduling for small grids: a work item's keys (one query tile,
// or a pair of them) are walked in chunks of kv_chunk tiles by separate CTAs;
// split items leave per-chunk partials that prefill_combine_kernel merges.
// kv_chunk = ~0u: no split.
// Chunks always cover whole 128-key blocks (kv_chunk is a multiple of
// kv_per_qtile), so every chunk that reaches a query tile's diagonal block
// holds a key for each of its rows.
constexpr uint32_t kNoSplit = 0xffffffffu;

struct SplitArgs {
    uint32_t kv_chunk;
    uint32_t n_chunks_max;
    uint32_t first_split_row;  // rows >= this belong to split pairs
    uint32_t m_pad;            // rows rounded up to whole query tiles
    uint32_t kv_per_qtile;     // key tiles per 128 keys (1: 128-key tiles, 2: 64-key tiles)
    float* part_o;             // [n_chunks_max, heads, m_pad, D] unnormalised
    float* part_ml;            // [n_chunks_max, heads, m_pad, 2] (max in log2 units, sum)
};

// Number of key tiles query tile `qt` attends to (0 when the tile is empty):
// every tile up to and including its diagonal 128-key block.
__device__ __forceinline__ uint32_t kv_tiles_for(uint32_t qt, uint32_t m, uint32_t per) {
    return (qt * kBM < m) ? (qt + 1) * per : 0;
}

// Output write-back.  An fp32 tile of O is staged as D/32 boxes of 128 rows
// x 128 bytes, box b holding columns [32b, 32b + 32) with the 16-byte chunks
// of row r XOR-swizzled by r % 8.  One warp writes rows [row0, row0 + 32) of
// it to dst (row r at dst + r * pitch floats) with whole-line stores: a store
// instruction covers one row at D = 128 (32 lanes x 16 bytes) and two rows at
// D = 64.  Rows at or past `rows` are not written.  (A TMA store of the same
// tile moves it out at the same rate, about 64 KB per us per SM; these stores
// need no tensor map, and the CTA need not wait for a bulk store's reads.)
template <int D>
__device__ __forceinline__ void store_warp_rows(const uint8_t* stage, uint32_t box_bytes,
                                                uint32_t row0, uint32_t rows, float* dst,
                                                size_t pitch, uint32_t lane) {
    constexpr uint32_t kChunks = D / 4;              // 16-byte chunks per row
    constexpr uint32_t kRowsPerStore = 32 / kChunks;
    const uint32_t sub = lane / kChunks, chunk = lane % kChunks;
    const uint32_t box = chunk / 8, c8 = chunk % 8;
#pragma unroll 8
    for (uint32_t i = 0; i < 32; i += kRowsPerStore) {
        const uint32_t r = row0 + i + sub;
        if (r < rows) {
            const float4 v = *reinterpret_cast<const float4*>(stage + box * box_bytes + r * 128 +
                                                              ((c8 ^ (r & 7u)) * 16));
            *reinterpret_cast<float4*>(dst + (size_t)r * pitch + chunk * 4) = v;
        }
    }
}

// Merge of the KV-chunk partials of split query-tile pairs.  A thread owns 8
// consecutive elements of one (row, head); the 16 (D = 128) threads of a row
// read and write whole 512-byte rows.  Up to kCombineBatch chunks are merged
// per round trip: every load of a batch is issued before any is used.
// Launched as a programmatic dependent of the prefill kernel.
constexpr uint32_t kCombineBatch = 4;

template <int D>
__global__ void __launch_bounds__(256)
prefill_combine_kernel(const SplitArgs split, float* __restrict__ o, uint32_t m,
                       uint32_t num_q_heads, uint32_t q_stride) {
    constexpr uint32_t kPerRow = D / 8;  // threads per (row, head)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t item = tid / kPerRow, e0 = (tid % kPerRow) * 8;
    const uint32_t row = split.first_split_row + item / num_q_heads;
    const uint32_t h = item % num_q_heads;
    if (row >= m) return;
    const uint32_t n_kv_tile = (row / kBM + 1) * split.kv_per_qtile;  // key tiles of this row's query tile
    const uint32_t nct = (n_kv_tile + split.kv_chunk - 1) / split.kv_chunk;
    // partial (c, h, row) sits at index (c * num_q_heads + h) * m_pad + row
    const size_t base = (size_t)h * split.m_pad + row;
    const size_t cstride = (size_t)num_q_heads * split.m_pad;
    float M = -CUDART_INF_F, L = 0.f, O[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) O[i] = 0.f;
    for (uint32_t c0 = 0; c0 < nct; c0 += kCombineBatch) {
        float2 ml[kCombineBatch];
        float4 lo[kCombineBatch], hi[kCombineBatch];
#pragma unroll
        for (uint32_t b = 0; b < kCombineBatch; ++b) {
            const uint32_t c = c0 + b;
            if (c < nct) {
                const size_t pidx = base + c * cstride;
                ml[b] = __ldcg(reinterpret_cast<const float2*>(split.part_ml) + pidx);
                const float4* po = reinterpret_cast<const float4*>(split.part_o + pidx * D + e0);
                lo[b] = __ldcg(po);
                hi[b] = __ldcg(po + 1);
            } else {
                ml[b] = make_float2(-CUDART_INF_F, 0.f);
                lo[b] = hi[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mb = M;
#pragma unroll
        for (uint32_t b = 0; b < kCombineBatch; ++b) Mb = fmaxf(Mb, ml[b].x);
        const float fo = ex2(M - Mb);  // M = -inf on the first batch: 0
        L *= fo;
#pragma unroll
        for (int i = 0; i < 8; ++i) O[i] *= fo;
#pragma unroll
        for (uint32_t b = 0; b < kCombineBatch; ++b) {
            const float f = ex2(ml[b].x - Mb);  // -inf (absent chunk): 0
            L = fmaf(ml[b].y, f, L);
            O[0] = fmaf(lo[b].x, f, O[0]);
            O[1] = fmaf(lo[b].y, f, O[1]);
            O[2] = fmaf(lo[b].z, f, O[2]);
            O[3] = fmaf(lo[b].w, f, O[3]);
            O[4] = fmaf(hi[b].x, f, O[4]);
            O[5] = fmaf(hi[b].y, f, O[5]);
            O[6] = fmaf(hi[b].z, f, O[6]);
            O[7] = fmaf(hi[b].w, f, O[7]);
        }
        M = Mb;
    }
    const float inv = 1.0f / L;
    float4* dst = reinterpret_cast<float4*>(o + (size_t)row * q_stride + (size_t)h * D + e0);
    dst[0] = make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
    dst[1] = make_float4(O[4] * inv, O[5] * inv, O[6] * inv, O[7] * inv);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 16-bit pre-pass: k [m, kv_stride] -> kh [m, kv_cols] rounded to fp16/bf16
// (grid.y = 0), likewise v (grid.y = 1).  Each thread converts 8 consecutive
// elements of one row (two 128-bit loads, one 128-bit store).
template <bool BF16>
__global__ void __launch_bounds__(256)
round_operands_kernel(const float* __restrict__ k, const float* __restrict__ v,
                      uint16_t* __restrict__ kh, uint16_t* __restrict__ vh, uint32_t m,
                      uint32_t kv_cols, uint32_t kv_stride, unsigned int* status) {
    // A programmatic dependent of the kernel before it: wait for that grid
    // before any global access, then let the prefill kernel launch (it reads
    // kh and vh only after this grid has completed).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const float* src = blockIdx.y == 0 ? k : v;
    uint16_t* dst = blockIdx.y == 0 ? kh : vh;
    const uint32_t per_row = kv_cols / 8;
    const size_t total = (size_t)m * per_row;
    bool overflow = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / per_row;
        const uint32_t c = (uint32_t)(i % per_row) * 8;
        const float4* s4 = reinterpret_cast<const float4*>(src + r * kv_stride + c);
        const float4 a = __ldcs(s4), b = __ldcs(s4 + 1);
        uint4 out;
        out.x = pack_half2(a.x, a.y, BF16);
        out.y = pack_half2(a.z, a.w, BF16);
        out.z = pack_half2(b.x, b.y, BF16);
        out.w = pack_half2(b.z, b.w, BF16);
        if (!BF16) {
            const float mx = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                   fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
            overflow |= !(mx <= 65504.f);
        }
        *reinterpret_cast<uint4*>(dst + r * kv_cols + c) = out;
    }
    if (__any_sync(0xffffffffu, overflow) && (threadIdx.x % 32) == 0)
        atomicOr(status, kStatusRange);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// fp32 map with 128-byte swizzle: rows of `cols` floats with a pitch of
// `row_stride` floats, boxes of 32 floats (128 bytes) x box_rows.  Used for
// the caller's Q and O, the chunks' partials, and the TF32 operands.
bool encode_output_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                       uint64_t row_stride, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {row_stride * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), gdim,
                     gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// fp16/bf16 operand map: tight rows of `cols` elements, boxes of 64
// elements (128 bytes) x box_rows, 128-byte swizzle.
bool encode_operand_map(CUtensorMap* map, const void* base, uint32_t cols, uint32_t rows,
                        uint32_t box_rows, bool bf16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     2, const_cast<void*>(base), gdim, gstride, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct PrefillPlan {
    uint32_t n_items;          // work items per head (pairs, or pair chunks)
    SplitArgs split;           // kv_chunk == kNoSplit: no split
    size_t part_o_bytes, part_ml_bytes;
};

// Split the KV walk only when the work items alone leave SMs idle: then
// take the smallest chunk (most parallelism, shortest item) whose items still
// fit in one wave.  A work item is `tiles_per_item` consecutive query tiles
// (a pair in the 16-bit kernel, one tile in the TF32 kernel); chunks are
// counted in 128-key blocks (nk(u) = blocks of item u's last tile) and
// converted to key tiles of 128 / kv_per_qtile keys.
PrefillPlan make_plan(uint32_t m, uint32_t num_q_heads, uint32_t head_dim, int sm_count,
                      uint32_t kv_per_qtile, uint32_t tiles_per_item) {
    PrefillPlan p{};
    const uint32_t n_qt = (m + kBM - 1) / kBM;
    const uint32_t n_units = (m + tiles_per_item * kBM - 1) / (tiles_per_item * kBM);
    auto nk = [&](uint32_t u) { return std::min(tiles_per_item * u + tiles_per_item, n_qt); };
    p.n_items = n_units;
    p.split.kv_chunk = kNoSplit;
    p.split.n_chunks_max = 1;
    p.split.first_split_row = m;
    p.split.m_pad = n_qt * kBM;
    p.split.kv_per_qtile = kv_per_qtile;
    const uint32_t sms = (uint32_t)std::max(sm_count, 1);
    if (n_units > 0 && (uint64_t)n_units * num_q_heads < sms) {
        const uint32_t nk_last = nk(n_units - 1);
        for (uint32_t c = 2; c < nk_last; ++c) {
            uint32_t items = 0;
            for (uint32_t u = 0; u < n_units; ++u) items += (nk(u) + c - 1) / c;
            if ((uint64_t)items * num_q_heads <= sms) {
                p.n_items = items;
                p.split.kv_chunk = c * kv_per_qtile;
                p.split.n_chunks_max = (nk_last + c - 1) / c;
                uint32_t first = 0;
                while (first < n_units && nk(first) <= c) ++first;
                p.split.first_split_row = std::min(m, first * tiles_per_item * kBM);
                break;
            }
        }
    }
    if (p.split.kv_chunk != kNoSplit) {
        const size_t rows = (size_t)p.split.n_chunks_max * num_q_heads * p.split.m_pad;
        p.part_o_bytes = align256(rows * head_dim * 4);
        p.part_ml_bytes = align256(rows * 2 * 4);
    }
    return p;
}

}  // namespace
}  // namespace attn
