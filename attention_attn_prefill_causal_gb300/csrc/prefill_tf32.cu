// prefill_tf32.cu -- causal grouped-query prefill on the Blackwell tensor cores
// with TF32 operands (tcgen05 kind::tf32 MMAs, fp32 accumulation in TMEM).
//
// Operation ("aprender-gpu 0.32.0 -- prefill_fused.rs", module doc,
// Algorithm 1-3): for query head h and KV head g = h / heads_per_kv, row i
// of O is sum_{j<=i} softmax_j(scale * Q[i].K[j]) V[j], with an online
// softmax.  The page packs fp32 Q, K, V; this path keeps them fp32 in memory
// and feeds the tensor core TF32 (fp32's 8-bit exponent, so no input range
// limit beyond fp32's own, and a 10-bit mantissa).
//
// Precision.  A kind::tf32 MMA uses the top 19 bits of each fp32 operand
// (the low 13 mantissa bits are dropped).  Q goes to the tensor core as the
// caller stored it.  K and V are rounded to nearest TF32 by a pre-pass: an
// operand dropped toward zero would bias the output (O = V[0] exactly for
// row 0), which rounding to nearest halves and unbiases.  P is truncated to
// TF32 by the softmax itself and the row sum is taken over the truncated
// weights, so the weights the MMA applies are normalised exactly (a row sum
// over the untruncated weights would scale every output down by up to
// 2^-10 where the running max lags the row's largest score).
//
// Layout.  The pre-pass writes K rounded, [m, kv_heads*D] fp32, and V
// rounded and transposed per KV head, [kv_heads*D, m4] fp32 (keys
// contiguous, m4 = m rounded up to 4), so that both MMAs read K-major
// operands in the 128-byte swizzled layout TMA writes: S = Q K^T takes Q
// (128 rows x D) and a K tile (64 keys x D); O += P V takes P from TMEM
// (128 rows x 64 keys, one fp32 per column) and a V^T tile (D rows x 64
// keys).
//
// CTA work unit: two consecutive 128-row query tiles of one head (as in the
// 16-bit kernel), keys walked in 64-key tiles up to the diagonal.  Shared
// memory holds both fp32 query tiles (2 x 64 KB at D = 128) and a ring of
// three 32 KB slots that K tiles and V^T tiles pass through in load order
// K(0), V(0), K(1), V(1), ...; a K tile is freed when both query tiles'
// S MMAs of it completed, a V^T tile when both P.V MMAs did.  Warp roles
// (320 threads): warps 0-3 softmax for tile A, 4-7 for tile B (thread =
// TMEM lane = query row), warp 8 TMA producer, warp 9 TMEM allocator and
// MMA issuer.  TMEM per tile: S/P in 64 columns and O in D columns.  The MMA
// thread ping-pongs the tiles exactly as the 16-bit kernel does.
// Epilogue: after the CTA's last MMA the query tiles are dead; each softmax
// thread writes its row of O into the 128-byte swizzled boxes that held its
// tile's Q, and one thread per tile stores them with TMA.
// Small grids split each pair's key walk into chunks of whole 128-key
// blocks, merged by the combine kernel shared with the 16-bit path.
// Launch chain (programmatic dependent launches): the pre-pass waits for the
// kernel before the call, then lets this kernel launch; this kernel stages
// the caller's Q at once and waits for the pre-pass before its first K/V
// load; the combine waits for this kernel.
// Every mbarrier wait is bounded; on a timeout a thread records
// kStatusTimeout, abandons its loop, and the CTA still drains its copies,
// waits for its MMAs and frees TMEM before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "attn_internal.h"
#include "prefill_tc_common.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int kBK = 64;                // keys per key tile
constexpr uint32_t kPerQ = kBM / kBK;  // key tiles per 128-key block
constexpr int kSlots = 3;              // operand ring slots
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTf32Mask = 0xFFFFE000u;  // the bits of an fp32 a TF32 operand keeps

template <int D>
struct Tf32Layout {
    static constexpr uint32_t kQBoxBytes = kBM * 128;           // 128 rows x 32 floats
    static constexpr uint32_t kQTileBytes = kBM * D * 4;        // D/32 boxes
    static constexpr uint32_t kKBoxBytes = kBK * 128;           // 64 keys x 32 floats
    static constexpr uint32_t kVBoxBytes = D * 128;             // D rows x 32 keys
    static constexpr uint32_t kSlotBytes = kBK * D * 4;         // one K or V^T tile
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kRingOff = kNQ * kQTileBytes;
    static constexpr uint32_t kBytes = kRingOff + kSlots * kSlotBytes;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;       // room to align to 1 KB
    static constexpr uint32_t kTileCols = D == 128 ? 256 : 128; // TMEM columns per tile
    static constexpr uint32_t kOCol = D == 128 ? 128 : 64;      // O's first column in a tile
    static constexpr uint32_t kTmemCols = kNQ * kTileCols;
    static_assert(kBK + D <= kTileCols && kOCol >= kBK, "TMEM tile layout");
    static_assert(kSmemAlloc <= 227 * 1024, "shared memory");
    // O staging (fp32, the same box layout as Q) reuses the query tiles.
    static_assert(kQTileBytes == kBM * D * 4, "O staging");
};

struct __align__(8) Tf32Barriers {
    uint64_t q_full[kNQ];
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t s_full[kNQ];
    uint64_t p_full[kNQ];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};

__device__ __forceinline__ void record_timeout(unsigned int* status, Tf32Barriers* bars) {
    atomicOr(status, kStatusTimeout);
    atomicExch(&bars->abort, 1u);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tf32_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_po, uint32_t m,
                    uint32_t num_q_heads, uint32_t heads_per_kv,
                    float scale_log2, unsigned int* status, uint64_t wait_ns,
                    const SplitArgs split) {
    using L = Tf32Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ Tf32Barriers bars;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t n_pairs = (m + kNQ * kBM - 1) / (kNQ * kBM);
    const uint32_t h = blockIdx.x % num_q_heads;
    const uint32_t kvh = h / heads_per_kv;
    // Work item: (query-tile pair, key chunk), heaviest pairs first.
    uint32_t pair = 0, chunk = 0, n_chunks = 1;
    if (split.kv_chunk == kNoSplit) {
        pair = n_pairs - 1 - blockIdx.x / num_q_heads;
    } else {
        uint32_t idx = blockIdx.x / num_q_heads;
        for (int p = (int)n_pairs - 1; p >= 0; --p) {
            const uint32_t nk = max(kv_tiles_for(p * kNQ, m, kPerQ),
                                    kv_tiles_for(p * kNQ + 1, m, kPerQ));
            const uint32_t nc = (nk + split.kv_chunk - 1) / split.kv_chunk;
            if (idx < nc) {
                pair = (uint32_t)p;
                chunk = idx;
                n_chunks = nc;
                break;
            }
            idx -= nc;
        }
    }
    const uint32_t qt0 = pair * kNQ;
    uint32_t n_kv[kNQ];
#pragma unroll
    for (int t = 0; t < kNQ; ++t) n_kv[t] = kv_tiles_for(qt0 + t, m, kPerQ);
    uint32_t n_kv_pair = 0;
#pragma unroll
    for (int t = 0; t < kNQ; ++t) n_kv_pair = max(n_kv_pair, n_kv[t]);
    // This item's key tiles are [j0, j0 + n_kv_all); tile t takes the first
    // tile_n[t] of them.
    const uint32_t j0 = split.kv_chunk == kNoSplit ? 0u : chunk * split.kv_chunk;
    const uint32_t n_kv_all =
        split.kv_chunk == kNoSplit ? n_kv_pair : min(n_kv_pair, j0 + split.kv_chunk) - j0;
    uint32_t tile_n[kNQ];
#pragma unroll
    for (int t = 0; t < kNQ; ++t) tile_n[t] = n_kv[t] > j0 ? min(n_kv[t] - j0, n_kv_all) : 0;

    const uint32_t sQ = smem_u32(smem + L::kQOff);
    const uint32_t sR = smem_u32(smem + L::kRingOff);

    if (threadIdx.x == 0) {
        for (int t = 0; t < kNQ; ++t) {
            mbar_init(smem_u32(&bars.q_full[t]), 1);
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), kBM);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(smem_u32(&bars.full[s]), 1);
            mbar_init(smem_u32(&bars.empty[s]), 1);
        }
        mbar_init(smem_u32(&bars.mma_done), 1);
        bars.abort = 0;
        fence_mbar_init();
        // A split's combine kernel may launch now; it waits for this grid.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars.tmem_base), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_vt);
            for (int t = 0; t < kNQ; ++t) {
                const uint32_t bar = smem_u32(&bars.q_full[t]);
                mbar_arrive_expect_tx(bar, L::kQTileBytes);
                for (uint32_t b = 0; b < D / 32; ++b)
                    tma_load_2d(sQ + t * L::kQTileBytes + b * L::kQBoxBytes, &tm_q, bar,
                                (int32_t)(h * D + b * 32), (int32_t)((qt0 + t) * kBM));
            }
            // K and V^T come from the pre-pass: read them only once its grid
            // (and with it every kernel before the call) has completed.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // Load n of the item: K(n/2) for even n, V^T(n/2) for odd n, into
            // slot n % kSlots (use n / kSlots of that slot).
            const uint32_t n_loads = 2 * n_kv_all;
            uint32_t issued = 0;
            bool ok = true;
            for (uint32_t n = 0; n < n_loads; ++n) {
                const uint32_t slot = n % kSlots, use = n / kSlots;
                if (use > 0) {
                    ok = mbar_wait(smem_u32(&bars.empty[slot]), (use - 1) & 1, wait_ns, status,
                                   kStatusTimeout);
                    if (!ok) break;
                }
                const uint32_t bar = smem_u32(&bars.full[slot]);
                const uint32_t dst = sR + slot * L::kSlotBytes;
                const uint32_t key0 = (j0 + n / 2) * kBK;
                mbar_arrive_expect_tx(bar, L::kSlotBytes);
                if ((n & 1) == 0) {
                    for (uint32_t b = 0; b < D / 32; ++b)
                        tma_load_2d(dst + b * L::kKBoxBytes, &tm_k, bar, (int32_t)(kvh * D + b * 32),
                                    (int32_t)key0);
                } else {
                    for (uint32_t b = 0; b < kBK / 32; ++b)
                        tma_load_2d(dst + b * L::kVBoxBytes, &tm_vt, bar, (int32_t)(key0 + b * 32),
                                    (int32_t)(kvh * D));
                }
                issued = n + 1;
            }
            if (!ok) record_timeout(status, &bars);
            // Drain: every copy this CTA issued must land before it exits.
            for (int t = 0; t < kNQ; ++t) mbar_wait(smem_u32(&bars.q_full[t]), 0, kDrainWaitNs);
            for (uint32_t n = (issued > kSlots ? issued - kSlots : 0); n < issued; ++n)
                mbar_wait(smem_u32(&bars.full[n % kSlots]), (n / kSlots) & 1, kDrainWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_tf32(kBK, kBM);
            constexpr uint32_t idesc_pv = idesc_tf32(D, kBM);
            bool ok = true;
            for (int t = 0; t < kNQ && ok; ++t)
                ok = mbar_wait(smem_u32(&bars.q_full[t]), 0, wait_ns, status, kStatusTimeout);
            // Descriptor bases, built once; an operand at byte offset off in a
            // tile is the base plus off >> 4.  K step ks (8 fp32 = 32 bytes)
            // sits (ks % 4) * 32 bytes into a 128-byte swizzled row, in box ks / 4.
            const uint64_t dq0 = smem_desc(sQ, 16, 1024, 2);
            const uint64_t dq1 = smem_desc(sQ + L::kQTileBytes, 16, 1024, 2);
            const uint64_t dr0 = smem_desc(sR, 16, 1024, 2);
            auto slot_desc = [&](uint32_t n) {  // descriptor of load n's slot
                return dr0 + (uint64_t)((n % kSlots) * (L::kSlotBytes / 16));
            };
            auto issue_s = [&](int t, uint32_t j) {
                const uint64_t a0 = t == 0 ? dq0 : dq1;
                const uint64_t b0 = slot_desc(2 * j);
                const uint32_t d = tmem + t * L::kTileCols;
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks) {
                    const uint64_t offa = (uint64_t)((ks / 4) * (L::kQBoxBytes / 16) + (ks % 4) * 2);
                    const uint64_t offb = (uint64_t)((ks / 4) * (L::kKBoxBytes / 16) + (ks % 4) * 2);
                    mma_tf32_ss(d, a0 + offa, b0 + offb, idesc_s, ks > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars.s_full[t]));
            };
            auto issue_pv = [&](int t, uint32_t j) {
                const uint64_t b0 = slot_desc(2 * j + 1);
                const uint32_t a = tmem + t * L::kTileCols, d = a + L::kOCol;
                const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
                for (int ks = 0; ks < kBK / 8; ++ks)
                    mma_tf32_ts(d, a + ks * 8,
                                b0 + (uint64_t)((ks / 4) * (L::kVBoxBytes / 16) + (ks % 4) * 2),
                                idesc_pv, ks > 0 ? 1u : acc0);
            };
            auto wait_load = [&](uint32_t n) {
                return mbar_wait(smem_u32(&bars.full[n % kSlots]), (n / kSlots) & 1, wait_ns, status,
                                 kStatusTimeout);
            };
            if (ok && n_kv_all > 0) {
                ok = wait_load(0);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < kNQ; ++t)
                        if (tile_n[t] > 0) issue_s(t, 0);
                    mma_commit(smem_u32(&bars.empty[0]));
                }
            }
            for (uint32_t j = 0; j < n_kv_all && ok; ++j) {
                ok = wait_load(2 * j + 1);
                if (!ok) break;
                tc_fence_after();
                bool k_next_ready = false;
                const uint32_t jn = j + 1;
                // V(j)'s slot is released as soon as its last P.V MMA is
                // issued (its commit completes with that MMA), so that the
                // K tile two steps ahead, which reuses the slot, loads during
                // the following S MMA rather than after it.
                const int last_pv = j < tile_n[1] ? 1 : 0;
                for (int t = 0; t < kNQ && ok; ++t) {
                    if (j < tile_n[t]) {
                        ok = mbar_wait(smem_u32(&bars.p_full[t]), j & 1, wait_ns, status, kStatusTimeout);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, j);
                    }
                    if (t == last_pv) mma_commit(smem_u32(&bars.empty[(2 * j + 1) % kSlots]));
                    if (jn < tile_n[t]) {
                        if (!k_next_ready) {
                            ok = wait_load(2 * jn);
                            if (!ok) break;
                            tc_fence_after();
                            k_next_ready = true;
                        }
                        issue_s(t, jn);
                    }
                }
                if (!ok) break;
                if (k_next_ready) mma_commit(smem_u32(&bars.empty[(2 * jn) % kSlots]));
            }
            if (!ok) record_timeout(status, &bars);
            // Wait until every MMA this thread issued has completed.
            mma_commit(smem_u32(&bars.mma_done));
            mbar_wait(smem_u32(&bars.mma_done), 0, kDrainWaitNs);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int t = warp / 4;                 // query tile of this warpgroup
        const int wq = warp % 4;                // TMEM lane quarter
        const uint32_t row_in_tile = wq * 32 + lane;
        const uint32_t tile_row0 = (qt0 + t) * kBM;
        const uint32_t row = tile_row0 + row_in_tile;
        const uint32_t t_s = tmem + t * L::kTileCols + ((uint32_t)(wq * 32) << 16);
        const uint32_t t_o = t_s + L::kOCol;
        bool ok = true;
        float m_used = -CUDART_INF_F;  // log2 units
        float l_sum = 0.f;
        const uint32_t nkv = tile_n[t];
        for (uint32_t j = 0; j < nkv; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full[t]), j & 1, wait_ns, status, kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
            tc_fence_after();
            float s[kBK];
            {
                uint32_t r[kBK];
                tmem_ld64_sync(t_s, r);
#pragma unroll
                for (int i = 0; i < kBK; ++i) s[i] = __uint_as_float(r[i]);
            }
            const uint32_t key0 = (j0 + j) * kBK;
            if (key0 + kBK > tile_row0) {  // the diagonal block: keys above the row are not attended
#pragma unroll
                for (int c = 0; c < kBK; ++c)
                    if (key0 + c > row) s[c] = -CUDART_INF_F;
            }
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
            for (int c = 8; c < kBK; ++c) mx8[c % 8] = fmaxf(mx8[c % 8], s[c]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_new = mx * scale_log2;
            float corr = 1.f;
            bool rescale = false;
            if (m_new > m_used + kRescaleThreshold) {
                corr = ex2(m_used - m_new);      // 0 on the first tile
                rescale = (j > 0);
                m_used = m_new;
            }
            // A row with no attended key so far (every score -inf) keeps its
            // weights at exactly 0 instead of forming -inf - (-inf).
            const float neg_m = m_used == -CUDART_INF_F ? 0.f : -m_used;
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nm2 = make_float2(neg_m, neg_m);
            float2 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBK / 32; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 x = __ffma2_rn(
                        make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sc2, nm2);
                    // The MMA reads the weights' top 19 bits; the row sum takes
                    // the same truncated values, so the output is an exact
                    // convex combination of the weights the MMA used.
                    const uint32_t b0 = __float_as_uint(ex2(x.x)) & kTf32Mask;
                    const uint32_t b1 = __float_as_uint(ex2(x.y)) & kTf32Mask;
                    acc[i % 4] = __fadd2_rn(acc[i % 4],
                                            make_float2(__uint_as_float(b0), __uint_as_float(b1)));
                    pk[2 * i] = b0;
                    pk[2 * i + 1] = b1;
                }
                tmem_st32(t_s + c * 32, pk);
            }
            const float rowsum = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                                 ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
            l_sum = fmaf(l_sum, corr, rowsum);
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? corr : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32_sync(t_o + c * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                    tmem_st32(t_o + c * 32, r);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.p_full[t]));
        }
        // ---- epilogue: O (normalised, or this chunk's unnormalised partial)
        // into the tile's query boxes, then TMA stores of whole lines.
        const bool split_item = n_chunks > 1;
        if (ok && nkv > 0) {
            ok = mbar_wait(smem_u32(&bars.mma_done), 0, wait_ns, status, kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) ok = false;
        }
        uint8_t* stage = smem + L::kQOff + t * L::kQTileBytes;
        if (ok && nkv > 0) {
            tc_fence_after();
            const float scale_o = split_item ? 1.f : 1.0f / l_sum;
            const uint32_t sw = row_in_tile & 7u;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32_sync(t_o + c * 32, r);
                uint8_t* box_row = stage + c * L::kQBoxBytes + row_in_tile * 128;
#pragma unroll
                for (uint32_t q4 = 0; q4 < 8; ++q4) {
                    const uint32_t i = 4 * q4;
                    const float4 v4 = make_float4(__uint_as_float(r[i]) * scale_o,
                                                  __uint_as_float(r[i + 1]) * scale_o,
                                                  __uint_as_float(r[i + 2]) * scale_o,
                                                  __uint_as_float(r[i + 3]) * scale_o);
                    *reinterpret_cast<float4*>(box_row + ((q4 ^ sw) * 16)) = v4;
                }
            }
            if (split_item && row < m) {
                const size_t pidx = ((size_t)chunk * num_q_heads + h) * split.m_pad + row;
                *reinterpret_cast<float2*>(split.part_ml + 2 * pidx) = make_float2(m_used, l_sum);
            }
            fence_proxy_async_smem();
        }
        named_barrier(1 + t, 128);
        if (ok && nkv > 0 && wq == 0 && lane == 0) {
            const int32_t y0 = (int32_t)tile_row0;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                const uint32_t src = smem_u32(stage + c * L::kQBoxBytes);
                if (split_item)
                    tma_store_2d(&tm_po, src, c * 32,
                                 (int32_t)((chunk * num_q_heads + h) * split.m_pad) + y0);
                else
                    tma_store_2d(&tm_o, src, (int32_t)(h * D + c * 32), y0);
            }
            bulk_commit_group();
            bulk_wait_all_read();  // the staging must outlive the reads, not the writes
        }
        if (!ok && lane == 0) record_timeout(status, &bars);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// Pre-pass: K rounded to nearest TF32 into kr [m, kv_cols] (grid.y = 0,
// eight elements per thread), and V rounded and transposed into
// vt [kv_cols, m4] (grid.y = 1, 32 x 32 tiles through shared memory: rows of
// V in, rows of V^T out, both as whole 128-byte lines).
__global__ void __launch_bounds__(256)
round_transpose_tf32_kernel(const float* __restrict__ k, const float* __restrict__ v,
                            float* __restrict__ kr, float* __restrict__ vt, uint32_t m,
                            uint32_t kv_cols, uint32_t kv_stride, uint32_t m4) {
    // A programmatic dependent of the kernel before it: wait for that grid
    // before any global access, then let the prefill kernel launch (it reads
    // kr and vt only after this grid has completed).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.y == 0) {
        const uint32_t per_row = kv_cols / 8;
        const size_t total = (size_t)m * per_row;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
             i += (size_t)gridDim.x * blockDim.x) {
            const size_t r = i / per_row;
            const uint32_t c = (uint32_t)(i % per_row) * 8;
            const float4* s4 = reinterpret_cast<const float4*>(k + r * kv_stride + c);
            float4 a = __ldcs(s4), b = __ldcs(s4 + 1);
            a = make_float4(round_tf32(a.x), round_tf32(a.y), round_tf32(a.z), round_tf32(a.w));
            b = make_float4(round_tf32(b.x), round_tf32(b.y), round_tf32(b.z), round_tf32(b.w));
            float4* d4 = reinterpret_cast<float4*>(kr + r * kv_cols + c);
            d4[0] = a;
            d4[1] = b;
        }
        return;
    }
    __shared__ float tile[32][33];
    const uint32_t tx = threadIdx.x % 32, ty = threadIdx.x / 32;  // 32 x 8 threads
    const uint32_t key_tiles = (m + 31) / 32, col_tiles = kv_cols / 32;
    for (uint32_t tid = blockIdx.x; tid < key_tiles * col_tiles; tid += gridDim.x) {
        const uint32_t j0 = (tid / col_tiles) * 32, c0 = (tid % col_tiles) * 32;
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
            const uint32_t j = j0 + ty + 8 * i;
            tile[ty + 8 * i][tx] = j < m ? round_tf32(__ldcs(v + (size_t)j * kv_stride + c0 + tx)) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
            const uint32_t c = c0 + ty + 8 * i, j = j0 + tx;
            if (j < m4) vt[(size_t)c * m4 + j] = tile[tx][ty + 8 * i];
        }
        __syncthreads();
    }
}

struct Tf32Workspace {
    size_t kr_bytes, vt_bytes;
    uint32_t m4;
};

Tf32Workspace tf32_operands(uint32_t m, uint32_t num_kv_heads, uint32_t head_dim) {
    Tf32Workspace w{};
    w.m4 = (m + 3) / 4 * 4;
    w.kr_bytes = align256((size_t)m * num_kv_heads * head_dim * 4);
    w.vt_bytes = align256((size_t)num_kv_heads * head_dim * w.m4 * 4);
    return w;
}

template <int D>
cudaError_t launch_tf32(const float* q, const float* k, const float* v, float* o, uint32_t m,
                        uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t q_stride,
                        uint32_t kv_stride, float scale, void* workspace, unsigned int* status,
                        uint64_t wait_ns, cudaStream_t stream) {
    using L = Tf32Layout<D>;
    const PrefillPlan plan = make_plan(m, num_q_heads, D, device_sm_count(), kPerQ);
    const Tf32Workspace w = tf32_operands(m, num_kv_heads, D);
    const uint32_t q_cols = num_q_heads * D, kv_cols = num_kv_heads * D;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* kr = reinterpret_cast<float*>(ws);
    float* vt = reinterpret_cast<float*>(ws + w.kr_bytes);
    SplitArgs split = plan.split;
    split.part_o = reinterpret_cast<float*>(ws + w.kr_bytes + w.vt_bytes);
    split.part_ml = reinterpret_cast<float*>(ws + w.kr_bytes + w.vt_bytes + plan.part_o_bytes);

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        const size_t k_work = (size_t)m * kv_cols / 8;
        const size_t v_tiles = (size_t)((m + 31) / 32) * (kv_cols / 32);
        const uint32_t blocks =
            (uint32_t)std::min<size_t>(std::max<size_t>((k_work + 255) / 256, v_tiles), 4096);
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(blocks, 2, 1);
        pcfg.blockDim = dim3(256, 1, 1);
        pcfg.stream = stream;
        pcfg.attrs = attr;
        pcfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&pcfg, round_transpose_tf32_kernel, k, v, kr, vt,
                                                 m, kv_cols, kv_stride, w.m4);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tq, tk, tvt, to, tpo;
    if (!encode_output_map(&tq, q, q_cols, m, q_stride, kBM) ||
        !encode_output_map(&tk, kr, kv_cols, m, kv_cols, kBK) ||
        !encode_output_map(&tvt, vt, m, kv_cols, w.m4, D) ||
        !encode_output_map(&to, o, q_cols, m, q_stride, kBM))
        return cudaErrorNotSupported;
    if (split.kv_chunk != kNoSplit) {
        if (!encode_output_map(&tpo, split.part_o, D,
                               (uint64_t)split.n_chunks_max * num_q_heads * split.m_pad, D, kBM))
            return cudaErrorNotSupported;
    } else {
        tpo = to;  // not used without a split
    }
    {
        const cudaError_t e = ensure_dynamic_smem<prefill_tf32_kernel<D>>((int)L::kSmemAlloc);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_items * num_q_heads, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemAlloc;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tf32_kernel<D>, tq, tk, tvt, to, tpo, m,
                                       num_q_heads, num_q_heads / num_kv_heads, scale * kLog2e,
                                       status, wait_ns, split);
    if (e != cudaSuccess || split.kv_chunk == kNoSplit) return e;
    const uint32_t rows = m - split.first_split_row;
    const uint64_t threads = (uint64_t)rows * num_q_heads * (D / 8);
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3((uint32_t)((threads + 255) / 256), 1, 1);
    ccfg.blockDim = dim3(256, 1, 1);
    ccfg.stream = stream;
    ccfg.attrs = attr;
    ccfg.numAttrs = 1;
    return cudaLaunchKernelEx(&ccfg, prefill_combine_kernel<D>, split, o, m, num_q_heads, q_stride);
}

}  // namespace

size_t prefill_tf32_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                    uint32_t head_dim) {
    const PrefillPlan p = make_plan(m, num_q_heads, head_dim, device_sm_count(), kPerQ);
    const Tf32Workspace w = tf32_operands(m, num_kv_heads, head_dim);
    return w.kr_bytes + w.vt_bytes + p.part_o_bytes + p.part_ml_bytes;
}

cudaError_t launch_prefill_tf32(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, void* workspace, unsigned int* status,
                                uint64_t wait_ns, cudaStream_t stream) {
    if (head_dim == 128)
        return launch_tf32<128>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                scale, workspace, status, wait_ns, stream);
    if (head_dim == 64)
        return launch_tf32<64>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                               scale, workspace, status, wait_ns, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
