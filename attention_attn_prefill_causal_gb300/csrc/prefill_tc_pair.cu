// prefill_tc_pair.cu -- the 16-bit (fp16 / bf16) causal prefill for grids
// of at least two waves of query-tile pairs: each CTA walks two 128-row
// query tiles over every K and V tile it loads, so a tile's load and its
// barrier round trip serve twice the MMAs of the single-tile kernel in
// prefill_tc.cu (which takes the smaller grids, where finer work items
// balance better).
//
// Operation ("aprender-gpu 0.32.0 -- prefill_fused.rs", module doc,
// Algorithm 1-3): for query head h and KV head g = h / heads_per_kv, row i
// of O is sum_{j<=i} softmax_j(scale * Q[i].K[j]) V[j], computed with an
// online softmax.  The page does this with one warp per head on CUDA cores;
// here the two contractions (S = Q K^T and O += P V) run on the tensor core.
//
// Precision: Q, K, V (fp32, packed strides) are rounded to fp16 with
// round-to-nearest (10-bit mantissa, the same as TF32): K and V by a pre-pass
// into a workspace, Q inside this kernel (each CTA stages its two fp32 query
// tiles with TMA and the softmax warps round them once).  The softmax writes
// P as fp16, and every MMA accumulates in fp32.  Softmax statistics (row max,
// row sum) and the output stay fp32.
//
// CTA work unit: two consecutive 128-row query tiles (A = rows q0..q0+127,
// B = q0+128..q0+255) of one head; keys are walked in 128-row tiles up to the
// diagonal.  Warp roles (352 threads):
//   warps 0-3  softmax for tile A  (thread r owns TMEM lane r = query row r)
//   warps 4-7  softmax for tile B
//   warp  8    TMA producer: both fp32 Q tiles once (staged in the K and
//              V rings, which the softmax warps then free by rounding them
//              into the fp16 Q tiles), then K and V tiles into a
//              two-stage ring
//   warp  9    TMEM allocator and MMA issuer (one thread)
//   warp 10    gate: for every step j at which tile A has keys, waits
//              for V(j) and K(j+1) to land, then arrives on tile A's P
//              barrier, so the MMA thread waits twice per step (P_A with
//              the loads, then P_B) instead of four times: each mbarrier
//              wait on the issuing thread stalls the tensor pipe even when
//              its phase has already completed.  The gate arrives for step
//              j only after the phase of step j - 1 has completed, and the
//              phase of step j completes only with tile A's P(j), whose S
//              the MMA thread issued after passing step j - 1: the barrier
//              stays within one phase of its waiters.  At the steps where
//              tile A has no keys (the last step of a pair) the MMA thread
//              waits for the loads itself.
// TMEM (512 columns): per tile, S/P in 128 columns (P is written as packed
// fp16 pairs over the first 64 columns of S) and O in head_dim columns.
// The MMA thread ping-pongs: while softmax A works on S_A(j), the tensor core
// runs PV_B(j-1) and S_B(j); while softmax B works, it runs PV_A(j) and
// S_A(j+1).  tcgen05 MMAs issued by one thread execute in order, so S_t(j+1)
// may overwrite the TMEM that held P_t(j) right after PV_t(j) is issued, and
// the commit that signals S_t(j+1) also covers PV_t(j): once softmax t sees
// S_t(j+1) its O accumulator is stable and can be rescaled.
// The MMA thread builds each operand tile's descriptor once and reaches the
// operand of every K step with one 64-bit add: work between consecutive MMAs
// on the issuing thread directly lowers the rate the tensor pipe is fed at.
// Rescaling is conditional: the running max used for the exponentials only
// moves when the row max grows by more than 8 (log2 units); the final O / l
// is exact either way, and P stays below 2^8.
// Epilogue: after the CTA's last MMA the K/V ring is free; each softmax
// thread writes its row of O into 128-byte swizzled staging boxes there, and
// each warp then writes the 32 rows it staged back, a whole row (or two at
// D = 64) per store instruction, so O leaves in whole 128-byte lines rather
// than one 16-byte piece per row and instruction.
// Small grids (query-tile pairs x heads below the SM count) split each
// pair's key walk into chunks of C tiles, one work item per chunk; chunks
// write unnormalised partials and a combine kernel merges them.
// Launch chain: the rounding pre-pass waits for the kernel before the call
// and then lets this kernel launch; this kernel stages the caller's fp32 Q at
// once and waits for the pre-pass only before its first K tile; the combine
// waits for this kernel (all programmatic dependent launches).
// Every mbarrier wait is bounded; on a timeout a thread records
// kStatusTimeout in the device status word, abandons its loop, and the CTA
// still drains its copies, waits for its MMAs and frees TMEM before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "prefill_tc_common.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int kBN = 128;            // keys per KV tile
constexpr int kStages = 2;          // K/V ring depth
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kGateWarp = 10;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct TcLayout {
    static constexpr uint32_t kBoxes = D / 64;                  // 64 fp16 = 128 B per box row
    static constexpr uint32_t kQTileBytes = kBM * D * 2;
    static constexpr uint32_t kKTileBytes = kBN * D * 2;
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKOff = kQOff + kNQ * kQTileBytes;
    static constexpr uint32_t kVOff = kKOff + kStages * kKTileBytes;
    static constexpr uint32_t kBytes = kVOff + kStages * kKTileBytes;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;        // room to align to 1 KB
    // Epilogue: once every MMA has completed, the K/V ring stages the fp32
    // output tiles for the write-back, as D/32 boxes of 128 rows x 128 bytes
    // (32 floats) in the 128-byte swizzled layout.
    static constexpr uint32_t kOBoxBytes = kBM * 128;
    static constexpr uint32_t kOTileBytes = kBM * D * 4;
    static constexpr uint32_t kStageOff = kKOff;
    static_assert(kStageOff + kNQ * kOTileBytes <= kBytes, "output staging exceeds the K/V ring");
    // Prologue: the two fp32 query tiles (D/32 boxes of 128 rows x 32 floats,
    // 128-byte swizzled) are staged at once, tile 0 in the K ring and tile 1
    // in the V ring, before K and V are first loaded.
    static constexpr uint32_t kQ32Bytes = kBM * D * 4;
    __host__ __device__ static constexpr uint32_t q32_off(int t) { return t == 0 ? kKOff : kVOff; }
    static_assert(kQ32Bytes <= kStages * kKTileBytes, "fp32 query tile exceeds a K/V ring");
};

struct __align__(8) TcBarriers {
    uint64_t q_staged[kNQ];   // fp32 Q tile t landed in the staging area
    uint64_t q_ready[kNQ];    // fp16 Q tile t written (every softmax thread arrives)
    uint64_t k_full[kStages];
    uint64_t k_empty[kStages];
    uint64_t v_full[kStages];
    uint64_t v_empty[kStages];
    uint64_t s_full[kNQ];
    uint64_t p_full[kNQ];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};

__device__ __forceinline__ void record_timeout(unsigned int* status, TcBarriers* bars) {
    atomicOr(status, kStatusTimeout);
    atomicExch(&bars->abort, 1u);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, float* __restrict__ o, uint32_t o_stride,
                  uint32_t m, uint32_t num_q_heads, uint32_t heads_per_kv,
                  float scale_log2, unsigned int* status, uint64_t wait_ns,
                  const SplitArgs split) {
    using L = TcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ TcBarriers bars;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t n_pairs = (m + kNQ * kBM - 1) / (kNQ * kBM);
    const uint32_t h = blockIdx.x % num_q_heads;
    const uint32_t kvh = h / heads_per_kv;
    // Work item: (query-tile pair, KV chunk).  Pairs are walked heaviest
    // first; without a split every pair is one chunk covering all its keys.
    uint32_t pair = 0, chunk = 0, n_chunks = 1;
    if (split.kv_chunk == kNoSplit) {
        pair = n_pairs - 1 - blockIdx.x / num_q_heads;
    } else {
        uint32_t idx = blockIdx.x / num_q_heads;
        for (int p = (int)n_pairs - 1; p >= 0; --p) {
            const uint32_t nk = max(kv_tiles_for(p * kNQ, m, 1), kv_tiles_for(p * kNQ + 1, m, 1));
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
    const uint32_t qt0 = pair * kNQ;                                // first query tile index
    uint32_t n_kv[kNQ];
#pragma unroll
    for (int t = 0; t < kNQ; ++t) n_kv[t] = kv_tiles_for(qt0 + t, m, 1);
    uint32_t n_kv_pair = 0;
#pragma unroll
    for (int t = 0; t < kNQ; ++t) n_kv_pair = max(n_kv_pair, n_kv[t]);
    // This item's KV tiles are [j0, j0 + n_it); tile t takes the first tile_n[t]
    // of them (its causal extent may end inside the chunk).
    const uint32_t j0 = split.kv_chunk == kNoSplit ? 0u : chunk * split.kv_chunk;
    const uint32_t n_kv_all =
        split.kv_chunk == kNoSplit ? n_kv_pair : min(n_kv_pair, j0 + split.kv_chunk) - j0;
    uint32_t tile_n[kNQ];
#pragma unroll
    for (int t = 0; t < kNQ; ++t) tile_n[t] = n_kv[t] > j0 ? min(n_kv[t] - j0, n_kv_all) : 0;

    const uint32_t sQ = smem_u32(smem + L::kQOff);
    const uint32_t sK = smem_u32(smem + L::kKOff);
    const uint32_t sV = smem_u32(smem + L::kVOff);

    if (threadIdx.x == 0) {
        for (int t = 0; t < kNQ; ++t) {
            mbar_init(smem_u32(&bars.q_staged[t]), 1);
            mbar_init(smem_u32(&bars.q_ready[t]), kSoftmaxThreads);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
            mbar_init(smem_u32(&bars.v_full[s]), 1);
            mbar_init(smem_u32(&bars.v_empty[s]), 1);
        }
        for (int t = 0; t < kNQ; ++t) {
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), t == 0 ? kBM + 1 : kBM);  // tile A: + the gate
        }
        mbar_init(smem_u32(&bars.mma_done), 1);
        bars.abort = 0;
        fence_mbar_init();
        // A split's combine kernel may launch now; it waits for this grid.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars.tmem_base), kTmemCols);
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
            prefetch_tmap(&tm_v);
            auto load_q32 = [&](int t) {
                const uint32_t dst = smem_u32(smem + L::q32_off(t));
                mbar_arrive_expect_tx(smem_u32(&bars.q_staged[t]), L::kQ32Bytes);
                for (uint32_t b = 0; b < D / 32; ++b)
                    tma_load_2d(dst + b * L::kOBoxBytes, &tm_q, smem_u32(&bars.q_staged[t]),
                                (int32_t)(h * D + b * 32), (int32_t)((qt0 + t) * kBM));
            };
            auto load_k = [&](uint32_t j) {
                const uint32_t st = j % kStages;
                mbar_arrive_expect_tx(smem_u32(&bars.k_full[st]), L::kKTileBytes);
                for (uint32_t b = 0; b < L::kBoxes; ++b)
                    tma_load_2d(sK + st * L::kKTileBytes + b * (kBN * 128), &tm_k,
                                smem_u32(&bars.k_full[st]), (int32_t)(kvh * D + b * 64),
                                (int32_t)((j0 + j) * kBN));
            };
            auto load_v = [&](uint32_t j) {
                const uint32_t st = j % kStages;
                mbar_arrive_expect_tx(smem_u32(&bars.v_full[st]), L::kKTileBytes);
                for (uint32_t b = 0; b < L::kBoxes; ++b)
                    tma_load_2d(sV + st * L::kKTileBytes + b * (kBN * 128), &tm_v,
                                smem_u32(&bars.v_full[st]), (int32_t)(kvh * D + b * 64),
                                (int32_t)((j0 + j) * kBN));
            };
            // Both query tiles at once; the first K tile as soon as tile 0
            // (staged in the K ring) is converted, V after tile 1.
            uint32_t q_issued = 0, k_issued = 0, v_issued = 0;
            load_q32(0);
            load_q32(1);
            q_issued = 2;
            // The kernel is a programmatic dependent of the rounding pre-pass.
            // Q is the caller's (its writer finished before the pre-pass
            // began), so it is staged at once; the fp16 K and V the pre-pass
            // writes are read only once that grid has completed.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            bool ok = mbar_wait(smem_u32(&bars.q_ready[0]), 0, wait_ns, status, kStatusTimeout);
            if (ok && n_kv_all > 0) {
                load_k(0);
                k_issued = 1;
            }
            if (ok) ok = mbar_wait(smem_u32(&bars.q_ready[1]), 0, wait_ns, status, kStatusTimeout);
            for (uint32_t j = 0; j < n_kv_all && ok; ++j) {
                const uint32_t st = j % kStages;
                const uint32_t use = j / kStages;
                if (j >= k_issued) {
                    if (use > 0) ok = mbar_wait(smem_u32(&bars.k_empty[st]), (use - 1) & 1, wait_ns, status, kStatusTimeout);
                    if (!ok) break;
                    load_k(j);
                    k_issued = j + 1;
                }
                if (use > 0) ok = mbar_wait(smem_u32(&bars.v_empty[st]), (use - 1) & 1, wait_ns, status, kStatusTimeout);
                if (!ok) break;
                load_v(j);
                v_issued = j + 1;
            }
            if (!ok) record_timeout(status, &bars);
            // Drain: every copy this CTA issued must land before it exits.
            for (uint32_t t = 0; t < q_issued; ++t)
                mbar_wait(smem_u32(&bars.q_staged[t]), 0, kDrainWaitNs);
            for (uint32_t j = (k_issued > kStages ? k_issued - kStages : 0); j < k_issued; ++j)
                mbar_wait(smem_u32(&bars.k_full[j % kStages]), (j / kStages) & 1, kDrainWaitNs);
            for (uint32_t j = (v_issued > kStages ? v_issued - kStages : 0); j < v_issued; ++j)
                mbar_wait(smem_u32(&bars.v_full[j % kStages]), (j / kStages) & 1, kDrainWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(BF16 ? 1u : 0u, 0, 0, kBN, kBM);
            const uint32_t idesc_pv = idesc_f16(BF16 ? 1u : 0u, 0, 1, D, kBM);
            bool ok = true;
            for (int t = 0; t < kNQ && ok; ++t)
                ok = mbar_wait(smem_u32(&bars.q_ready[t]), 0, wait_ns, status, kStatusTimeout);
            // Descriptor bases, built once.  A descriptor keeps the start
            // address as (address >> 4) in its low 14 bits, so an operand at
            // byte offset off inside a tile is the tile's descriptor plus
            // off >> 4 (shared-memory offsets stay below 256 KB: no carry).
            // Each MMA below is then one 64-bit add away from issue: building
            // descriptors between MMAs measured at less than half the MMA
            // rate a single issuing thread reaches without it.
            const uint64_t dq0 = smem_desc(sQ, 16, 1024, 2);
            const uint64_t dq1 = smem_desc(sQ + L::kQTileBytes, 16, 1024, 2);
            const uint64_t dk0 = smem_desc(sK, 16, 1024, 2);
            const uint64_t dk1 = smem_desc(sK + L::kKTileBytes, 16, 1024, 2);
            const uint64_t dv0 = smem_desc(sV, kBN * 128, 1024, 2);
            const uint64_t dv1 = smem_desc(sV + L::kKTileBytes, kBN * 128, 1024, 2);
            static_assert(kNQ == 2 && kStages == 2, "descriptor bases assume two tiles and two stages");
            auto issue_s = [&](int t, uint32_t j) {
                const uint64_t a0 = t == 0 ? dq0 : dq1;
                const uint64_t b0 = (j % kStages) == 0 ? dk0 : dk1;
                const uint32_t d = tmem + t * 256;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t offa = (uint64_t)((ks / 4) * (kBM * 128 / 16) + (ks % 4) * 2);
                    const uint64_t offb = (uint64_t)((ks / 4) * (kBN * 128 / 16) + (ks % 4) * 2);
                    mma_f16_ss(d, a0 + offa, b0 + offb, idesc_s, ks > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars.s_full[t]));
            };
            auto issue_pv = [&](int t, uint32_t j) {
                // V tile is MN-major: 64-column boxes are kBN*128 bytes apart
                // (leading byte offset), 8-key groups 1024 bytes apart (stride);
                // K-step ks starts 16 keys (2048 bytes) further on.
                const uint64_t b0 = (j % kStages) == 0 ? dv0 : dv1;
                const uint32_t d = tmem + t * 256 + 128, a = tmem + t * 256;
                const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    mma_f16_ts(d, a + ks * 8, b0 + (uint64_t)(ks * (2048 / 16)), idesc_pv,
                               ks > 0 ? 1u : acc0);
            };
            if (ok && n_kv_all > 0) {
                ok = mbar_wait(smem_u32(&bars.k_full[0]), 0, wait_ns, status, kStatusTimeout);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < kNQ; ++t)
                        if (tile_n[t] > 0) issue_s(t, 0);
                    mma_commit(smem_u32(&bars.k_empty[0]));
                }
            }
            for (uint32_t j = 0; j < n_kv_all && ok; ++j) {
                const uint32_t st = j % kStages;
                const uint32_t jn = j + 1;
                // Tile A's P barrier also carries the gate's word that V(j)
                // and K(j+1) have landed; without tile A the loads are
                // waited for here.
                if (j >= tile_n[0]) {
                    ok = mbar_wait(smem_u32(&bars.v_full[st]), (j / kStages) & 1, wait_ns, status,
                                   kStatusTimeout);
                    if (ok && jn < n_kv_all)
                        ok = mbar_wait(smem_u32(&bars.k_full[jn % kStages]), (jn / kStages) & 1,
                                       wait_ns, status, kStatusTimeout);
                    if (!ok) break;
                    tc_fence_after();
                }
                for (int t = 0; t < kNQ && ok; ++t) {
                    if (j < tile_n[t]) {
                        ok = mbar_wait(smem_u32(&bars.p_full[t]), j & 1, wait_ns, status, kStatusTimeout);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, j);
                    }
                    if (jn < tile_n[t]) issue_s(t, jn);
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars.v_empty[st]));
                if (jn < n_kv_all) mma_commit(smem_u32(&bars.k_empty[jn % kStages]));
            }
            if (!ok) record_timeout(status, &bars);
            // Wait until every MMA this thread issued has completed.
            mma_commit(smem_u32(&bars.mma_done));
            mbar_wait(smem_u32(&bars.mma_done), 0, kDrainWaitNs);
        }
    } else if (warp == kGateWarp) {
        // ------------------------------------------------------------ gate
        if (lane == 0) {
            bool ok = true;
            for (uint32_t j = 0; j < tile_n[0] && ok; ++j) {
                // the phase of step j - 1 completed: this arrival opens step j's
                if (j > 0)
                    ok = mbar_wait(smem_u32(&bars.p_full[0]), (j - 1) & 1, wait_ns, status,
                                   kStatusTimeout);
                if (ok)
                    ok = mbar_wait(smem_u32(&bars.v_full[j % kStages]), (j / kStages) & 1, wait_ns,
                                   status, kStatusTimeout);
                if (ok && j + 1 < n_kv_all)
                    ok = mbar_wait(smem_u32(&bars.k_full[(j + 1) % kStages]), ((j + 1) / kStages) & 1,
                                   wait_ns, status, kStatusTimeout);
                if (!ok) break;
                mbar_arrive(smem_u32(&bars.p_full[0]));
            }
            if (!ok) record_timeout(status, &bars);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int t = warp / 4;                 // query tile of this warpgroup
        const int wq = warp % 4;                // TMEM lane quarter
        const uint32_t row_in_tile = wq * 32 + lane;
        const uint32_t row = (qt0 + t) * kBM + row_in_tile;
        const uint32_t t_s = tmem + t * 256 + ((uint32_t)(wq * 32) << 16);
        const uint32_t t_o = t_s + 128;
        bool ok = true;
        // ---- prologue: round the staged fp32 query tiles to fp16/bf16 into
        // the MMA's 128-byte swizzled K-major layout (all eight warps, one
        // tile after the other: thread = row wq*32+lane, half the columns per
        // warpgroup), checking the fp16 range like the pre-pass does for K, V.
        {
            const uint32_t qr = row_in_tile;             // row converted by this thread
            const uint32_t sw = qr & 7u;

            bool overflow = false;
            for (int tq = 0; tq < kNQ; ++tq) {
                ok = ok && mbar_wait(smem_u32(&bars.q_staged[tq]), 0, wait_ns, status, kStatusTimeout);
                if (ok) {
                    const uint8_t* q32 = smem + L::q32_off(tq);
                    uint8_t* q16 = smem + L::kQOff + tq * L::kQTileBytes;
#pragma unroll
                    for (uint32_t c = (uint32_t)t * (D / 16); c < (uint32_t)(t + 1) * (D / 16); ++c) {
                        // fp16 chunk c = columns 8c..8c+7 = fp32 chunks 2c, 2c+1
                        const uint32_t k0 = 2 * c, k1 = 2 * c + 1;
                        const float4 a = *reinterpret_cast<const float4*>(
                            q32 + (k0 / 8) * L::kOBoxBytes + qr * 128 + (((k0 % 8) ^ sw) * 16));
                        const float4 b = *reinterpret_cast<const float4*>(
                            q32 + (k1 / 8) * L::kOBoxBytes + qr * 128 + (((k1 % 8) ^ sw) * 16));
                        if (!BF16) {
                            const float mx = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                                   fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
                            overflow |= !(mx <= 65504.f);
                        }
                        uint4 out;
                        out.x = pack_half2(a.x, a.y, BF16);
                        out.y = pack_half2(a.z, a.w, BF16);
                        out.z = pack_half2(b.x, b.y, BF16);
                        out.w = pack_half2(b.z, b.w, BF16);
                        *reinterpret_cast<uint4*>(q16 + (c / 8) * (kBM * 128) + qr * 128 +
                                                  (((c % 8) ^ sw) * 16)) = out;
                    }
                }
                // Generic-proxy reads and writes of the staging and of the Q
                // tile are ordered before the next TMA write and the MMAs.
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bars.q_ready[tq]));
            }
            if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(status, kStatusRange);
        }
        float m_used = -CUDART_INF_F;  // log2 units
        float l_sum = 0.f;
        const uint32_t nkv = tile_n[t];
        for (uint32_t j = 0; j < nkv; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full[t]), j & 1, wait_ns, status, kStatusTimeout);
            const bool any_fail = __any_sync(0xffffffffu, !ok);
            if (any_fail) { ok = false; break; }
            tc_fence_after();
            float s[kBN];
            {
                uint32_t r[kBN];
                tmem_ld128_sync(t_s, r);
#pragma unroll
                for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(r[i]);
            }
            if (j0 + j + 1 == n_kv[t]) {  // diagonal tile: keys above the row are not attended
                const uint32_t key0 = (j0 + j) * kBN;
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (key0 + c > row) s[c] = -CUDART_INF_F;
            }
            // Row max as 8 independent chains (a single 128-long chain of
            // dependent max operations would sit on the ping-pong's critical path).
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
            for (int c = 8; c < kBN; ++c) mx8[c % 8] = fmaxf(mx8[c % 8], s[c]);
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_new = mx * scale_log2;
            float corr = 1.f;
            bool rescale = false;
            if (m_new > m_used + kRescaleThreshold) {
                corr = ex2(m_used - m_new);      // 0 on the first tile
                rescale = (j > 0);
                m_used = m_new;
            }
            const float neg_m = -m_used;
            // exponent arguments two at a time (packed fp32x2), row sum as four
            // independent packed accumulators
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nm2 = make_float2(neg_m, neg_m);
            float2 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 x = __ffma2_rn(
                        make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sc2, nm2);
                    const float p0 = ex2(x.x), p1 = ex2(x.y);
                    acc[i % 4] = __fadd2_rn(acc[i % 4], make_float2(p0, p1));
                    pk[i] = pack_half2(p0, p1, BF16);
                }
                tmem_st16(t_s + c * 16, pk);
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
        // ---- epilogue.  After the CTA's last MMA the K/V ring is free: each
        // thread writes its row of O (normalised, or this chunk's unnormalised
        // partial) into the swizzled staging boxes, and each warp then writes
        // the 32 rows it staged back with whole-line stores (rows past m are
        // not written).
        const bool split_item = n_chunks > 1;
        if (ok && nkv > 0) {
            ok = mbar_wait(smem_u32(&bars.mma_done), 0, wait_ns, status, kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) ok = false;
        }
        uint8_t* stage = smem + L::kStageOff + t * L::kOTileBytes;
        if (ok && nkv > 0) {
            tc_fence_after();
            const float scale_o = split_item ? 1.f : 1.0f / l_sum;
            const uint32_t sw = row_in_tile & 7u;
            // the whole row of O in one TMEM load (one wait)
            uint32_t r[D];
            if constexpr (D == 128) {
                tmem_ld128_sync(t_o, r);
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    tmem_ld32(t_o + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
                tmem_wait_ld();
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint8_t* box_row = stage + c * L::kOBoxBytes + row_in_tile * 128;
#pragma unroll
                for (uint32_t q4 = 0; q4 < 8; ++q4) {
                    const uint32_t i = c * 32 + 4 * q4;
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
            __syncwarp();
            const uint32_t tile_row0 = (qt0 + t) * kBM;
            float* dst = split_item
                             ? split.part_o + ((size_t)(chunk * num_q_heads + h) * split.m_pad + tile_row0) * D
                             : o + (size_t)tile_row0 * o_stride + h * D;
            store_warp_rows<D>(stage, L::kOBoxBytes, (uint32_t)wq * 32, min(m - tile_row0, (uint32_t)kBM),
                               dst, split_item ? (size_t)D : (size_t)o_stride, lane);
        }
        if (!ok && lane == 0) record_timeout(status, &bars);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Workspace bytes of the rounded fp16/bf16 K and V (each 256-byte aligned).
size_t operand_bytes_16(uint32_t m, uint32_t num_kv_heads, uint32_t head_dim) {
    return 2 * align256((size_t)m * num_kv_heads * head_dim * 2);
}

template <int D, bool BF16>
cudaError_t launch_tc(const float* q, const float* k, const float* v, float* o, uint32_t m,
                      uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t q_stride,
                      uint32_t kv_stride, float scale, void* workspace, unsigned int* status,
                      uint64_t wait_ns, cudaStream_t stream) {
    using L = TcLayout<D>;
    const PrefillPlan plan = make_plan(m, num_q_heads, D, device_sm_count(), 1, kNQ);
    const size_t operand_bytes = operand_bytes_16(m, num_kv_heads, D);
    const uint32_t q_cols = num_q_heads * D, kv_cols = num_kv_heads * D;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* kh = reinterpret_cast<uint16_t*>(ws);
    uint16_t* vh = reinterpret_cast<uint16_t*>(ws + align256((size_t)m * kv_cols * 2));
    SplitArgs split = plan.split;
    split.part_o = reinterpret_cast<float*>(ws + operand_bytes);
    split.part_ml = reinterpret_cast<float*>(ws + operand_bytes + plan.part_o_bytes);

    {
        const size_t work = (size_t)m * kv_cols / 8;
        const uint32_t threads = 256;
        uint32_t blocks = (uint32_t)std::min<size_t>((work + threads - 1) / threads, 4096);
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(blocks, 2, 1);
        pcfg.blockDim = dim3(threads, 1, 1);
        pcfg.stream = stream;
        pcfg.attrs = pattr;
        pcfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&pcfg, round_operands_kernel<BF16>, k, v, kh, vh, m,
                                           kv_cols, kv_stride, status);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tq, tk, tv;
    if (!encode_output_map(&tq, q, q_cols, m, q_stride, kBM) ||
        !encode_operand_map(&tk, kh, kv_cols, m, kBN, BF16) ||
        !encode_operand_map(&tv, vh, kv_cols, m, kBN, BF16))
        return cudaErrorNotSupported;

    {
        const cudaError_t e = ensure_dynamic_smem<prefill_pair_kernel<D, BF16>>((int)L::kSmemAlloc);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_items * num_q_heads, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemAlloc;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel<D, BF16>, tq, tk, tv, o, q_stride, m,
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

size_t prefill_pair_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                    uint32_t head_dim) {
    const PrefillPlan p = make_plan(m, num_q_heads, head_dim, device_sm_count(), 1, kNQ);
    return operand_bytes_16(m, num_kv_heads, head_dim) + p.part_o_bytes + p.part_ml_bytes;
}

cudaError_t launch_prefill_pair(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, bool bf16, void* workspace, unsigned int* status,
                                uint64_t wait_ns, cudaStream_t stream) {
#define ATTN_TC_CASE(DD)                                                                     \
    if (head_dim == DD) {                                                                    \
        return bf16 ? launch_tc<DD, true>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, \
                                          kv_stride, scale, workspace, status, wait_ns,       \
                                          stream)                                            \
                    : launch_tc<DD, false>(q, k, v, o, m, num_q_heads, num_kv_heads,          \
                                           q_stride, kv_stride, scale, workspace, status,     \
                                           wait_ns, stream);                                 \
    }
    ATTN_TC_CASE(64)
    ATTN_TC_CASE(128)
#undef ATTN_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace attn
