// prefill_tc.cu -- causal grouped-query prefill on the Blackwell tensor cores
// (tcgen05 MMAs with TMEM accumulators, TMA-staged tiles), one kernel for the
// three operand types: fp16, bf16 (kind::f16) and TF32 (kind::tf32).
//
// Operation ("aprender-gpu 0.32.0 -- prefill_fused.rs", module doc,
// Algorithm 1-3): for query head h and KV head g = h / heads_per_kv, row i
// of O is sum_{j<=i} softmax_j(scale * Q[i].K[j]) V[j], with an online
// softmax.  The page does this with one warp per head on CUDA cores; here
// the two contractions (S = Q K^T and O += P V) run on the tensor core, and
// the softmax statistics (row max, row sum) and the output stay fp32.
//
// Precision.  fp16 / bf16: Q, K, V are rounded to nearest (K and V by a
// pre-pass into a workspace, Q by the softmax warps as they move it into
// TMEM); P is rounded to nearest as the softmax packs it; fp16 inputs must
// stay below 65504 (kStatusRange otherwise, after the fact).  TF32: a
// kind::tf32 MMA uses the top 19 bits of each fp32 operand (the low 13
// mantissa bits are dropped), so every operand is rounded to nearest TF32
// first: Q by the softmax warps as they move it into TMEM, K and V by the
// pre-pass.  An operand dropped toward zero would bias the output (O = V[0]
// exactly for row 0), which rounding to nearest halves and unbiases.  P is truncated to TF32 by
// the softmax itself and the row sum is taken over the truncated weights, so
// the weights the MMA applies are normalised exactly (a row sum over the
// untruncated weights would scale every output down by up to 2^-10 where the
// running max lags the row's largest score).
//
// Layout.  16-bit: the pre-pass writes K and V rounded, [m, kv_heads*D];
// S reads K K-major and P.V reads V MN-major (keys are the K dimension, D is
// contiguous).  TF32 MMAs take only K-major operands, so the pre-pass writes
// V rounded and transposed per KV head, [kv_heads*D, m4] fp32 (keys
// contiguous, m4 = m rounded up to 4).
//
// CTA work unit: one 128-row query tile of one head; keys are walked in
// 128-key steps up to the diagonal.  With S double-buffered in TMEM the
// tensor core computes S(j+1) and P(j-1).V while the softmax works on S(j),
// so a single tile keeps it busy.  TMEM (512 columns): S/P buffers 0 and 1
// (128 columns each; 16-bit P is packed in pairs over the first 64), O (D
// columns) and the query tile (D columns in TF32, D/2 packed 16-bit pairs;
// the S MMA takes A from TMEM, so shared memory feeds it only K).  Shared
// memory holds only a ring of seven 32 KB slots: a K or V tile is one piece
// (16-bit) or D/64 pieces (TF32) of at most 32 KB, loaded in the order the
// MMAs consume them: K(0), K(1), V(0), K(2), V(1), K(3), ...  The MMA thread
// issues S(0), S(1), then per step j: P(j).V, then S(j+2) into the buffer
// P(j) occupied (MMAs execute in issue order, so S(j+2) overwrites P(j)
// after P(j).V has read it).  With one piece per tile a slot is reused once
// the S that follows its tile's MMAs has completed (every tcgen05.commit
// between MMAs costs the tensor pipe); with two, a K slot once its own S has
// completed, a V slot by a commit right after the P.V MMAs that read it.
// Warp roles (224 threads): warps 0-3 softmax (thread = TMEM lane = query
// row), warp 4 TMA producer, warp 5 TMEM allocator and MMA issuer, warp 6
// gate.  An mbarrier wait on the issuing thread stalls the tensor pipe even
// when the phase has already completed (about 26 ns each, measured), so the
// MMA thread waits once per step: on go(j), which the 128 softmax threads
// complete with P(j) and the gate thread with the slots of V(j) and K(j+2)
// (the gate waits for each slot's load in turn).
// The softmax rescales O only when the running max grows by more than 8
// (log2 units); it then first waits for the previous P.V (O stable).
// Epilogue: O (normalised, or a chunk's unnormalised partial) into the ring's
// first slots, then each warp writes its 32 rows back with whole-line
// stores.  Small grids split each tile's key walk into chunks merged by the
// combine kernel.
// Launch chain (programmatic dependent launches): the pre-pass waits for the
// kernel before the call, then lets this kernel launch; this kernel stages
// the caller's Q at once and waits for the pre-pass before its first K/V
// load; the combine waits for this kernel.
// Every mbarrier wait is bounded; on a timeout a thread records
// kStatusTimeout, abandons its loop, and the CTA still drains its copies,
// waits for its MMAs and frees TMEM before exiting.
// 16-bit grids of at least two waves of query-tile pairs run the pair kernel
// of prefill_tc_pair.cu instead (prefill_use_pairs below), whose loads and
// hand-offs each serve twice the MMAs; TF32 calls always run this kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdint>

#include "attn_internal.h"
#include "prefill_tc_common.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

enum class Op : int { FP16 = 0, BF16 = 1, TF32 = 2 };

constexpr int kBK = 128;               // keys per step
constexpr uint32_t kPerQ = kBM / kBK;  // key tiles per 128-key block (1)
constexpr int kSlots = 7;              // operand ring slots
constexpr uint32_t kSlotBytes = 32 * 1024;
constexpr int kSoftmaxThreads = 128;   // warps 0-3
constexpr int kThreads = 224;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kGateWarp = 6;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTf32Mask = 0xFFFFE000u;  // the bits of an fp32 a TF32 operand keeps
constexpr uint32_t kBoxBytes = kBK * 128;    // 128 rows x 128 bytes, 128-byte swizzled

template <int D, Op OP>
struct TcLayout {
    static constexpr bool k16 = OP != Op::TF32;
    static constexpr uint32_t kElem = k16 ? 2 : 4;
    static constexpr uint32_t kBoxElems = 128 / kElem;               // elements per box row
    static constexpr uint32_t kTileBytes = kBK * D * kElem;          // one K or V tile
    static constexpr int kPieces = kTileBytes > kSlotBytes ? (int)(kTileBytes / kSlotBytes) : 1;
    static constexpr uint32_t kPieceBytes = kTileBytes / kPieces;
    static constexpr int kKBoxesPerPiece = (int)(D * kElem / 128) / kPieces;  // D-column boxes
    // 16-bit V: boxes of 64 D-columns x 128 keys; TF32 V^T: boxes of 32 keys x D rows.
    static constexpr uint32_t kVBoxBytes = k16 ? kBoxBytes : D * 128;
    static constexpr int kVBoxesPerPiece = k16 ? kKBoxesPerPiece : 4 / kPieces;
    static constexpr int kSSteps = (int)(D * kElem / 32) / kPieces;  // S MMAs per K piece (32 B of K each)
    static constexpr int kVSteps = k16 ? kBK / 16 : kBK / 8 / kPieces;  // P.V MMAs per V piece
    static constexpr uint32_t kQ32Bytes = kBM * D * 4;               // fp32 query or output tile
    static constexpr int kQSlots = (int)(kQ32Bytes / kSlotBytes);
    static constexpr int kQStageSlot = kSlots - kQSlots;
    static constexpr uint32_t kBytes = kSlots * kSlotBytes;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;            // room to align to 1 KB
    static constexpr uint32_t kOCol = 2 * kBK;                       // TMEM: S0 | S1 | O | Q
    static constexpr uint32_t kQCol = kOCol + D;
    static constexpr uint32_t kQCols = k16 ? D / 2 : D;
    static_assert(kQCol + kQCols <= kTmemCols, "TMEM layout");
    static_assert(kPieceBytes <= kSlotBytes && kPieces * kPieceBytes == kTileBytes, "pieces");
    static_assert(kKBoxesPerPiece * kBoxBytes == kPieceBytes, "K piece");
    static_assert(kVBoxesPerPiece * kVBoxBytes == kPieceBytes, "V piece");
    static_assert(kQSlots * kSlotBytes == kQ32Bytes, "query staging");
    static_assert(kSmemAlloc <= 227 * 1024, "shared memory");
    // One piece per tile: the ring holds seven tiles, so a slot can wait to
    // be released by the completion of the next S (no release commits).  Two
    // pieces per tile (TF32 at D = 128) leave 3.5 tiles, and a slot must be
    // released as soon as its own MMAs complete: a K slot by its S's
    // completion, a V slot by a commit after its P.V.
    static constexpr bool kReleaseByS = kPieces == 1;
};

struct __align__(8) TcBarriers {
    uint64_t q_full;        // the fp32 query tile landed in the staging slots
    uint64_t q_ready;       // the query tile is in TMEM (every softmax thread arrives)
    uint64_t full[kSlots];
    uint64_t empty[kSlots];  // a V piece's P.V completed (two-piece tiles only)
    uint64_t s_full[4];      // S(j) computed, by step j % 4 (its buffer is j % 2)
    uint64_t go[2];         // step j % 2: P(j) written and the slots of V(j), K(j+2) loaded
    uint64_t pv_last;       // P.V of the second-to-last step completed (one phase)
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};

__device__ __forceinline__ void record_timeout(unsigned int* status, TcBarriers* bars) {
    atomicOr(status, kStatusTimeout);
    atomicExch(&bars->abort, 1u);
}

template <Op OP>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    if constexpr (OP == Op::TF32)
        mma_tf32_ts(d, a, b, idesc, accumulate);
    else
        mma_f16_ts(d, a, b, idesc, accumulate);
}

template <int D, Op OP>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, float* __restrict__ o, uint32_t o_stride,
                  uint32_t m, uint32_t num_q_heads, uint32_t heads_per_kv,
                  float scale_log2, unsigned int* status, uint64_t wait_ns,
                  const SplitArgs split) {
    using L = TcLayout<D, OP>;
    constexpr bool k16 = L::k16;
    constexpr bool kBf16 = OP == Op::BF16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ TcBarriers bars;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t n_qt = (m + kBM - 1) / kBM;
    const uint32_t h = blockIdx.x % num_q_heads;
    const uint32_t kvh = h / heads_per_kv;
    // Work item: (query tile, key chunk), heaviest tiles first.
    uint32_t qt = 0, chunk = 0, n_chunks = 1;
    if (split.kv_chunk == kNoSplit) {
        qt = n_qt - 1 - blockIdx.x / num_q_heads;
    } else {
        uint32_t idx = blockIdx.x / num_q_heads;
        for (int t = (int)n_qt - 1; t >= 0; --t) {
            const uint32_t nc = (kv_tiles_for(t, m, kPerQ) + split.kv_chunk - 1) / split.kv_chunk;
            if (idx < nc) {
                qt = (uint32_t)t;
                chunk = idx;
                n_chunks = nc;
                break;
            }
            idx -= nc;
        }
    }
    const uint32_t n_kv_tile = kv_tiles_for(qt, m, kPerQ);
    // This item's key steps are [j0, j0 + nkv).
    const uint32_t j0 = split.kv_chunk == kNoSplit ? 0u : chunk * split.kv_chunk;
    const uint32_t nkv =
        split.kv_chunk == kNoSplit ? n_kv_tile : min(n_kv_tile, j0 + split.kv_chunk) - j0;
    const uint32_t tile_row0 = qt * kBM;

    const uint32_t sR = smem_u32(smem);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars.q_full), 1);
        mbar_init(smem_u32(&bars.q_ready), kSoftmaxThreads);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(smem_u32(&bars.full[s]), 1);
            mbar_init(smem_u32(&bars.empty[s]), 1);
        }
        for (int b = 0; b < 4; ++b) mbar_init(smem_u32(&bars.s_full[b]), 1);
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&bars.go[b]), kSoftmaxThreads + 1);
        mbar_init(smem_u32(&bars.pv_last), 1);
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

    // Loads of the item, in the order the MMAs consume them: K(0), K(1),
    // then V(i) and K(i + 2) alternately.  Unit u is one tile; load n is
    // piece n % kPieces of unit n / kPieces.
    const uint32_t n_units = nkv > 0 ? 2 * nkv : 0;
    auto unit_of = [&](uint32_t u, bool& is_k, uint32_t& step) {
        if (u < 2 && u < nkv) { is_k = true; step = u; return; }
        // after K(0) and K(1): V(i) at 2 + 2i (with K(i+2) at 3 + 2i while i + 2 < nkv);
        // once the keys run out, the remaining units are V tiles only
        const uint32_t first_v = nkv < 2 ? nkv : 2u;
        const uint32_t r = u - first_v;
        const uint32_t paired = nkv > 2 ? nkv - 2 : 0u;  // V(i) followed by K(i+2) for i < paired
        if (r < 2 * paired) {
            is_k = (r & 1u) != 0;
            step = is_k ? r / 2 + 2 : r / 2;
        } else {
            is_k = false;
            step = paired + (r - 2 * paired);
        }
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            {
                const uint32_t bar = smem_u32(&bars.q_full);
                mbar_arrive_expect_tx(bar, L::kQ32Bytes);
                for (uint32_t b = 0; b < D / 32; ++b)
                    tma_load_2d(sR + L::kQStageSlot * kSlotBytes + b * kBoxBytes, &tm_q, bar,
                                (int32_t)(h * D + b * 32), (int32_t)tile_row0);
            }
            // K and V come from the pre-pass: read them only once its grid
            // (and with it every kernel before the call) has completed.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const uint32_t n_loads = n_units * L::kPieces;
            uint32_t issued = 0;
            // Two-piece tiles: per slot, the parity of the V pieces loaded
            // into it so far (its release barrier completes once per V piece).
            uint32_t v_parity = 0;
            bool ok = true;
            for (uint32_t n = 0; n < n_loads; ++n) {
                const uint32_t slot = n % kSlots, use = n / kSlots;
                bool prev_k = false;
                uint32_t prev_step = 0;
                if (use > 0) unit_of((n - kSlots) / L::kPieces, prev_k, prev_step);
                if (use > 0 && !L::kReleaseByS && prev_k) {
                    // A K tile's slots are free once its S has completed
                    // (S(x + 4) needs K(x + 4), not issued yet: the wait is
                    // exact).
                    ok = mbar_wait(smem_u32(&bars.s_full[prev_step & 3u]), (prev_step >> 2) & 1,
                                   wait_ns, status, kStatusTimeout);
                } else if (use > 0 && L::kReleaseByS) {
                    // The slot's previous tile has been read once S(x)
                    // completed: S(i) for K(i), and for V(i) the S(i + 2)
                    // issued right after P(i).V (a V tile with no later S is
                    // among the last loads, whose slots are never reused).
                    // The witnesses never decrease, and S(x + 4) needs
                    // K(x + 4), not issued yet: each parity wait is exact.
                    bool was_k;
                    uint32_t was_step;
                    unit_of((n - kSlots) / L::kPieces, was_k, was_step);
                    const uint32_t x = was_k ? was_step : was_step + 2;
                    ok = mbar_wait(smem_u32(&bars.s_full[x & 3u]), (x >> 2) & 1, wait_ns, status,
                                   kStatusTimeout);
                } else if (use > 0) {
                    // a V piece: released by the commit after its P.V MMAs
                    ok = mbar_wait(smem_u32(&bars.empty[slot]), ((v_parity >> slot) & 1u) ^ 1u,
                                   wait_ns, status, kStatusTimeout);
                } else if (slot >= (uint32_t)L::kQStageSlot) {
                    // the query staging slots are free once the tile is in TMEM
                    ok = mbar_wait(smem_u32(&bars.q_ready), 0, wait_ns, status, kStatusTimeout);
                }
                if (!ok) break;
                bool is_k;
                uint32_t step;
                unit_of(n / L::kPieces, is_k, step);
                if (!is_k) v_parity ^= 1u << slot;
                const uint32_t piece = n % L::kPieces;
                const uint32_t bar = smem_u32(&bars.full[slot]);
                const uint32_t dst = sR + slot * kSlotBytes;
                const uint32_t key0 = (j0 + step) * kBK;
                mbar_arrive_expect_tx(bar, L::kPieceBytes);
                if (is_k) {
                    for (int b = 0; b < L::kKBoxesPerPiece; ++b)
                        tma_load_2d(dst + b * kBoxBytes, &tm_k, bar,
                                    (int32_t)(kvh * D + (piece * L::kKBoxesPerPiece + b) * L::kBoxElems),
                                    (int32_t)key0);
                } else if constexpr (k16) {
                    for (int b = 0; b < L::kVBoxesPerPiece; ++b)
                        tma_load_2d(dst + b * kBoxBytes, &tm_v, bar,
                                    (int32_t)(kvh * D + b * L::kBoxElems), (int32_t)key0);
                } else {
                    for (int b = 0; b < L::kVBoxesPerPiece; ++b)
                        tma_load_2d(dst + b * L::kVBoxBytes, &tm_v, bar,
                                    (int32_t)(key0 + (piece * L::kVBoxesPerPiece + b) * 32),
                                    (int32_t)(kvh * D));
                }
                issued = n + 1;
            }
            if (!ok) record_timeout(status, &bars);
            // Drain: every copy this CTA issued must land before it exits.
            mbar_wait(smem_u32(&bars.q_full), 0, kDrainWaitNs);
            for (uint32_t n = (issued > kSlots ? issued - kSlots : 0); n < issued; ++n)
                mbar_wait(smem_u32(&bars.full[n % kSlots]), (n / kSlots) & 1, kDrainWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kAb = kBf16 ? 1u : 0u;
            constexpr uint32_t idesc_s = k16 ? idesc_f16(kAb, 0, 0, kBK, kBM) : idesc_tf32(kBK, kBM);
            constexpr uint32_t idesc_pv = k16 ? idesc_f16(kAb, 0, 1, D, kBM) : idesc_tf32(D, kBM);
            bool ok = nkv == 0 ||
                      mbar_wait(smem_u32(&bars.q_ready), 0, wait_ns, status, kStatusTimeout);
            // Slot descriptors: the ring's base plus slot * 32 KB (>> 4).  A
            // K step (32 bytes: 16 halves or 8 fp32) sits (ks % 4) * 32 bytes
            // into a 128-byte swizzled row, in box ks / 4 of its piece.  The
            // 16-bit V tile is MN-major: its 64-column boxes are 16 KB apart
            // (leading byte offset), 8-key groups 1024 bytes (stride), and a
            // K step of 16 keys starts 2048 bytes further on.
            const uint64_t dk0 = smem_desc(sR, 16, 1024, 2);
            const uint64_t dv0 = k16 ? smem_desc(sR, kBoxBytes, 1024, 2) : dk0;
            uint32_t load = 0;  // next load the MMAs consume
            // S(0) and S(1) wait for their slots here; every later slot is
            // covered by the go barrier of its step.
            auto take = [&](uint32_t& slot, bool wait) {
                slot = load % kSlots;
                const bool got = !wait || mbar_wait(smem_u32(&bars.full[slot]), (load / kSlots) & 1,
                                                    wait_ns, status, kStatusTimeout);
                ++load;
                if (got && wait) tc_fence_after();
                return got;
            };
            auto issue_s = [&](uint32_t j) {
                const uint32_t d = tmem + (j & 1u) * kBK;
                for (int p = 0; p < L::kPieces; ++p) {
                    uint32_t slot;
                    if (!take(slot, j < 2)) return false;
                    const uint64_t b0 = dk0 + (uint64_t)(slot * (kSlotBytes / 16));
#pragma unroll
                    for (int ks = 0; ks < L::kSSteps; ++ks) {
                        const int k = p * L::kSSteps + ks;  // 32 bytes of the D columns per MMA
                        mma_ts<OP>(d, tmem + L::kQCol + k * 8,
                                   b0 + (uint64_t)((ks / 4) * (kBoxBytes / 16) + (ks % 4) * 2),
                                   idesc_s, k > 0 ? 1u : 0u);
                    }
                }
                mma_commit(smem_u32(&bars.s_full[j & 3u]));
                return true;
            };
            auto issue_pv = [&](uint32_t j) {
                const uint32_t a = tmem + (j & 1u) * kBK, d = tmem + L::kOCol;
                for (int p = 0; p < L::kPieces; ++p) {
                    uint32_t slot;
                    take(slot, false);
                    const uint64_t b0 = dv0 + (uint64_t)(slot * (kSlotBytes / 16));
#pragma unroll
                    for (int ks = 0; ks < L::kVSteps; ++ks) {
                        const int k = p * L::kVSteps + ks;  // 16 (16-bit) or 8 (TF32) keys per MMA
                        const uint64_t boff =
                            k16 ? (uint64_t)(ks * (2048 / 16))
                                : (uint64_t)((ks / 4) * (L::kVBoxBytes / 16) + (ks % 4) * 2);
                        mma_ts<OP>(d, a + k * 8, b0 + boff, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                    }
                    if (!L::kReleaseByS) mma_commit(smem_u32(&bars.empty[slot]));
                }
                // The last step's softmax rescales O only after this group
                // (S(j+2), whose completion tells the other steps, does not exist).
                if (j + 2 == nkv) mma_commit(smem_u32(&bars.pv_last));
            };
            if (ok && nkv > 0) ok = issue_s(0);
            if (ok && nkv > 1) ok = issue_s(1);
            for (uint32_t j = 0; j < nkv && ok; ++j) {
                ok = mbar_wait(smem_u32(&bars.go[j & 1u]), (j >> 1) & 1, wait_ns, status,
                               kStatusTimeout);
                if (!ok) break;
                tc_fence_after();
                issue_pv(j);
                if (j + 2 < nkv) issue_s(j + 2);
            }
            if (!ok) record_timeout(status, &bars);
            // Wait until every MMA this thread issued has completed.
            mma_commit(smem_u32(&bars.mma_done));
            mbar_wait(smem_u32(&bars.mma_done), 0, kDrainWaitNs);
        }
    } else if (warp == kGateWarp) {
        // ------------------------------------------------------------ gate
        // Step j's MMAs read the loads of V(j), then those of K(j+2), in
        // load order; S(0) and S(1) took the first ones.  go(j) reuses the
        // barrier of step j - 2, whose phase must complete first (its P
        // arrivals precede this step's, so none can land in the old phase).
        // A slot's parity wait is exact only once the slot's previous load
        // has landed: the gate checks every load after those of S(0) and
        // S(1) itself, and first waits for S(0) and S(1) to complete, which
        // the MMA thread issued only after their loads had landed (with two
        // pieces per tile, K(2)'s second piece reuses the slot of K(0)'s
        // first, and a wait for it could otherwise pass on the earlier phase).
        if (lane == 0) {
            uint32_t load = (uint32_t)L::kPieces * min(nkv, 2u);
            bool ok = true;
            for (uint32_t j = 0; j < nkv && ok; ++j) {
                if (j >= 2)
                    ok = mbar_wait(smem_u32(&bars.go[j & 1u]), ((j - 2) >> 1) & 1, wait_ns, status,
                                   kStatusTimeout);
                else
                    ok = mbar_wait(smem_u32(&bars.s_full[j]), 0, wait_ns, status, kStatusTimeout);
                const uint32_t n = (uint32_t)L::kPieces * (j + 2 < nkv ? 2u : 1u);
                for (uint32_t i = 0; i < n && ok; ++i, ++load)
                    ok = mbar_wait(smem_u32(&bars.full[load % kSlots]), (load / kSlots) & 1, wait_ns,
                                   status, kStatusTimeout);
                if (!ok) break;
                mbar_arrive(smem_u32(&bars.go[j & 1u]));
            }
            if (!ok) record_timeout(status, &bars);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const uint32_t row_in_tile = warp * 32 + lane;
        const uint32_t row = tile_row0 + row_in_tile;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t t_o = lane_base + L::kOCol;
        const uint32_t sw = row_in_tile & 7u;
        bool ok = true;
        // ---- prologue: the query row from the fp32 staging boxes into TMEM
        // (16-bit: rounded and packed in pairs, fp16 range checked).
        if (nkv > 0) {
            ok = mbar_wait(smem_u32(&bars.q_full), 0, wait_ns, status, kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) ok = false;
            if (ok) {
                const uint8_t* stage = smem + L::kQStageSlot * kSlotBytes;
                bool overflow = false;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    const uint8_t* box_row = stage + c * kBoxBytes + row_in_tile * 128;
#pragma unroll
                    for (uint32_t q4 = 0; q4 < 8; ++q4) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(box_row + ((q4 ^ sw) * 16));
                        r[4 * q4] = v4.x;
                        r[4 * q4 + 1] = v4.y;
                        r[4 * q4 + 2] = v4.z;
                        r[4 * q4 + 3] = v4.w;
                    }
                    if constexpr (k16) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a = __uint_as_float(r[2 * i]), b = __uint_as_float(r[2 * i + 1]);
                            if (!kBf16) overflow |= !(fmaxf(fabsf(a), fabsf(b)) <= 65504.f);
                            pk[i] = pack_half2(a, b, kBf16);
                        }
                        tmem_st16(lane_base + L::kQCol + c * 16, pk);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(round_tf32(__uint_as_float(r[i])));
                        tmem_st32(lane_base + L::kQCol + c * 32, r);
                    }
                }
                tmem_wait_st();
                if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(status, kStatusRange);
            }
            // The staging reads come before the TMA writes that reuse the
            // slots, the TMEM stores before the MMAs that read them.
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.q_ready));
        }
        float m_used = -CUDART_INF_F;  // log2 units
        float l_sum = 0.f;
        for (uint32_t j = 0; j < nkv && ok; ++j) {
            const uint32_t buf = j & 1u;
            ok = mbar_wait(smem_u32(&bars.s_full[j & 3u]), (j >> 2) & 1, wait_ns, status,
                           kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t_s = lane_base + buf * kBK;
            float s[kBK];
            {
                uint32_t r[kBK];
                tmem_ld128_sync(t_s, r);
#pragma unroll
                for (int i = 0; i < kBK; ++i) s[i] = __uint_as_float(r[i]);
            }
            const uint32_t key0 = (j0 + j) * kBK;
            if (key0 + kBK > tile_row0) {  // the diagonal block: keys above the row are not attended
#pragma unroll
                for (int c = 0; c < kBK; ++c)
                    if (key0 + c > row) s[c] = -CUDART_INF_F;
            }
            // Row max as 8 independent chains.
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
                corr = ex2(m_used - m_new);      // 0 on the first step
                rescale = (j > 0);
                m_used = m_new;
            }
            // A row with no attended key so far (every score -inf) keeps its
            // weights at exactly 0 instead of forming -inf - (-inf).
            const float neg_m = m_used == -CUDART_INF_F ? 0.f : -m_used;
            // exponent arguments two at a time (packed fp32x2), row sum as four
            // independent packed accumulators
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nm2 = make_float2(neg_m, neg_m);
            float2 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBK / 32; ++c) {
                if constexpr (k16) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 x = __ffma2_rn(
                            make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sc2, nm2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        acc[i % 4] = __fadd2_rn(acc[i % 4], make_float2(p0, p1));
                        pk[i] = pack_half2(p0, p1, kBf16);
                    }
                    tmem_st16(t_s + c * 16, pk);
                } else {
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
            }
            const float rowsum = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                                 ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
            l_sum = fmaf(l_sum, corr, rowsum);
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds every P.V up to step j-1 once P.V(j-1) has completed:
                // S(j+1) was issued right after it, and the last step has its
                // own barrier.  (Waiting on S(j+1) here consumes the same phase
                // the next step waits for.)
                ok = j + 1 < nkv ? mbar_wait(smem_u32(&bars.s_full[(j + 1) & 3u]), ((j + 1) >> 2) & 1,
                                             wait_ns, status, kStatusTimeout)
                                 : mbar_wait(smem_u32(&bars.pv_last), 0, wait_ns, status,
                                             kStatusTimeout);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                tc_fence_after();
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
            mbar_arrive(smem_u32(&bars.go[buf]));
        }
        // ---- epilogue: O (normalised, or this chunk's unnormalised partial)
        // into the ring's first slots; each warp then writes the 32 rows it
        // staged back with whole-line stores.
        const bool split_item = n_chunks > 1;
        if (ok && nkv > 0) {
            ok = mbar_wait(smem_u32(&bars.mma_done), 0, wait_ns, status, kStatusTimeout);
            if (__any_sync(0xffffffffu, !ok)) ok = false;
        }
        uint8_t* stage = smem;
        if (ok && nkv > 0) {
            tc_fence_after();
            const float scale_o = split_item ? 1.f : 1.0f / l_sum;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32_sync(t_o + c * 32, r);
                uint8_t* box_row = stage + c * kBoxBytes + row_in_tile * 128;
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
            __syncwarp();
            float* dst = split_item
                             ? split.part_o + ((size_t)(chunk * num_q_heads + h) * split.m_pad + tile_row0) * D
                             : o + (size_t)tile_row0 * o_stride + h * D;
            store_warp_rows<D>(stage, kBoxBytes, (uint32_t)warp * 32, min(m - tile_row0, (uint32_t)kBM),
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

// TF32 pre-pass: K rounded to nearest TF32 into kr [m, kv_cols] (grid.y = 0,
// eight elements per thread), and V rounded and transposed into
// vt [kv_cols, m4] (grid.y = 1, 32 x 32 tiles through shared memory: rows of
// V in, rows of V^T out, both as whole 128-byte lines).
__global__ void __launch_bounds__(256)
round_transpose_tf32_kernel(const float* __restrict__ k, const float* __restrict__ v,
                            float* __restrict__ kr, float* __restrict__ vt, uint32_t m,
                            uint32_t kv_cols, uint32_t kv_stride, uint32_t m4) {
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

__global__ void wait_timeout_selftest_kernel(unsigned int* status, uint64_t wait_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Nothing ever arrives on this barrier: the bounded wait must give up.
    if (!mbar_wait(smem_u32(&bar), 0, wait_ns, status, kStatusTimeout)) atomicOr(status, kStatusTimeout);
}

// Workspace: the rounded K and V (TF32: K rounded, V rounded and transposed
// with rows of m4 keys), each 256-byte aligned, then the split partials.
struct OperandBytes {
    size_t k_bytes, v_bytes;
    uint32_t m4;
};

OperandBytes operand_bytes(uint32_t m, uint32_t num_kv_heads, uint32_t head_dim, bool tf32) {
    OperandBytes w{};
    w.m4 = (m + 3) / 4 * 4;
    const size_t elem = tf32 ? 4 : 2;
    w.k_bytes = align256((size_t)m * num_kv_heads * head_dim * elem);
    w.v_bytes = tf32 ? align256((size_t)num_kv_heads * head_dim * w.m4 * 4) : w.k_bytes;
    return w;
}

template <int D, Op OP>
cudaError_t launch_tc(const float* q, const float* k, const float* v, float* o, uint32_t m,
                      uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t q_stride,
                      uint32_t kv_stride, float scale, void* workspace, unsigned int* status,
                      uint64_t wait_ns, cudaStream_t stream) {
    using L = TcLayout<D, OP>;
    constexpr bool kTf32 = OP == Op::TF32;
    const PrefillPlan plan = make_plan(m, num_q_heads, D, device_sm_count(), kPerQ, 1);
    const OperandBytes w = operand_bytes(m, num_kv_heads, D, kTf32);
    const uint32_t q_cols = num_q_heads * D, kv_cols = num_kv_heads * D;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* kw = ws;
    void* vw = ws + w.k_bytes;
    SplitArgs split = plan.split;
    split.part_o = reinterpret_cast<float*>(ws + w.k_bytes + w.v_bytes);
    split.part_ml = reinterpret_cast<float*>(ws + w.k_bytes + w.v_bytes + plan.part_o_bytes);

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        const size_t k_work = (size_t)m * kv_cols / 8;
        const size_t v_work = kTf32 ? (size_t)((m + 31) / 32) * (kv_cols / 32) : 0;
        const uint32_t blocks =
            (uint32_t)std::min<size_t>(std::max<size_t>((k_work + 255) / 256, v_work), 4096);
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(blocks, 2, 1);
        pcfg.blockDim = dim3(256, 1, 1);
        pcfg.stream = stream;
        pcfg.attrs = attr;
        pcfg.numAttrs = 1;
        cudaError_t e;
        if constexpr (kTf32)
            e = cudaLaunchKernelEx(&pcfg, round_transpose_tf32_kernel, k, v,
                                   static_cast<float*>(kw), static_cast<float*>(vw), m, kv_cols,
                                   kv_stride, w.m4);
        else
            e = cudaLaunchKernelEx(&pcfg, round_operands_kernel<OP == Op::BF16>, k, v,
                                   static_cast<uint16_t*>(kw), static_cast<uint16_t*>(vw), m,
                                   kv_cols, kv_stride, status);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tq, tk, tv;
    bool maps = encode_output_map(&tq, q, q_cols, m, q_stride, kBM);
    if constexpr (kTf32)
        maps = maps && encode_output_map(&tk, kw, kv_cols, m, kv_cols, kBK) &&
               encode_output_map(&tv, vw, m, kv_cols, w.m4, D);
    else
        maps = maps && encode_operand_map(&tk, kw, kv_cols, m, kBK, OP == Op::BF16) &&
               encode_operand_map(&tv, vw, kv_cols, m, kBK, OP == Op::BF16);
    if (!maps) return cudaErrorNotSupported;
    {
        const cudaError_t e = ensure_dynamic_smem<prefill_tc_kernel<D, OP>>((int)L::kSmemAlloc);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_items * num_q_heads, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemAlloc;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, OP>, tq, tk, tv, o, q_stride, m,
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

template <Op OP>
cudaError_t launch_d(const float* q, const float* k, const float* v, float* o, uint32_t m,
                     uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                     uint32_t q_stride, uint32_t kv_stride, float scale, void* workspace,
                     unsigned int* status, uint64_t wait_ns, cudaStream_t stream) {
    if (head_dim == 128)
        return launch_tc<128, OP>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                  scale, workspace, status, wait_ns, stream);
    if (head_dim == 64)
        return launch_tc<64, OP>(q, k, v, o, m, num_q_heads, num_kv_heads, q_stride, kv_stride,
                                 scale, workspace, status, wait_ns, stream);
    return cudaErrorInvalidValue;
}

size_t workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                       uint32_t head_dim, bool tf32) {
    const PrefillPlan p = make_plan(m, num_q_heads, head_dim, device_sm_count(), kPerQ, 1);
    const OperandBytes w = operand_bytes(m, num_kv_heads, head_dim, tf32);
    return w.k_bytes + w.v_bytes + p.part_o_bytes + p.part_ml_bytes;
}

}  // namespace

// Pairs of query tiles halve the loads and hand-offs per MMA, single tiles
// balance a small grid better: pairs once they fill the SMs twice over.
bool prefill_use_pairs(uint32_t m, uint32_t num_q_heads, int sm_count) {
    const uint64_t pairs = (m + 2 * kBM - 1) / (2 * kBM);
    return pairs * num_q_heads >= 2 * (uint64_t)std::max(sm_count, 1);
}

size_t prefill_tc_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                  uint32_t head_dim) {
    if (prefill_use_pairs(m, num_q_heads, device_sm_count()))
        return prefill_pair_workspace_bytes(m, num_q_heads, num_kv_heads, head_dim);
    return workspace_bytes(m, num_q_heads, num_kv_heads, head_dim, false);
}

size_t prefill_tf32_workspace_bytes(uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                    uint32_t head_dim) {
    return workspace_bytes(m, num_q_heads, num_kv_heads, head_dim, true);
}

cudaError_t launch_prefill_tc(const float* q, const float* k, const float* v, float* o,
                              uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                              uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                              float scale, bool bf16, void* workspace, unsigned int* status,
                              uint64_t wait_ns, cudaStream_t stream) {
    if (prefill_use_pairs(m, num_q_heads, device_sm_count()))
        return launch_prefill_pair(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                   kv_stride, scale, bf16, workspace, status, wait_ns, stream);
    return bf16 ? launch_d<Op::BF16>(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                     kv_stride, scale, workspace, status, wait_ns, stream)
                : launch_d<Op::FP16>(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                                     kv_stride, scale, workspace, status, wait_ns, stream);
}

cudaError_t launch_prefill_tf32(const float* q, const float* k, const float* v, float* o,
                                uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                                uint32_t head_dim, uint32_t q_stride, uint32_t kv_stride,
                                float scale, void* workspace, unsigned int* status,
                                uint64_t wait_ns, cudaStream_t stream) {
    return launch_d<Op::TF32>(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim, q_stride,
                              kv_stride, scale, workspace, status, wait_ns, stream);
}

cudaError_t launch_wait_timeout_selftest(unsigned int* status, uint64_t limit_ns) {
    wait_timeout_selftest_kernel<<<1, 32>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace attn
