// fa_fwd_bf16.cu -- bf16 (and fp16) attention forward on the Blackwell tensor
// cores.
//
// The loop is the tiled online-softmax forward of "vectorized-flash-
// attention-kernel" (Core algorithm; Key design decisions 1-3) laid out for
// one sm_103a SM:
//
//   * one CTA owns a work item = (batch*head, 256 query rows) split into two
//     128-row query tiles; each tile's scores S = Q K_j^T and output O live in
//     tensor memory (one TMEM lane per query row, fp32);
//   * warp 0 streams Q once and K_j, V_j through a ring of shared-memory slots
//     with TMA (128-byte swizzled boxes of 128 rows x 64 columns; a head
//     dimension below 64 / 128 reads zero-filled columns).  The tiles move in
//     the pairs the MMA warp consumes together, (V_j, K_{j+1}): one barrier
//     signals a pair's arrival and one commit its release;
//   * warp 1 issues the tcgen05.mma products: S_i = Q_i K_j^T (both
//     operands in shared memory) and O_i += P_i V_j (P_i read from tensor
//     memory).  At D = 64, where P_i has TMEM columns of its own, warp 3
//     issues the S products instead, as soon as the softmax warps hold the
//     previous S_i in registers, so S_i(j+1) is computed while they work on
//     block j and the two products of a tile come from two threads (one
//     thread issues at most one N=128 product per ~90-100 clk on this GPU;
//     two keep the tensor core at its 64 clk rate);
//   * warps 4-7 and 8-11 run the online softmax of tile 0 and tile 1: each
//     thread loads its row of S_i from TMEM, masks, updates the running max m
//     and sum l, writes P_i = exp2(S*scale*log2e - m) as bf16 back into TMEM
//     (over S_i at D = 128, into P_i's own columns at D = 64), and rescales
//     O_i in TMEM when the max moved;
//   * while one tile's softmax runs, the tensor core works on the other tile,
//     so the two softmax warpgroups alternate with the MMAs;
//   * at the end each tile's warps stage O (16-bit) in the tile's Q buffer and
//     one thread writes it with TMA stores (split-KV partials, fp32, are
//     stored by the threads).
//
// The one-tile kernel (fa_fwd_onetile.cu) serves D = 256 and small grids;
// both share the per-row softmax step of fa_fwd_softmax.cuh.
//
// The reference max is lazy: after the first key block it moves only when a
// block's sum of p exceeds 2^64, so almost every block needs no max scan and
// no O rescale; l and O always share the reference, which keeps the result
// exact in real arithmetic, and P <= 2^64 stays far inside fp32/bf16 range.
//
// Causal key blocks that lie wholly after the item's last query row are never
// loaded (Key design decisions 3); key blocks at or past the key length are
// skipped too, and items whose key length is 0 write O = 0, LSE = -inf
// without touching the tensor core ("js-flash-attention-tiled-online-softmax-
// exactness", Root causes 2).
//
// Every mbarrier wait is bounded by a time budget; a wait that runs out sets
// the library's device status word, raises a CTA-wide abort flag, and every
// role then drains its in-flight copies / MMAs, frees tensor memory and exits.
#include "fa_fwd_softmax.cuh"
#include "fa_internal.h"
#include "fa_tc_common.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {

__device__ uint32_t g_status;

namespace {

constexpr int BM = 128;          // query rows per tile (= TMEM lanes)
constexpr int BN = 128;          // keys per step
constexpr int kThreads = 384;    // 12 warps
constexpr int kFirstSoftmaxWarp = 4;
// setmaxnreg split: the control warpgroup's and the softmax warpgroups'
// registers per thread, which must fit the block's launch allocation (384
// threads x 168) or setmaxnreg.inc would wait forever.
constexpr int kRegsControl = 96;
constexpr int kRegsSoftmax = 200;
// P apart (D = 64): chunks of 32 scores a softmax thread exponentiates before
// it waits for the previous PV product and stores P.
constexpr int kEarlyChunks = 2;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * ((65536 / kThreads) / 8 * 8), "register split");

template <int D>
struct Layout {
    static constexpr int kChunks = D / 64;            // 128-byte swizzle atoms per row
    static constexpr int kChunkBytes = BM * 128;      // one 128 x 64 bf16 box
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kSlots = (D == 64) ? 8 : 4;  // K/V ring depth (K_j, V_j alternate)
    // K/V tiles move in pairs (V_{m-1}, K_m) -- "pair m"; K_0 alone is pair
    // 0 and V of the last block alone the last pair.  Pair m fills the slots
    // of pair m - kPairs, so each pair has one "full" and one "empty"
    // barrier, used round-robin over kPairs.
    static constexpr int kPairs = kSlots / 2;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 after it.
    // At D = 128 P_i (16-bit pairs) overwrites the first 64 columns of S_i.
    // At D = 64 the O tiles leave 128 columns free and P_i has 64 of its own
    // (kPApart): O_i += P_i V_j and S_i = Q_i K_{j+1}^T then touch disjoint
    // columns, and two threads issue them side by side (see the MMA roles).
    static constexpr bool kPApart = (D == 64);
    __device__ static constexpr uint32_t col_s(int i) { return (uint32_t)i * 128u; }
    __device__ static constexpr uint32_t col_o(int i) { return 256u + (uint32_t)i * D; }
    __device__ static constexpr uint32_t col_p(int i) { return kPApart ? 384u + (uint32_t)i * 64u : col_s(i); }
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!kPApart || 256 + 2 * D + 2 * 64 <= (int)kTmemCols, "P tiles of their own");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert((1 + 2 * kPairs + 12) * 8 + 8 <= kBarBytes, "barrier area");
};


template <int D, bool kSplit, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const FwdParams p, const int q_pairs)
{
    using Lay = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *q_full = bars;
    // The MMA warp consumes K/V as pairs: P V_j and the S_{j+1} = Q K_{j+1}^T
    // issued right after it read (V_j, K_{j+1}) -- pair j+1 -- and the last
    // products over that pair are issued in the same iteration.  So a pair
    // arrives together (pair_full) and is released together (pair_empty).
    uint64_t *pair_full = bars + 1;                   // [kPairs]
    uint64_t *pair_empty = pair_full + Lay::kPairs;   // [kPairs]
    uint64_t *s_full = pair_empty + Lay::kPairs;   // [2]
    uint64_t *p_full = s_full + 2;                 // [2]
    uint64_t *o_final = p_full + 2;                // [2]
    uint64_t *mma_drain = o_final + 2;
    // P apart (D = 64) only: PV_i of a block done (its P columns may be
    // rewritten, O_i rescaled); S_i of a block loaded into the softmax
    // warps' registers (its columns may be rewritten); the drain of the
    // second MMA thread.
    uint64_t *pv_done = mma_drain + 1;             // [2]
    uint64_t *s_read = pv_done + 2;                // [2]
    uint64_t *mma_drain_s = s_read + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_drain_s + 1);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);
    const Abort ab{abort_word, &g_status};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: heaviest causal items first --------------------------
    // (split-KV: the num_splits CTAs of one item are adjacent and each takes a
    // contiguous range of its key blocks)
    const int64_t BH = p.B * p.H;
    const int splits = kSplit ? p.num_splits : 1;
    const int64_t item = (int64_t)blockIdx.x / splits;
    const int split = (int)((int64_t)blockIdx.x % splits);
    const int64_t pair = (int64_t)q_pairs - 1 - item / BH;
    const int64_t bh = item % BH;
    const int64_t b = bh / p.H;
    const int64_t N = p.N;
    const int64_t q0 = pair * (2 * BM);
    int64_t L = N;
    if (p.kv_len) {
        L = p.kv_len[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    const int64_t kv_end = p.causal ? (L < q0 + 2 * BM ? L : q0 + 2 * BM) : L;
    const int n_all = (int)((kv_end + BN - 1) / BN);
    const int blk0 = kSplit ? (int)((int64_t)n_all * split / splits) : 0;   // first key block of this CTA
    const int n_kv = kSplit ? (int)((int64_t)n_all * (split + 1) / splits) - blk0 : n_all;

    // ---- set-up -----------------------------------------------------------
    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        for (int s = 0; s < Lay::kPairs; ++s) {
            ptx::mbar_init(&pair_full[s], 1);
            // with two MMA threads, each releases every pair once
            ptx::mbar_init(&pair_empty[s], Lay::kPApart ? 2 : 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 4);          // one arrival per softmax warp
            ptx::mbar_init(&o_final[i], 1);
            ptx::mbar_init(&pv_done[i], 1);
            ptx::mbar_init(&s_read[i], 4);          // one arrival per softmax warp
        }
        ptx::mbar_init(mma_drain, 1);
        ptx::mbar_init(mma_drain_s, 1);
        *abort_word = 0;
        ptx::fence_mbarrier_init();
        // Thread 0 is also the producer: the item's Q tiles and K_0 (pair 0)
        // are requested now, so that their latency overlaps the TMEM
        // allocation and the CTA-wide barrier below.
        if (n_kv > 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::mbar_arrive_expect_tx(q_full, 2 * Lay::kTileBytes);
            for (int i = 0; i < 2; ++i)
                for (int c = 0; c < Lay::kChunks; ++c)
                    ptx::tma_load_3d(smem + Lay::kQOff + i * Lay::kTileBytes + c * Lay::kChunkBytes,
                                     &tm_q, q_full, c * 64, (int32_t)(q0 + i * BM), (int32_t)bh);
            ptx::mbar_arrive_expect_tx(&pair_full[0], Lay::kTileBytes);
            for (int c = 0; c < Lay::kChunks; ++c)
                ptx::tma_load_3d(smem + Lay::kKVOff + c * Lay::kChunkBytes, &tm_k, &pair_full[0], c * 64,
                                 (int32_t)(blk0 * BN), (int32_t)bh);
        }
    }
    // An item with no visible key only writes O = 0 and LSE = -inf: it needs
    // no tensor memory.
    if (warp == 1 && n_kv > 0) {
        ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = n_kv > 0 ? *tmem_slot : 0u;

    // Registers: the producer / MMA warpgroup needs few; the softmax
    // warpgroups hold a 128-column score row each.  128*96 + 256*200 fits in
    // the 384*168 registers the CTA is launched with.  Each setmaxnreg sits
    // in the branch of the role it serves.
    if (warp < kFirstSoftmaxWarp) {
    ptx::regs_dec<kRegsControl>();
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0 && n_kv > 0) {
            // Q and pair 0 (K_0 alone) were requested before the CTA-wide
            // barrier.  Pair m (0 <= m <= n_kv) holds V_{m-1} in slot 2m-1 and
            // K_m in slot 2m (mod kSlots); from m = kPairs on, those slots are
            // the ones of pair m - kPairs, which the MMA warp must have released.
            int pairs_armed = 1;    // pairs 0 .. pairs_armed-1 have had their copies issued
            for (int m = 1; m <= n_kv; ++m) {
                if (m >= Lay::kPairs) {
                    const int pm = m - Lay::kPairs;
                    if (!wait_bounded(&pair_empty[pm % Lay::kPairs], (pm / Lay::kPairs) & 1, p.wait_limit_ns,
                                      kSiteSlotEmpty, ab))
                        break;
                }
                const bool has_v = m >= 1, has_k = m < n_kv;
                uint64_t *bar = &pair_full[m % Lay::kPairs];
                ptx::mbar_arrive_expect_tx(bar, (uint32_t)(has_v + has_k) * Lay::kTileBytes);
                for (int w = has_v ? 1 : 0; w >= (has_k ? 0 : 1); --w) {   // V_{m-1}, then K_m
                    const int slot = (2 * m - w) % Lay::kSlots;
                    const int blk = m - w;
                    const CUtensorMap *tm = w ? &tm_v : &tm_k;
                    for (int c = 0; c < Lay::kChunks; ++c)
                        ptx::tma_load_3d(smem + Lay::kKVOff + slot * Lay::kTileBytes + c * Lay::kChunkBytes,
                                         tm, bar, c * 64, (int32_t)((blk0 + blk) * BN), (int32_t)bh);
                }
                pairs_armed = m + 1;
            }
            // Drain: no copy may still be landing in shared memory at exit.
            wait_bounded(q_full, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            for (int m = pairs_armed > Lay::kPairs ? pairs_armed - Lay::kPairs : 0; m < pairs_armed; ++m)
                wait_bounded(&pair_full[m % Lay::kPairs], (m / Lay::kPairs) & 1, p.wait_limit_ns, kSiteDrain,
                             ab, false);
        }
    } else if (warp == 1 || (Lay::kPApart && warp == 3)) {
        // ================= MMA issuers =================
        // D = 128: warp 1 issues every product, PV_0(j), S_0(j+1), PV_1(j),
        // S_1(j+1) in turn, which keeps S_i(j+1) behind the PV_i(j) that
        // reads the P columns it overwrites.  D = 64 (P apart): warp 1 issues
        // the PV products and warp 3 the S products.  The two streams share no
        // TMEM columns, and two issuing threads keep the tensor core busier
        // than one: a probe on this GPU ran one thread's N=128 products at
        // ~110 clk each and two threads' at ~70 clk per product together.
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_qk = make_idesc(BM, BN, 0, 0, kF16);
            constexpr uint32_t idesc_pv = make_idesc(BM, D, 0, 1, kF16);
            const uint32_t q_base = ptx::smem_u32(smem + Lay::kQOff);
            const uint32_t kv_base = ptx::smem_u32(smem + Lay::kKVOff);

            // The start-address field of a descriptor is the byte address / 16,
            // and every operand lies below 256 KiB, so moving an operand by a
            // byte offset moves its descriptor by offset / 16: the descriptors
            // are built once here, and each K-step adds a constant.
            const uint64_t q_desc = make_sdesc(q_base, 16, 1024);            // K-major Q tiles
            const uint64_t k_desc = make_sdesc(kv_base, 16, 1024);           // K-major K slots
            const uint64_t v_desc = make_sdesc(kv_base, Lay::kChunkBytes, 1024);   // MN-major V slots
            constexpr uint64_t kTileStep = Lay::kTileBytes >> 4;
            auto issue_s = [&](int i, int slot) {
                const uint64_t qd = q_desc + (uint64_t)i * kTileStep;
                const uint64_t kd = k_desc + (uint64_t)slot * kTileStep;
                const uint32_t ts = tmem + Lay::col_s(i);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * Lay::kChunkBytes + (k % 4) * 32) >> 4);
                    ptx::mma_ss(ts, qd + off, kd + off, idesc_qk, k > 0);
                }
            };
            auto issue_pv = [&](int i, int slot, uint32_t acc) {
                const uint64_t vd = v_desc + (uint64_t)slot * kTileStep;
                const uint32_t to = tmem + Lay::col_o(i), tp = tmem + Lay::col_p(i);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ts(to, tp + k * 8, vd + (uint64_t)((k * 2048) >> 4), idesc_pv, (acc | (uint32_t)k) != 0);
            };

            if constexpr (!Lay::kPApart) {
                bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab) &&
                          wait_bounded(&pair_full[0], 0, p.wait_limit_ns, kSiteSlotFull, ab);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s(0, 0);
                    ptx::mma_commit(&s_full[0]);
                    issue_s(1, 0);
                    ptx::mma_commit(&s_full[1]);
                    ptx::mma_commit(&pair_empty[0]);      // K_0 is read
                }
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int slot_v = (2 * j + 1) % Lay::kSlots, slot_k = (2 * j + 2) % Lay::kSlots;
                    const bool more = (j + 1 < n_kv);
                    // pair j+1: V_j, and K_{j+1} when there is a next block
                    if (!wait_bounded(&pair_full[(j + 1) % Lay::kPairs], ((j + 1) / Lay::kPairs) & 1,
                                      p.wait_limit_ns, kSiteSlotFull, ab) ||
                        !wait_bounded(&p_full[0], j & 1, p.wait_limit_ns, kSitePFull, ab))
                        break;
                    ptx::tc_fence_after();
                    issue_pv(0, slot_v, j > 0);
                    if (!more) ptx::mma_commit(&o_final[0]);
                    if (more) {
                        issue_s(0, slot_k);
                        ptx::mma_commit(&s_full[0]);
                    }
                    if (!wait_bounded(&p_full[1], j & 1, p.wait_limit_ns, kSitePFull, ab)) break;
                    ptx::tc_fence_after();
                    issue_pv(1, slot_v, j > 0);
                    if (!more) ptx::mma_commit(&o_final[1]);
                    if (more) {
                        issue_s(1, slot_k);
                        ptx::mma_commit(&s_full[1]);
                    }
                    ptx::mma_commit(&pair_empty[(j + 1) % Lay::kPairs]);   // V_j and K_{j+1} are read
                }
            } else if (warp == 1) {
                // PV products.  Pair 0 (K_0 alone) has nothing for them.
                ptx::mma_commit(&pair_empty[0]);
                for (int j = 0; j < n_kv; ++j) {
                    const int slot_v = (2 * j + 1) % Lay::kSlots;
                    bool ok = wait_bounded(&pair_full[(j + 1) % Lay::kPairs], ((j + 1) / Lay::kPairs) & 1,
                                           p.wait_limit_ns, kSiteSlotFull, ab);
                    for (int i = 0; i < 2 && ok; ++i) {
                        ok = wait_bounded(&p_full[i], j & 1, p.wait_limit_ns, kSitePFull, ab);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_pv(i, slot_v, j > 0);
                        ptx::mma_commit(&pv_done[i]);
                        if (j + 1 == n_kv) ptx::mma_commit(&o_final[i]);
                    }
                    if (!ok) break;
                    ptx::mma_commit(&pair_empty[(j + 1) % Lay::kPairs]);   // V_j is read
                }
            } else {
                // S products: S_i(j+1) may overwrite S_i(j) as soon as tile
                // i's softmax warps hold S_i(j) in registers, so it is
                // computed while they work on block j.
                bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab) &&
                          wait_bounded(&pair_full[0], 0, p.wait_limit_ns, kSiteSlotFull, ab);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s(0, 0);
                    ptx::mma_commit(&s_full[0]);
                    issue_s(1, 0);
                    ptx::mma_commit(&s_full[1]);
                    ptx::mma_commit(&pair_empty[0]);      // K_0 is read
                }
                for (int j = 0; j < n_kv && ok; ++j) {
                    if (j + 1 < n_kv) {
                        const int slot_k = (2 * j + 2) % Lay::kSlots;
                        ok = wait_bounded(&pair_full[(j + 1) % Lay::kPairs], ((j + 1) / Lay::kPairs) & 1,
                                          p.wait_limit_ns, kSiteSlotFull, ab);
                        for (int i = 0; i < 2 && ok; ++i) {
                            ok = wait_bounded(&s_read[i], j & 1, p.wait_limit_ns, kSiteSFull, ab);
                            if (!ok) break;
                            ptx::tc_fence_after();
                            issue_s(i, slot_k);
                            ptx::mma_commit(&s_full[i]);
                        }
                        if (!ok) break;
                    }
                    ptx::mma_commit(&pair_empty[(j + 1) % Lay::kPairs]);   // K_{j+1} is read
                }
            }
            // Drain: every MMA this thread issued is complete before TMEM is
            // freed (on the normal path o_final already covered them; after an
            // abort some may still be in flight).
            uint64_t *drain = (Lay::kPApart && warp == 3) ? mma_drain_s : mma_drain;
            ptx::mma_commit(drain);
            wait_bounded(drain, 0, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        // ================= online softmax + epilogue =================
        const int i = (warp - kFirstSoftmaxWarp) / 4;      // query tile of this warpgroup
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter ..
        const int r_local = quarter * 32 + lane;
        const int64_t row = q0 + i * BM + r_local;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + Lay::col_s(i);
        const uint32_t tO = tmem + lane_off + Lay::col_o(i);
        const uint32_t tP = tmem + lane_off + Lay::col_p(i);
        const int64_t lim = p.causal ? (L < row + 1 ? L : row + 1) : L;   // visible keys: j < lim
        const float sl2 = p.scale_log2;

        OnlineRow<D, kF16> st;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const bool got = wait_bounded(&s_full[i], j & 1, p.wait_limit_ns, kSiteSFull, ab);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t s_raw[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, s_raw[c]);
            ptx::tmem_wait_ld();
            if constexpr (Lay::kPApart) {
                // S_i(j) is in registers: its columns are free for S_i(j+1)
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&s_read[i]);
            }

            const int64_t vis = lim - (int64_t)(blk0 + j) * BN;   // columns k < vis are visible
            if (vis < BN) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (c * 32 + t >= vis) s_raw[c][t] = f2u(-INFINITY);
            }
            if constexpr (!Lay::kPApart) {
                // O_i is never being written here: s_full[i] for block j is
                // committed after PV_i of block j-1.
                st.block(s_raw, sl2, j > 0, tP, tO, [] {});
            } else {
                // PV_i(j-1) runs on the other MMA thread and may still read
                // P_i and write O_i: it has to end before the first P store
                // and before any access to O.
                auto pv_prev = [&] {
                    if (j > 0) {
                        const bool done = wait_bounded(&pv_done[i], (j - 1) & 1, p.wait_limit_ns, kSitePFull, ab);
                        if (!__all_sync(0xffffffffu, done)) ok = false;
                        ptx::tc_fence_after();
                    }
                };
                st.block<kEarlyChunks>(s_raw, sl2, j > 0, tP, tO, pv_prev, pv_prev);
                if (!ok) break;
            }
            // every lane's P stores have landed (block() waited for them);
            // after the warp has synchronised, one lane tells the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[i]);
        }
        const float l = st.l, l_o = st.l_o, m_ref = st.m_ref;

        // ---- epilogue: O = acc / l_o, LSE = (m + log2 l) ln 2 --------------
        bool have = (n_kv > 0) && ok;
        if (have) have = wait_bounded(&o_final[i], 0, p.wait_limit_ns, kSiteOFinal, ab);
        // the tile's four warps agree, so that its named barrier below is
        // reached by all of them or by none
        have = ptx::bar_and(1 + i, 128, have);
        if (have || n_kv == 0) {
            ptx::tc_fence_after();
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l_o;      // O / (sum of the P the MMA used)
            const float lse_row = empty ? -INFINITY : (m_ref + log2f(l)) * 0.69314718055994530942f;
            // Only the first p.D (a multiple of 8, <= D) columns exist in
            // memory; the rest of the D computed ones are the zero padding.
            const int Dv = (int)p.D;
            const int64_t flat = bh * N + row;
            if constexpr (kSplit) {
                float *prow = p.part_o + ((int64_t)split * BH * N + flat) * Dv;
#pragma unroll 1
                for (int c = 0; c < D / 32 && c * 32 < Dv; ++c) {
                    uint32_t o[32];
                    if (n_kv > 0) {
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_wait_ld();
                    }
                    if (row < N) {
                        float f[32];
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            float lo, hi;
                            ptx::unpack2(ptx::mul2(ptx::pack2(u2f(o[2 * t]), u2f(o[2 * t + 1])),
                                                   ptx::pack2(inv, inv)), lo, hi);
                            f[2 * t] = empty ? 0.f : lo;
                            f[2 * t + 1] = empty ? 0.f : hi;
                        }
                        // normalised fp32 partial output of this key range
                        float4 *dst = reinterpret_cast<float4 *>(prow + c * 32);
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            if (c * 32 + 4 * t < Dv)
                                dst[t] = make_float4(f[4 * t], f[4 * t + 1], f[4 * t + 2], f[4 * t + 3]);
                    }
                }
            } else {
                // O = acc / l_o as 16-bit, staged in this tile's Q buffer (free:
                // every MMA has completed) as 128-byte-swizzled 128 x 64 boxes,
                // then written by TMA stores that clip rows >= N and columns
                // >= p.D.
                uint8_t *obuf = smem + Lay::kQOff + i * Lay::kTileBytes;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (n_kv > 0) {
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_wait_ld();
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float lo = 0.f, hi = 0.f;
                        if (n_kv > 0)
                            ptx::unpack2(ptx::mul2(ptx::pack2(u2f(o[2 * t]), u2f(o[2 * t + 1])), ptx::pack2(inv, inv)),
                                         lo, hi);
                        w[t] = empty ? 0u : ptx::pack16x2<kF16>(lo, hi);
                    }
                    // 32 columns = 4 of the 8 16-byte units of a 64-column box row
                    const uint32_t row_addr = ptx::smem_u32(obuf + (c / 2) * Lay::kChunkBytes + r_local * 128);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t unit = (uint32_t)((c % 2) * 4 + u) ^ (uint32_t)(r_local & 7);
                        ptx::st_shared_v4(row_addr + (unit << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::bar_sync(1 + i, 128);                 // this tile's four warps
                if (r_local == 0) {
                    for (int c = 0; c < Lay::kChunks; ++c)
                        ptx::tma_store_3d(&tm_o, obuf + c * Lay::kChunkBytes, c * 64, (int32_t)(q0 + i * BM),
                                          (int32_t)bh);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read<0>();       // the boxes have left shared memory
                }
            }
            if (row < N) {
                if (kSplit)
                    p.part_lse[(int64_t)split * BH * N + flat] = lse_row;
                else if (p.lse)
                    p.lse[flat] = lse_row;
            }
        }
    }
    // ---- teardown ----------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1 && n_kv > 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

template <int D, bool kSplit, bool kF16>
cudaError_t launch_d(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, const CUtensorMap &to, cudaStream_t stream)
{
    using Lay = Layout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D, kSplit, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int q_pairs = (int)((p.N + 2 * BM - 1) / (2 * BM));
    const int64_t ctas = p.B * p.H * (int64_t)q_pairs * (kSplit ? p.num_splits : 1);
    fwd_bf16_kernel<D, kSplit, kF16><<<(unsigned)ctas, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, to, p,
                                                                                           q_pairs);
    return cudaGetLastError();
}

// Merge of the split-KV partial states ("FlashAttention" module, Math: partial
// softmax states merge associatively).  Partial s of a row carries its
// normalised output O_s and LSE_s over its key range; with m = max_s LSE_s and
// w_s = exp(LSE_s - m): O = sum_s w_s O_s / sum_s w_s, LSE = m + ln sum_s w_s.
// Ranges with no visible key have LSE_s = -inf and weight 0; a row with none
// at all gets O = +0 and LSE = -inf.  One warp per row, D/32 columns per lane
// (D = the padded head dimension; lanes past the Dv real columns only help
// with the LSE).
template <int D, bool kF16>
__global__ void __launch_bounds__(256)
merge_splits_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                    uint16_t *__restrict__ out, float *__restrict__ lse, int64_t rows, int splits,
                    int Dv)
{
    constexpr int kPer = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const bool cols = lane * kPer < Dv;   // Dv is a multiple of 8: a lane's columns are all in or all out
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, part_lse[(int64_t)s * rows + row]);
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    if (m > -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float ls = part_lse[(int64_t)s * rows + row];
            if (!(ls > -INFINITY)) continue;
            const float w = expf(ls - m);
            wsum += w;
            if (!cols) continue;
            const float *src = part_o + ((int64_t)s * rows + row) * Dv + lane * kPer;
            if constexpr (kPer == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
                acc[2] = fmaf(w, v.z, acc[2]);
                acc[3] = fmaf(w, v.w, acc[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
            }
        }
    }
    const bool empty = !(wsum > 0.f);
    const float inv = empty ? 0.f : 1.f / wsum;
    uint32_t packed[kPer / 2];
#pragma unroll
    for (int c = 0; c < kPer / 2; ++c)
        packed[c] = empty ? 0u : ptx::pack16x2<kF16>(acc[2 * c] * inv, acc[2 * c + 1] * inv);
    uint16_t *dst = out + row * Dv + lane * kPer;
    if (cols) {
        if constexpr (kPer == 4)
            *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
        else
            *reinterpret_cast<uint32_t *>(dst) = packed[0];
    }
    if (lse && lane == 0) lse[row] = empty ? -INFINITY : m + logf(wsum);
}

template <int D, bool kF16>
cudaError_t launch_split(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, cudaStream_t stream)
{
    cudaError_t e = launch_d<D, true, kF16>(p, tq, tk, tv, tq, stream);   // tq: no O map is read
    if (e != cudaSuccess) return e;
    const int64_t rows = p.B * p.H * p.N;
    merge_splits_kernel<D, kF16><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        p.part_o, p.part_lse, static_cast<uint16_t *>(p.o), p.lse, rows, p.num_splits, (int)p.D);
    return cudaGetLastError();
}

}  // namespace

// A head dimension D that is a multiple of 8 runs in the kernel for the next
// of 64 / 128: the TMA boxes (64 columns) fill the columns past D with zeros,
// which leaves every score unchanged, and the padded output columns are never
// stored.
cudaError_t launch_fwd_bf16(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream)
{
    if (p.D % 8 != 0 || p.D <= 0 || p.D > 128) return cudaErrorInvalidValue;
    if (p.D <= 64)
        return p.f16 ? launch_d<64, false, true>(p, tm_q, tm_k, tm_v, tm_o, stream)
                     : launch_d<64, false, false>(p, tm_q, tm_k, tm_v, tm_o, stream);
    return p.f16 ? launch_d<128, false, true>(p, tm_q, tm_k, tm_v, tm_o, stream)
                 : launch_d<128, false, false>(p, tm_q, tm_k, tm_v, tm_o, stream);
}

cudaError_t launch_fwd_bf16_split(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                  const CUtensorMap &tm_v, cudaStream_t stream)
{
    if (p.f16) return cudaErrorInvalidValue;   // the split-KV path is bf16 only
    if (p.D % 8 != 0 || p.D <= 0 || p.D > 128) return cudaErrorInvalidValue;
    if (p.D <= 64) return launch_split<64, false>(p, tm_q, tm_k, tm_v, stream);
    return launch_split<128, false>(p, tm_q, tm_k, tm_v, stream);
}

cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *out)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    uint32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace fa
