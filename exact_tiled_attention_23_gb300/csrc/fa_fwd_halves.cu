// fa_fwd_halves.cu -- bf16 / fp16 attention forward on the tensor cores with
// one 128-row query tile per CTA and each row's keys split between two
// softmax warpgroups.
//
// The computation is the tiled online-softmax forward of "vectorized-flash-
// attention-kernel" (Core algorithm; Key design decisions 1-3).  Each key
// block of 128 keys is split into two halves of 64: warps 4-7 run the online
// softmax of every row over the first half of every block, warps 8-11 over
// the second half.  The two halves of a row are two independent online
// softmax states: each keeps its own reference max m, sums l and l_o, and its
// own output accumulator O_h += P_h V_h in TMEM.  They meet once, in the
// epilogue, through the associative merge of partial softmax states
// ("FlashAttention" module, Math): with m = max(m_A, m_B) and
// w_h = 2^(m_h - m), O = (w_A O_A + w_B O_B) / (w_A l_oA + w_B l_oB) and
// LSE = (m + log2(w_A l_A + w_B l_B)) ln 2.  This is exact in real
// arithmetic, like the per-row recurrence it replaces.
//
// Why split rows: the softmax step of a block has a chain of short waits
// (the score hand-off, the P hand-off, the TMEM load and store waits) of
// ~90-150 clk each on this GPU.  With one softmax warp per SM sub-partition
// nothing hides them; with two, one computes while the other waits, and each
// has half the scores of a block to process.
//
// On the SM:
//   * TMEM (512 columns): one score tile S [0,128); two P tiles of 64
//     columns (P for block j goes to tile j % 2; half h writes its 32
//     columns at 32h); O_A and O_B, D columns each.
//   * warp 0 streams Q once and K_t, V_t through rings of kRing slots each
//     (K_0, K_1, V_0, K_2, V_1, ...), as the one-tile kernel does;
//   * warp 3 issues S_{j+1} = Q K_{j+1}^T into the score tile as soon as all
//     eight softmax warps hold S_j in registers (s_read), so the scores of the
//     next block are computed while the softmax works on this one;
//   * warp 1 issues O_h += P_h(j) V_j[64h .. 64h+63] (four K=16 products per
//     half) when half h hands P_h(j) over.  Two issuing threads keep the
//     tensor core busier than one can (one thread issues at most one N=128
//     product per ~90-100 clk on this GPU, two reach the 64 clk rate);
//   * the softmax of half h stores P_h(j) into P tile j % 2 after
//     O_h += P_h(j-2) V_{j-2}, its last reader, is done, and rescales O_h
//     (when its lazy reference moves) after O_h += P_h(j-1) V_{j-1} is done.
//
// Causal key blocks wholly after the tile's last query row are never loaded;
// key blocks at or past the key length are skipped, and a tile with no
// visible key writes O = 0, LSE = -inf without touching the tensor core
// ("js-flash-attention-tiled-online-softmax-exactness", Root causes 2).
//
// Every mbarrier wait is bounded; a wait that runs out records the site in
// this file's status word, raises the CTA's abort flag, and every role drains
// its copies / MMAs, frees TMEM and exits.
#include "fa_fwd_softmax.cuh"
#include "fa_internal.h"
#include "fa_tc_common.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {

__device__ uint32_t g_status_halves;

namespace {

constexpr int BM = 128;                   // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;                   // keys per block
constexpr int kHalf = 64;                 // keys of a block per softmax warpgroup
constexpr int kThreads = 384;             // warp 0 TMA, warps 1 and 3 MMA, warps 4-11 softmax
constexpr int kSoftmaxWarp0 = 4;
constexpr int kChunkBytes = 128 * 128;    // one 128-row x 64-column 16-bit box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;             // S [0,128)
constexpr uint32_t kColP = 128;           // P tiles [128,192), [192,256)
constexpr uint32_t kColO = 256;           // O_A [256,256+D), O_B after it

template <int D>
struct HalvesLayout {
    static constexpr int kChunks = D / 64;                      // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = kChunks * kChunkBytes;    // Q, a K or a V tile
    // K and V slots each.  At D = 128 two measured ~1 % faster than three
    // (the S thread consumes K two blocks ahead at most, and a V slot is
    // refilled once both halves' products of its block are done).
    static constexpr int kRing = D == 128 ? 2 : 4;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kTileBytes;
    static constexpr int kVOff = kKOff + kRing * kTileBytes;
    static constexpr int kBarOff = kVOff + kRing * kTileBytes;
    // q_full, k_full/k_empty/v_full/v_empty [R], s_full, s_read, p_full[2][2],
    // pv_done[2][2], o_final, mma_drain, mma_drain_s
    static constexpr int kBars = 1 + 4 * kRing + 2 + 4 + 4 + 3;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;       // + alignment slack
    __device__ static constexpr uint32_t col_o(int h) { return kColO + (uint32_t)(h * D); }
    __device__ static constexpr uint32_t col_p(int buf, int h) { return kColP + (uint32_t)(buf * 64 + h * 32); }
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(kColO + 2 * D <= kTmemCols, "TMEM columns");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kBars * 8 + 8 <= 256, "barrier area");
    // the epilogue's exchange of (m, l, l_o) uses the first V slot
    static_assert(2 * BM * 3 * 4 <= kTileBytes, "exchange area");
};

template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_halves_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p, const int q_tiles)
{
    using Lay = HalvesLayout<D>;
    constexpr int kChunks = Lay::kChunks, kTileBytes = Lay::kTileBytes, R = Lay::kRing;
    constexpr int kQOff = Lay::kQOff, kKOff = Lay::kKOff, kVOff = Lay::kVOff;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;               // [R]
    uint64_t *k_empty = k_full + R;            // [R]
    uint64_t *v_full = k_empty + R;            // [R]
    uint64_t *v_empty = v_full + R;            // [R]
    uint64_t *s_full = v_empty + R;            // S_j complete
    uint64_t *s_read = s_full + 1;             // all softmax warps hold S_j in registers (8 arrivals)
    uint64_t *p_full = s_read + 1;             // [half][P tile]: P_h(j) stored (4 arrivals)
    uint64_t *pv_done = p_full + 4;            // [half][P tile]: O_h += P_h(j) V_j done
    uint64_t *o_final = pv_done + 4;           // every product complete
    uint64_t *mma_drain = o_final + 1;
    uint64_t *mma_drain_s = mma_drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Lay::kBars);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);
    const Abort ab{abort_word, &g_status_halves};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item (batch*head, query tile) ----------------------------------
    // CTAs go in groups of p.head_group heads (the last group may be
    // smaller), and within a group heaviest causal tiles first, heads
    // alternating: the CTAs on the GPU at one time then read the K and V of
    // a few heads, which stay in L2, instead of one head each.
    const int64_t BH = p.B * p.H;
    const int64_t G = p.head_group;
    const int64_t per_group = G * q_tiles;
    const int64_t g0 = ((int64_t)blockIdx.x / per_group) * G;
    const int64_t r = (int64_t)blockIdx.x % per_group;
    const int64_t gsize = BH - g0 < G ? BH - g0 : G;
    const int64_t qt = (int64_t)q_tiles - 1 - r / gsize;
    const int64_t bh = g0 + r % gsize;
    const int64_t b = bh / p.H;
    const int64_t N = p.N;
    const int64_t q0 = qt * BM;
    int64_t L = N;
    if (p.kv_len) {
        L = p.kv_len[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    const int64_t kv_end = p.causal ? (L < q0 + BM ? L : q0 + BM) : L;
    const int n_kv = (int)((kv_end + BN - 1) / BN);

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lay::kBars; ++i) {
            uint32_t count = 1;
            if (&bars[i] == s_read) count = 8;                     // one arrival per softmax warp
            if (&bars[i] >= p_full && &bars[i] < p_full + 4) count = 4;   // the four warps of a half
            ptx::mbar_init(&bars[i], count);
        }
        *abort_word = 0;
        ptx::fence_mbarrier_init();
        // Thread 0 is also the producer: Q and K_0 are requested now, so that
        // their latency overlaps the TMEM allocation and the barrier below.
        if (n_kv > 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::mbar_arrive_expect_tx(q_full, kTileBytes);
            for (int c = 0; c < kChunks; ++c)
                ptx::tma_load_3d(smem + kQOff + c * kChunkBytes, &tm_q, q_full, c * 64, (int32_t)q0, (int32_t)bh);
            ptx::mbar_arrive_expect_tx(&k_full[0], kTileBytes);
            for (int c = 0; c < kChunks; ++c)
                ptx::tma_load_3d(smem + kKOff + c * kChunkBytes, &tm_k, &k_full[0], c * 64, 0, (int32_t)bh);
        }
    }
    // A tile with no visible key only writes O = 0 and LSE = -inf: it needs
    // no tensor memory.
    if (warp == 1 && n_kv > 0) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = n_kv > 0 ? *tmem_slot : 0u;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0 && n_kv > 0) {
            auto load_tile = [&](const CUtensorMap *tm, int off, uint64_t *bar, int64_t row0) {
                ptx::mbar_arrive_expect_tx(bar, kTileBytes);
                for (int c = 0; c < kChunks; ++c)
                    ptx::tma_load_3d(smem + off + c * kChunkBytes, tm, bar, c * 64, (int32_t)row0, (int32_t)bh);
            };
            // Loads in the order the MMAs read them: K_0, K_1, then V_t and
            // K_{t+2} in turn (Q and K_0 were requested before the CTA-wide
            // barrier).  K_t goes into slot t % R once S_{t-R} has read that
            // slot, V_t once both halves' products of block t-R have.
            int k_issued = 1, v_issued = 0;
            auto load_k = [&]() -> bool {
                const int t = k_issued;
                if (t >= R &&
                    !wait_bounded(&k_empty[t % R], ((t - R) / R) & 1, p.wait_limit_ns, kSiteSlotEmpty, ab))
                    return false;
                load_tile(&tm_k, kKOff + (t % R) * kTileBytes, &k_full[t % R], (int64_t)t * BN);
                ++k_issued;
                return true;
            };
            auto load_v = [&]() -> bool {
                const int t = v_issued;
                if (t >= R &&
                    !wait_bounded(&v_empty[t % R], ((t - R) / R) & 1, p.wait_limit_ns, kSiteSlotEmpty, ab))
                    return false;
                load_tile(&tm_v, kVOff + (t % R) * kTileBytes, &v_full[t % R], (int64_t)t * BN);
                ++v_issued;
                return true;
            };
            bool ok = true;
            if (n_kv > 1) ok = load_k();
            while (ok && v_issued < n_kv) {
                ok = load_v();
                if (ok && k_issued < n_kv) ok = load_k();
            }
            // Drain: no copy may still be landing in shared memory at exit.
            wait_bounded(q_full, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            for (int t = k_issued > R ? k_issued - R : 0; t < k_issued; ++t)
                wait_bounded(&k_full[t % R], (t / R) & 1, p.wait_limit_ns, kSiteDrain, ab, false);
            for (int t = v_issued > R ? v_issued - R : 0; t < v_issued; ++t)
                wait_bounded(&v_full[t % R], (t / R) & 1, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    } else if (warp == 1 || warp == 3) {
        // ================= MMA issuers: warp 3 S, warp 1 PV =================
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_qk = make_idesc(BM, BN, 0, 0, kF16);
            constexpr uint32_t idesc_pv = make_idesc(BM, D, 0, 1, kF16);
            // The start-address field of a descriptor is the byte address / 16,
            // and every operand lies below 256 KiB: the descriptors are built
            // once, and each slot and K-step adds its byte offset / 16.
            const uint64_t q_desc = make_sdesc(ptx::smem_u32(smem + kQOff), 16, 1024);
            const uint64_t k_desc = make_sdesc(ptx::smem_u32(smem + kKOff), 16, 1024);
            const uint64_t v_desc = make_sdesc(ptx::smem_u32(smem + kVOff), kChunkBytes, 1024);
            constexpr uint64_t kTileStep = kTileBytes >> 4;
            if (warp == 3) {
                // S_t = Q K_t^T into the score tile, once the softmax warps
                // hold S_{t-1} in registers.  K_t has normally landed long
                // before, so it is waited for first and the products follow
                // the s_read hand-off directly.
                bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab);
                for (int t = 0; t < n_kv && ok; ++t) {
                    ok = wait_bounded(&k_full[t % R], (t / R) & 1, p.wait_limit_ns, kSiteSlotFull, ab);
                    if (ok && t > 0) ok = wait_bounded(s_read, (t - 1) & 1, p.wait_limit_ns, kSiteSFull, ab);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint64_t kd = k_desc + (uint64_t)(t % R) * kTileStep;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t off = (uint64_t)(((k / 4) * kChunkBytes + (k % 4) * 32) >> 4);
                        ptx::mma_ss(tmem + kColS, q_desc + off, kd + off, idesc_qk, k > 0);
                    }
                    ptx::mma_commit(s_full);
                    ptx::mma_commit(&k_empty[t % R]);
                }
                ptx::mma_commit(mma_drain_s);
                wait_bounded(mma_drain_s, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            } else {
                // O_h += P_h(j) V_j[64h ..]: K-steps 4h .. 4h+3 of the block,
                // A from the half's 32 columns of P tile j % 2.
                for (int j = 0; j < n_kv; ++j) {
                    const int buf = j & 1;
                    bool ok = wait_bounded(&v_full[j % R], (j / R) & 1, p.wait_limit_ns, kSiteSlotFull, ab);
                    const uint64_t vd = v_desc + (uint64_t)(j % R) * kTileStep;
                    for (int h = 0; h < 2 && ok; ++h) {
                        ok = wait_bounded(&p_full[h * 2 + buf], (j >> 1) & 1, p.wait_limit_ns, kSitePFull, ab);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        const uint32_t to = tmem + Lay::col_o(h), tp = tmem + Lay::col_p(buf, h);
#pragma unroll
                        for (int k = 0; k < kHalf / 16; ++k)
                            ptx::mma_ts(to, tp + k * 8, vd + (uint64_t)(((4 * h + k) * 2048) >> 4), idesc_pv,
                                        (j > 0 || k > 0) ? 1u : 0u);
                        ptx::mma_commit(&pv_done[h * 2 + buf]);
                    }
                    if (!ok) break;
                    ptx::mma_commit(&v_empty[j % R]);
                    if (j + 1 == n_kv) ptx::mma_commit(o_final);
                }
                ptx::mma_commit(mma_drain);
                wait_bounded(mma_drain, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            }
        }
    } else if (warp >= kSoftmaxWarp0) {
        // ================= online softmax of one key half + epilogue =================
        const int h = (warp - kSoftmaxWarp0) / 4;     // key half: columns 64h .. 64h+63 of every block
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter ..
        const int r_local = quarter * 32 + lane;
        const int64_t row = q0 + r_local;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColS + (uint32_t)(h * kHalf);
        const int64_t lim = p.causal ? (L < row + 1 ? L : row + 1) : L;   // visible keys: k < lim
        const float sl2 = p.scale_log2;

        OnlineRow<D, kF16, kHalf> st;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            const uint32_t tP = tmem + lane_off + Lay::col_p(buf, h);
            const uint32_t tO = tmem + lane_off + Lay::col_o(h);
            const bool got = wait_bounded(s_full, j & 1, p.wait_limit_ns, kSiteSFull, ab);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            // Whether O_h += P_h(j-2) V_{j-2}, the last reader of P tile
            // `buf`, is already done: tested now, so that the test's latency
            // overlaps the score load, and waited for only if it was not.
            const bool p_free = j < 2 || ptx::mbar_test(&pv_done[h * 2 + buf], ((j - 2) >> 1) & 1);
            ptx::tc_fence_after();
            uint32_t s_raw[2][32];
            ptx::tmem_ld32(tS, s_raw[0]);
            ptx::tmem_ld32(tS + 32, s_raw[1]);
            ptx::tmem_wait_ld();
            // S_j is in registers: the score tile is free for S_{j+1}
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(s_read);

            const int64_t vis = lim - (int64_t)j * BN - h * kHalf;   // columns k < vis are visible
            if (vis < kHalf) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (c * 32 + t >= vis) s_raw[c][t] = f2u(-INFINITY);
            }
            // O_h += P_h(j-1) V_{j-1} may still be running: an O_h rescale
            // waits for it.  P tile `buf` was last read by O_h += P_h(j-2)
            // V_{j-2}: the first P store waits for that product.
            bool hook_ok = true;
            auto before_o = [&] {
                if (j > 0) {
                    hook_ok = wait_bounded(&pv_done[h * 2 + ((j - 1) & 1)], ((j - 1) >> 1) & 1, p.wait_limit_ns,
                                           kSiteOFinal, ab) && hook_ok;
                    ptx::tc_fence_after();
                }
            };
            auto before_p = [&] {
                if (!__all_sync(0xffffffffu, p_free)) {
                    hook_ok = wait_bounded(&pv_done[h * 2 + buf], ((j - 2) >> 1) & 1, p.wait_limit_ns, kSiteOFinal,
                                           ab) && hook_ok;
                    ptx::tc_fence_after();
                }
            };
            st.template block<1>(s_raw, sl2, j > 0, tP, tO, before_o, before_p);
            // every lane's P stores have landed; after the warp has
            // synchronised, one lane tells the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[h * 2 + buf]);
            if (!__all_sync(0xffffffffu, hook_ok)) {
                ok = false;
                break;
            }
        }

        // ---- epilogue: merge the two halves' states ---------------------------
        // m = max(m_A, m_B), w_h = 2^(m_h - m) (0 for a half with no visible
        // key), O = (w_A O_A + w_B O_B) / (w_A l_oA + w_B l_oB),
        // LSE = (m + log2(w_A l_A + w_B l_B)) ln 2.
        bool have = (n_kv > 0) && ok;
        if (have) have = wait_bounded(o_final, 0, p.wait_limit_ns, kSiteOFinal, ab);
        // all eight softmax warps agree, so that the named barriers below are
        // reached by all of them or by none
        have = ptx::bar_and(1, 256, have);
        if (have || n_kv == 0) {
            ptx::tc_fence_after();
            // (m, l, l_o) of both halves, through the first V slot: every
            // product that read it is complete (o_final), and no copy is in
            // flight after the last block's V.
            float *xch = reinterpret_cast<float *>(smem + kVOff);   // [half][3][BM]
            xch[(h * 3 + 0) * BM + r_local] = st.m_ref;
            xch[(h * 3 + 1) * BM + r_local] = st.l;
            xch[(h * 3 + 2) * BM + r_local] = st.l_o;
            ptx::bar_sync(2, 256);
            float mh[2], lh[2], loh[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mh[e] = xch[(e * 3 + 0) * BM + r_local];
                lh[e] = xch[(e * 3 + 1) * BM + r_local];
                loh[e] = xch[(e * 3 + 2) * BM + r_local];
            }
            const float m = fmaxf(lh[0] > 0.f ? mh[0] : -INFINITY, lh[1] > 0.f ? mh[1] : -INFINITY);
            float w[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) w[e] = lh[e] > 0.f ? ptx::ex2_approx(mh[e] - m) : 0.f;
            const float l_all = w[0] * lh[0] + w[1] * lh[1];
            const float lo_all = w[0] * loh[0] + w[1] * loh[1];
            const bool empty = !(l_all > 0.f);
            const float inv = empty ? 0.f : 1.f / lo_all;
            const float c0 = w[0] * inv, c1 = w[1] * inv;
            const float lse_row = empty ? -INFINITY : (m + log2f(l_all)) * 0.69314718055994530942f;

            // This thread writes columns [h*D/2, (h+1)*D/2) of its row: O as
            // 16-bit, staged in the Q buffer (free: every product is complete)
            // as 128-byte-swizzled 128 x 64 boxes, then written by TMA stores
            // that clip rows >= N and columns >= p.D.
            uint8_t *obuf = smem + kQOff;
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                const int col = h * (D / 2) + c * 32;
                uint32_t oa[32], ob[32];
                if (n_kv > 0) {
                    ptx::tmem_ld32(tmem + lane_off + Lay::col_o(0) + (uint32_t)col, oa);
                    ptx::tmem_ld32(tmem + lane_off + Lay::col_o(1) + (uint32_t)col, ob);
                    ptx::tmem_wait_ld();
                }
                uint32_t wd[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float lo = 0.f, hi = 0.f;
                    if (n_kv > 0) {
                        lo = fmaf(c0, u2f(oa[2 * t]), c1 * u2f(ob[2 * t]));
                        hi = fmaf(c0, u2f(oa[2 * t + 1]), c1 * u2f(ob[2 * t + 1]));
                    }
                    wd[t] = empty ? 0u : ptx::pack16x2<kF16>(lo, hi);
                }
                // 32 columns = 4 of the 8 16-byte units of a 64-column box row
                const uint32_t row_addr = ptx::smem_u32(obuf + (col / 64) * kChunkBytes + r_local * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)((col % 64) / 8 + u) ^ (uint32_t)(r_local & 7);
                    ptx::st_shared_v4(row_addr + (unit << 4), wd[4 * u], wd[4 * u + 1], wd[4 * u + 2], wd[4 * u + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::bar_sync(2, 256);                         // every softmax warp's part is staged
            if (h == 0 && r_local == 0) {
                for (int c = 0; c < kChunks; ++c)
                    ptx::tma_store_3d(&tm_o, obuf + c * kChunkBytes, c * 64, (int32_t)q0, (int32_t)bh);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read<0>();           // the boxes have left shared memory
            }
            if (h == 0 && row < N && p.lse) p.lse[bh * N + row] = lse_row;
        }
    }
    // ---- teardown ----------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1 && n_kv > 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kF16>
cudaError_t launch(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   const CUtensorMap &to, cudaStream_t stream)
{
    using Lay = HalvesLayout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fwd_halves_kernel<D, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int q_tiles = (int)((p.N + BM - 1) / BM);
    const int64_t ctas = p.B * p.H * (int64_t)q_tiles;
    // Heads per group: as many as keep the group's K and V (2 N D 16-bit
    // values per head) within 48 MiB of the 126 MiB L2.
    FwdParams pg = p;
    const int64_t kv_bytes = 4 * p.N * (int64_t)D;
    const int64_t budget = (int64_t)48 << 20;
    int64_t G = kv_bytes > 0 ? budget / kv_bytes : 1;
    const int64_t BH = p.B * p.H;
    pg.head_group = (int)(G < 1 ? 1 : (G > BH ? BH : G));
    fwd_halves_kernel<D, kF16><<<(unsigned)ctas, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, to, pg, q_tiles);
    return cudaGetLastError();
}

}  // namespace

// A multiple of 8 up to 128 runs at the next of 64 / 128 with zero-filled
// columns (as in the other tensor-core kernels).
cudaError_t launch_fwd_halves(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream)
{
    if (p.D % 8 != 0 || p.D <= 0 || p.D > 128) return cudaErrorInvalidValue;
    if (p.D <= 64)
        return p.f16 ? launch<64, true>(p, tm_q, tm_k, tm_v, tm_o, stream)
                     : launch<64, false>(p, tm_q, tm_k, tm_v, tm_o, stream);
    return p.f16 ? launch<128, true>(p, tm_q, tm_k, tm_v, tm_o, stream)
                 : launch<128, false>(p, tm_q, tm_k, tm_v, tm_o, stream);
}

cudaError_t read_and_clear_status_halves(uint32_t *out)
{
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_halves, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_halves, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace fa
