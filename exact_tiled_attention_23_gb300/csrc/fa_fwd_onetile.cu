// fa_fwd_onetile.cu -- bf16 / fp16 attention forward on the tensor cores with
// one 128-row query tile per CTA.
//
// The computation is the tiled online-softmax forward of "vectorized-flash-
// attention-kernel" (Core algorithm; Key design decisions 1-3), with the same
// per-row softmax step as the two-tile kernel (fa_fwd_softmax.cuh).  Only the
// layout on the SM differs:
//
//   * one CTA owns one 128-row query tile; TMEM holds two score tiles S_a,
//     S_b (128 columns each), O (D columns) and, for D <= 128, two P tiles of
//     their own (64 columns each: 16-bit pairs);
//   * with P apart (D <= 128) warp 3 issues S_0, S_1 and then S_{j+2} =
//     Q K_{j+2}^T into the score tile of S_j as soon as the softmax warps
//     hold S_j in registers, and warp 1 issues O += P_j V_j once they hand
//     P_j over.  The tensor core so holds the next block's scores ready while
//     warps 4-7 run the softmax of this one, and two issuing threads keep it
//     busier than one (one thread issues at most one N=128 product per
//     ~90-100 clk on this GPU, two reach the 64 clk rate);
//   * warp 0 streams K and V through rings of kRing slots each, in the order
//     the MMAs read them (K_0, K_1, V_0, K_2, V_1, ...), so a load has several
//     blocks' time to land;
//   * at D = 256 the output tile takes 256 TMEM columns, so P is written over
//     the first 64 columns of its score tile and K, V have one slot each.
//
// O is rescaled in TMEM only when the lazy reference max moves; because
// O += P_{j-1} V_{j-1} may still be running when the softmax of block j
// starts, such a rescale first waits for that product.  P tile j % 2 is free
// for block j once O += P_{j-2} V_{j-2}, its last reader, is done: with P
// apart the softmax waits for that product's commit before its first P
// store; with P over S (D = 256) the commit that completed S_j covers it,
// because one thread issued S_j after it.
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

__device__ uint32_t g_status_onetile;

namespace {

constexpr int BM = 128;                         // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;                         // keys per block
constexpr int kThreads = 256;                   // warp 0 TMA, warps 1 and 3 MMA, warps 4-7 softmax
constexpr int kSoftmaxWarp0 = 4;
constexpr int kChunkBytes = 128 * 128;          // one 128-row x 64-column 16-bit box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;                 // S_a [0,128), S_b [128,256), O [256,256+D)

template <int D>
struct OneTileLayout {
    static constexpr int kChunks = D / 64;                  // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = kChunks * kChunkBytes;    // Q, a K or a V tile
    // K and V slots each: as many as shared memory holds next to Q
    static constexpr int kRing = D == 256 ? 1 : (D == 128 ? 3 : 4);
    // P in TMEM columns of its own (two tiles of 64) where O leaves room
    static constexpr bool kPApart = D <= 128;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kTileBytes;                        // K slots
    static constexpr int kVOff = kKOff + kRing * kTileBytes;        // V slots
    static constexpr int kBarOff = kVOff + kRing * kTileBytes;
    static constexpr int kBars = 1 + 4 * kRing + 12;
    // At least 120 KB, so that one CTA (and its 512 TMEM columns) sits on an SM.
    static constexpr int kNeed = kBarOff + 256 + 1024;      // + alignment slack
    static constexpr int kSmemBytes = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
    // TMEM column of P tile `buf`
    __device__ static constexpr uint32_t col_p(int buf)
    {
        return kPApart ? kColO + (uint32_t)D + (uint32_t)buf * 64u : (uint32_t)buf * 128u;
    }
    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kBars * 8 + 8 <= 256, "barrier area");
    static_assert(!kPApart || kColO + D + 128 <= kTmemCols, "TMEM columns");
};

__device__ __forceinline__ uint32_t col_s(int buf) { return (uint32_t)buf * 128u; }

template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_onetile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdParams p, const int q_tiles)
{
    using Lay = OneTileLayout<D>;
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
    uint64_t *s_full = v_empty + R;            // [2], per score tile
    uint64_t *p_full = s_full + 2;             // [2], per P tile
    uint64_t *pv_done = p_full + 2;            // [2], per P tile: O += P V has read it
    uint64_t *o_final = pv_done + 2;
    uint64_t *mma_drain = o_final + 1;
    // P apart only: score tile read into the softmax warps' registers (it may
    // be overwritten), and the drain of the second MMA thread.
    uint64_t *s_read = mma_drain + 1;          // [2], per score tile
    uint64_t *mma_drain_s = s_read + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Lay::kBars);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);
    const Abort ab{abort_word, &g_status_onetile};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item (batch*head, query tile), heaviest causal tiles first ----
    const int64_t BH = p.B * p.H;
    const int64_t qt = (int64_t)q_tiles - 1 - (int64_t)blockIdx.x / BH;
    const int64_t bh = (int64_t)blockIdx.x % BH;
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
        // P hand-offs take one arrival per softmax warp, the rest one
        for (int i = 0; i < Lay::kBars; ++i)
            ptx::mbar_init(&bars[i], (&bars[i] == &p_full[0] || &bars[i] == &p_full[1] || &bars[i] == &s_read[0] ||
                                      &bars[i] == &s_read[1]) ? 4 : 1);
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
    // An item with no visible key only writes O = 0 and LSE = -inf: it needs
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
            // slot, V_t once O += P_{t-R} V_{t-R} has.
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
    } else if (warp == 1 || (Lay::kPApart && warp == 3)) {
        // ================= MMA issuers =================
        // With P apart (D <= 128) warp 1 issues the PV products and warp 3
        // the S products: the two streams touch disjoint TMEM columns, and
        // two issuing threads keep the tensor core busier than one (a probe
        // on this GPU ran one thread's N=128 products at ~110 clk each, two
        // threads' at ~70 clk per product together).  At D = 256 (P over S)
        // warp 1 issues both, S_{j+1} behind the PV that reads its columns.
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_qk = make_idesc(BM, BN, 0, 0, kF16);
            constexpr uint32_t idesc_pv = make_idesc(BM, D, 0, 1, kF16);
            const uint32_t qa = ptx::smem_u32(smem + kQOff);
            const uint32_t ka = ptx::smem_u32(smem + kKOff);
            const uint32_t va = ptx::smem_u32(smem + kVOff);
            // The start-address field of a descriptor is the byte address / 16,
            // and every operand lies below 256 KiB: the descriptors are built
            // once, and each slot and K-step adds its byte offset / 16.
            const uint64_t q_desc = make_sdesc(qa, 16, 1024);
            const uint64_t k_desc = make_sdesc(ka, 16, 1024);
            const uint64_t v_desc = make_sdesc(va, kChunkBytes, 1024);
            constexpr uint64_t kTileStep = kTileBytes >> 4;
            auto issue_s = [&](int buf, int slot) {
                const uint64_t kd = k_desc + (uint64_t)slot * kTileStep;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * kChunkBytes + (k % 4) * 32) >> 4);
                    ptx::mma_ss(tmem + col_s(buf), q_desc + off, kd + off, idesc_qk, k > 0);
                }
            };
            auto issue_pv = [&](int buf, int slot, bool acc) {
                const uint64_t vd = v_desc + (uint64_t)slot * kTileStep;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ts(tmem + kColO, tmem + Lay::col_p(buf) + k * 8, vd + (uint64_t)((k * 2048) >> 4),
                                idesc_pv, acc || k > 0);
            };
            // S_t into score tile t % 2 (K_t in slot t % R)
            auto next_s = [&](int t) -> bool {
                if (!wait_bounded(&k_full[t % R], (t / R) & 1, p.wait_limit_ns, kSiteSlotFull, ab)) return false;
                ptx::tc_fence_after();
                issue_s(t & 1, t % R);
                ptx::mma_commit(&s_full[t & 1]);
                ptx::mma_commit(&k_empty[t % R]);
                return true;
            };
            if constexpr (!Lay::kPApart) {
                bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab) && next_s(0);
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int buf = j & 1;
                    // P over S: S_{j+1} goes into the score tile P_{j-1} has
                    // left, after O += P_{j-1} V_{j-1} (issued before it, so
                    // read before).
                    if (j + 1 < n_kv && !next_s(j + 1)) break;
                    if (!wait_bounded(&v_full[j % R], (j / R) & 1, p.wait_limit_ns, kSiteSlotFull, ab) ||
                        !wait_bounded(&p_full[buf], (j >> 1) & 1, p.wait_limit_ns, kSitePFull, ab))
                        break;
                    ptx::tc_fence_after();
                    issue_pv(buf, j % R, j > 0);
                    ptx::mma_commit(&v_empty[j % R]);
                    ptx::mma_commit(&pv_done[buf]);
                    if (j + 1 == n_kv) ptx::mma_commit(o_final);
                }
            } else if (warp == 1) {
                // PV products: O += P_j V_j once the softmax has handed P_j over.
                for (int j = 0; j < n_kv; ++j) {
                    const int buf = j & 1;
                    if (!wait_bounded(&v_full[j % R], (j / R) & 1, p.wait_limit_ns, kSiteSlotFull, ab) ||
                        !wait_bounded(&p_full[buf], (j >> 1) & 1, p.wait_limit_ns, kSitePFull, ab))
                        break;
                    ptx::tc_fence_after();
                    issue_pv(buf, j % R, j > 0);
                    ptx::mma_commit(&v_empty[j % R]);
                    ptx::mma_commit(&pv_done[buf]);
                    if (j + 1 == n_kv) ptx::mma_commit(o_final);
                }
            } else {
                // S products: S_0 and S_1 into the two score tiles, then S_t
                // into tile t % 2 as soon as the softmax warps hold S_{t-2}
                // in registers.
                bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab) && next_s(0);
                if (ok && n_kv > 1) ok = next_s(1);
                for (int t = 2; t < n_kv && ok; ++t)
                    ok = wait_bounded(&s_read[t & 1], ((t - 2) >> 1) & 1, p.wait_limit_ns, kSiteSFull, ab) &&
                         next_s(t);
            }
            // Drain: every MMA issued here completes before TMEM is freed.
            uint64_t *drain = (Lay::kPApart && warp == 3) ? mma_drain_s : mma_drain;
            ptx::mma_commit(drain);
            wait_bounded(drain, 0, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    } else if (warp >= kSoftmaxWarp0) {
        // ================= online softmax + epilogue =================
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter ..
        const int r_local = quarter * 32 + lane;
        const int64_t row = q0 + r_local;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kColO;
        const int64_t lim = p.causal ? (L < row + 1 ? L : row + 1) : L;   // visible keys: j < lim
        const float sl2 = p.scale_log2;

        OnlineRow<D, kF16> st;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            const uint32_t tS = tmem + lane_off + col_s(buf);
            const uint32_t tP = tmem + lane_off + Lay::col_p(buf);
            const bool got = wait_bounded(&s_full[buf], (j >> 1) & 1, p.wait_limit_ns, kSiteSFull, ab);
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
                // S_j is in registers: its tile is free for S_{j+2}
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&s_read[buf]);
            }
            const int64_t vis = lim - (int64_t)j * BN;   // columns k < vis are visible
            if (vis < BN) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (c * 32 + t >= vis) s_raw[c][t] = f2u(-INFINITY);
            }
            // O += P_{j-1} V_{j-1} may still be running: an O rescale waits
            // for it first.  P tile `buf` was last read by O += P_{j-2}
            // V_{j-2}.  With P over S (D = 256), S_j was issued after that
            // product by the same thread, so the commit that completed S_j
            // covers it; with P apart, the PV thread's own commit is waited
            // for before the first P store.
            bool hook_ok = true;
            auto before_o = [&] {
                hook_ok = wait_bounded(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.wait_limit_ns, kSiteOFinal,
                                       ab) && hook_ok;
                ptx::tc_fence_after();
            };
            auto before_p = [&] {
                if (Lay::kPApart && j >= 2) {
                    hook_ok = wait_bounded(&pv_done[buf], ((j - 2) >> 1) & 1, p.wait_limit_ns, kSiteOFinal, ab) &&
                              hook_ok;
                    ptx::tc_fence_after();
                }
            };
            st.block(s_raw, sl2, j > 0, tP, tO, before_o, before_p);
            // every lane's P stores have landed; after the warp has
            // synchronised, one lane tells the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[buf]);
            if (!__all_sync(0xffffffffu, hook_ok)) {
                ok = false;
                break;
            }
        }

        // ---- epilogue: O = acc / l_o, LSE = (m + log2 l) ln 2 --------------
        bool have = (n_kv > 0) && ok;
        if (have) have = wait_bounded(o_final, 0, p.wait_limit_ns, kSiteOFinal, ab);
        // the four softmax warps agree, so that the named barrier below is
        // reached by all of them or by none
        have = ptx::bar_and(1, 128, have);
        if (have || n_kv == 0) {
            ptx::tc_fence_after();
            const bool empty = !(st.l > 0.f);
            const float inv = empty ? 0.f : 1.f / st.l_o;   // O / (sum of the P the MMA used)
            const float lse_row = empty ? -INFINITY : (st.m_ref + log2f(st.l)) * 0.69314718055994530942f;
            // Only the first p.D (a multiple of 8, <= D) columns exist in
            // memory; the rest of the D computed ones are the zero padding.
            const int Dv = (int)p.D;
            const int64_t flat = bh * N + row;
            (void)Dv;
            // O = acc / l_o as 16-bit, staged in the Q buffer (free: every MMA
            // has completed) as 128-byte-swizzled 128 x 64 boxes, then written
            // by TMA stores that clip rows >= N and columns >= p.D.
            uint8_t *obuf = smem + kQOff;
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
                const uint32_t row_addr = ptx::smem_u32(obuf + (c / 2) * kChunkBytes + r_local * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)((c % 2) * 4 + u) ^ (uint32_t)(r_local & 7);
                    ptx::st_shared_v4(row_addr + (unit << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::bar_sync(1, 128);                         // the four softmax warps
            if (r_local == 0) {
                for (int c = 0; c < kChunks; ++c)
                    ptx::tma_store_3d(&tm_o, obuf + c * kChunkBytes, c * 64, (int32_t)q0, (int32_t)bh);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read<0>();           // the boxes have left shared memory
            }
            if (row < N && p.lse) p.lse[flat] = lse_row;
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
    using Lay = OneTileLayout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fwd_onetile_kernel<D, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int q_tiles = (int)((p.N + BM - 1) / BM);
    const int64_t ctas = p.B * p.H * (int64_t)q_tiles;
    fwd_onetile_kernel<D, kF16><<<(unsigned)ctas, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, to, p, q_tiles);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_f(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                     const CUtensorMap &to, cudaStream_t stream)
{
    return p.f16 ? launch<D, true>(p, tq, tk, tv, to, stream) : launch<D, false>(p, tq, tk, tv, to, stream);
}

}  // namespace

// D = 256, or a multiple of 8 up to 128 run at the next of 64 / 128 with
// zero-filled columns (as in the two-tile kernel).
cudaError_t launch_fwd_onetile(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream)
{
    if (p.D == 256) return launch_f<256>(p, tm_q, tm_k, tm_v, tm_o, stream);
    if (p.D % 8 != 0 || p.D <= 0 || p.D > 128) return cudaErrorInvalidValue;
    if (p.D <= 64) return launch_f<64>(p, tm_q, tm_k, tm_v, tm_o, stream);
    return launch_f<128>(p, tm_q, tm_k, tm_v, tm_o, stream);
}

cudaError_t read_and_clear_status_onetile(uint32_t *out)
{
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_onetile, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_onetile, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace fa
