// fa_fwd_onetile.cu -- bf16 / fp16 attention forward on the tensor cores with
// one 128-row query tile per CTA.
//
// The computation is the tiled online-softmax forward of "vectorized-flash-
// attention-kernel" (Core algorithm; Key design decisions 1-3), with the same
// per-row softmax step as the two-tile kernel (fa_fwd_softmax.cuh).  Only the
// layout on the SM differs.  It serves head dimension 256, whose output tile
// takes 256 of the 512 TMEM columns, and grids where the two-tile kernel's
// 256-row items would not fill the GPU (twice as many CTAs):
//
//   * one CTA owns one 128-row query tile; TMEM holds two score tiles S_a,
//     S_b (128 columns each) and O (D columns);
//   * warp 1 issues S_{j+1} = Q K_{j+1}^T into the other score tile before
//     O += P_j V_j, so the tensor core computes the next block's scores while
//     warps 4-7 run the softmax of this one;
//   * shared memory holds Q and one K and one V tile (D x 256 bytes each);
//     warp 0 loads K_{j+1} as soon as S_j has consumed K_j, ahead of V_j,
//     which waits for O += P_{j-1} V_{j-1}.
//
// O is rescaled in TMEM only when the lazy reference max moves; because
// O += P_{j-1} V_{j-1} may still be running when the softmax of block j
// starts, such a rescale first waits for that product (pv_done).
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
constexpr int kThreads = 256;                   // warp 0 TMA, warp 1 MMA, warps 4-7 softmax
constexpr int kSoftmaxWarp0 = 4;
constexpr int kChunkBytes = 128 * 128;          // one 128-row x 64-column 16-bit box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;                 // S_a [0,128), S_b [128,256), O [256,256+D)

template <int D>
struct OneTileLayout {
    static constexpr int kChunks = D / 64;                  // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = kChunks * kChunkBytes;    // Q, a K or a V tile
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kTileBytes;
    static constexpr int kVOff = 2 * kTileBytes;
    static constexpr int kBarOff = 3 * kTileBytes;
    // At least 120 KB, so that one CTA (and its 512 TMEM columns) sits on an SM.
    static constexpr int kNeed = kBarOff + 256 + 1024;      // + alignment slack
    static constexpr int kSmemBytes = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t col_s(int buf) { return (uint32_t)buf * 128u; }

template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_onetile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdParams p, const int q_tiles)
{
    using Lay = OneTileLayout<D>;
    constexpr int kChunks = Lay::kChunks, kTileBytes = Lay::kTileBytes;
    constexpr int kQOff = Lay::kQOff, kKOff = Lay::kKOff, kVOff = Lay::kVOff;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;
    uint64_t *k_empty = bars + 2;
    uint64_t *v_full = bars + 3;
    uint64_t *v_empty = bars + 4;
    uint64_t *s_full = bars + 5;     // [2], per score tile
    uint64_t *p_full = bars + 7;     // [2], per score tile
    uint64_t *pv_done = bars + 9;    // one phase per O += P V
    uint64_t *o_final = bars + 10;
    uint64_t *mma_drain = bars + 11;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
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
        for (int i = 0; i < 12; ++i)   // p_full: one arrival per softmax warp; the rest: one
            ptx::mbar_init(&bars[i], (&bars[i] == &p_full[0] || &bars[i] == &p_full[1]) ? 4 : 1);
        *abort_word = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0 && n_kv > 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            auto load_tile = [&](const CUtensorMap *tm, int off, uint64_t *bar, int64_t row0) {
                ptx::mbar_arrive_expect_tx(bar, kTileBytes);
                for (int c = 0; c < kChunks; ++c)
                    ptx::tma_load_3d(smem + off + c * kChunkBytes, tm, bar, c * 64, (int32_t)row0, (int32_t)bh);
            };
            load_tile(&tm_q, kQOff, q_full, q0);
            load_tile(&tm_k, kKOff, k_full, 0);
            load_tile(&tm_v, kVOff, v_full, 0);
            // K_t (t >= 1) waits until S_{t-1} has read K_{t-1}; V_t waits
            // until O += P_{t-1} V_{t-1} is done.  The MMA order (S_{j+1}
            // before P_j V_j) frees K first, so K_{j+1} goes before V_j.
            int k_issued = 1, v_issued = 1;
            bool ok = true;
            if (n_kv > 1) {
                ok = wait_bounded(k_empty, 0, p.wait_limit_ns, kSiteSlotEmpty, ab);
                if (ok) load_tile(&tm_k, kKOff, k_full, (int64_t)BN);
                k_issued += ok ? 1 : 0;
            }
            for (int j = 1; j < n_kv && ok; ++j) {
                if (j + 1 < n_kv) {
                    if (!wait_bounded(k_empty, j & 1, p.wait_limit_ns, kSiteSlotEmpty, ab)) break;
                    load_tile(&tm_k, kKOff, k_full, (int64_t)(j + 1) * BN);
                    ++k_issued;
                }
                if (!wait_bounded(v_empty, (j - 1) & 1, p.wait_limit_ns, kSiteSlotEmpty, ab)) break;
                load_tile(&tm_v, kVOff, v_full, (int64_t)j * BN);
                ++v_issued;
            }
            // Drain: no copy may still be landing in shared memory at exit.
            wait_bounded(q_full, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            wait_bounded(k_full, (k_issued - 1) & 1, p.wait_limit_ns, kSiteDrain, ab, false);
            wait_bounded(v_full, (v_issued - 1) & 1, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_qk = make_idesc(BM, BN, 0, 0, kF16);
            constexpr uint32_t idesc_pv = make_idesc(BM, D, 0, 1, kF16);
            const uint32_t qa = ptx::smem_u32(smem + kQOff);
            const uint32_t ka = ptx::smem_u32(smem + kKOff);
            const uint32_t va = ptx::smem_u32(smem + kVOff);
            // The start-address field of a descriptor is the byte address / 16,
            // and every operand lies below 256 KiB: the descriptors are built
            // once, and each K-step adds its byte offset / 16.
            const uint64_t q_desc = make_sdesc(qa, 16, 1024);
            const uint64_t k_desc = make_sdesc(ka, 16, 1024);
            const uint64_t v_desc = make_sdesc(va, kChunkBytes, 1024);
            auto issue_s = [&](int buf) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * kChunkBytes + (k % 4) * 32) >> 4);
                    ptx::mma_ss(tmem + col_s(buf), q_desc + off, k_desc + off, idesc_qk, k > 0);
                }
            };
            auto issue_pv = [&](int buf, bool acc) {
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ts(tmem + kColO, tmem + col_s(buf) + k * 8, v_desc + (uint64_t)((k * 2048) >> 4),
                                idesc_pv, acc || k > 0);
            };
            bool ok = wait_bounded(q_full, 0, p.wait_limit_ns, kSiteQFull, ab) &&
                      wait_bounded(k_full, 0, p.wait_limit_ns, kSiteSlotFull, ab);
            if (ok) {
                ptx::tc_fence_after();
                issue_s(0);
                ptx::mma_commit(&s_full[0]);
                ptx::mma_commit(k_empty);
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                if (j + 1 < n_kv) {
                    if (!wait_bounded(k_full, (j + 1) & 1, p.wait_limit_ns, kSiteSlotFull, ab)) break;
                    ptx::tc_fence_after();
                    issue_s((j + 1) & 1);
                    ptx::mma_commit(&s_full[(j + 1) & 1]);
                    ptx::mma_commit(k_empty);
                }
                if (!wait_bounded(v_full, j & 1, p.wait_limit_ns, kSiteSlotFull, ab) ||
                    !wait_bounded(&p_full[j & 1], (j >> 1) & 1, p.wait_limit_ns, kSitePFull, ab))
                    break;
                ptx::tc_fence_after();
                issue_pv(j & 1, j > 0);
                ptx::mma_commit(v_empty);
                ptx::mma_commit(pv_done);
                if (j + 1 == n_kv) ptx::mma_commit(o_final);
            }
            // Drain: every MMA issued here completes before TMEM is freed.
            ptx::mma_commit(mma_drain);
            wait_bounded(mma_drain, 0, p.wait_limit_ns, kSiteDrain, ab, false);
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
            const int64_t vis = lim - (int64_t)j * BN;   // columns k < vis are visible
            if (vis < BN) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (c * 32 + t >= vis) s_raw[c][t] = f2u(-INFINITY);
            }
            // O += P_{j-1} V_{j-1} may still be running: an O rescale waits
            // for it first.
            bool hook_ok = true;
            st.block(s_raw, sl2, j > 0, tS, tO, [&] {
                hook_ok = wait_bounded(pv_done, (j - 1) & 1, p.wait_limit_ns, kSiteOFinal, ab);
                ptx::tc_fence_after();
            });
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

        // ---- epilogue: O = acc / l, LSE = (m + log2 l) ln 2 ----------------
        bool have = (n_kv > 0) && ok;
        if (have) have = wait_bounded(o_final, 0, p.wait_limit_ns, kSiteOFinal, ab);
        // the four softmax warps agree, so that the named barrier below is
        // reached by all of them or by none
        have = ptx::bar_and(1, 128, have);
        if (have || n_kv == 0) {
            ptx::tc_fence_after();
            const bool empty = !(st.l > 0.f);
            const float inv = empty ? 0.f : 1.f / st.l;
            const float lse_row = empty ? -INFINITY : (st.m_ref + log2f(st.l)) * 0.69314718055994530942f;
            // Only the first p.D (a multiple of 8, <= D) columns exist in
            // memory; the rest of the D computed ones are the zero padding.
            const int Dv = (int)p.D;
            const int64_t flat = bh * N + row;
            (void)Dv;
            // O = acc / l as 16-bit, staged in the Q buffer (free: every MMA
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
    if (warp == 1) {
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
