// fa_bwd_bf16.cu -- bf16 attention backward on the Blackwell tensor cores.
//
// The backward by recomputation of "FlashAttention" (module F08, Math:
// "backward pass via recomputation and the rowsum(dP*P) = rowsum(dO*O)
// identity"; "vectorized-flash-attention-kernel", Key design decisions 4:
// the forward's saved row statistics rebuild P without a second softmax).
// With P = 2^(S*scale*log2e - LSE*log2e) rebuilt from the forward's LSE:
//
//   dV = P^T dO,   dP = dO V^T,   Delta = rowsum(dO * O),
//   dS = P * (dP - Delta),   dQ = scale * dS K,   dK = scale * dS^T Q.
//
// Kernels, all on the caller's stream:
//   1. bwd_prep_kernel: Delta per query row (fp32) and a zeroed fp32 dQ
//      accumulator, both in the caller's workspace;
//   2. bwd_kernel<D, kF16>: one CTA per (batch*head, 128-key tile).  K_j, V_j stay
//      in shared memory; the query tiles that see them stream through a
//      two-stage TMA ring with their dO.  Per query tile, in tensor memory
//      (one TMEM lane per key):
//        S^T = K_j Q_i^T and dP^T = V_j dO_i^T        (SS MMAs)
//        P^T, dS^T (bf16) written back over them by the key-row threads
//        dV += P^T dO_i and dK += dS^T Q_i             (TS MMAs, TMEM accumulators)
//        dQ_i = dS K_j                                 (SS MMA, dS staged in shared memory)
//      and dQ_i is added into the fp32 accumulator by TMA reduce-add of
//      staged 32-column boxes; at the end dK (times scale) and dV are
//      written as bf16;
//   3. bwd_dq_kernel: dQ = scale * accumulator, rounded to bf16.
// Keys at or past kv_len get zero dK, dV; query rows whose mask hides every
// key contribute nothing (P = 0 there).
#include "fa_internal.h"
#include "fa_tc_common.cuh"
#include "sm103_ptx.cuh"

#include <cuda_fp16.h>

#include <cmath>

namespace fa {

__device__ uint32_t g_status_bwd;

namespace {

constexpr int BK = 128;              // keys per CTA (= TMEM lanes of S^T, dP^T, dK, dV)
constexpr int BQ = 128;              // query rows per step
constexpr int kThreads = 384;        // warp 0 TMA, warp 1 MMA, warps 4-7 key rows, warps 8-11 query rows
constexpr int kWorkWarp0 = 4;
constexpr int kDQWarp0 = 8;

template <int D>
struct BwdLayout {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = 128 * 128;             // one 128-row x 64-column bf16 box
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // 128 rows x D
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kStages = 2;
    static constexpr int kStageOff = 2 * kTileBytes;          // stage s: Q_i then dO_i
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kDSOff = kStageOff + kStages * kStageBytes;
    static constexpr int kDSBytes = 2 * kChunkBytes;          // dS: 128 keys x 128 queries bf16
    static constexpr int kSmemBytes = kDSOff + kDSBytes + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    // TMEM: S^T [0,128) then P^T (bf16) over [0,64) and dQ_i over [0,D);
    // dP^T [128,256) then dS^T (bf16) over [128,192); dV and dK after them.
    static constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 256 + D;
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(kSmemBytes + 2048 <= 232448, "shared memory budget");
};

template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
           const __grid_constant__ CUtensorMap tm_dq, const BwdParams p)
{
    using Lay = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bars[17];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_word;
    __shared__ __align__(16) float nlse2_s[BQ];    // -LSE of the current query tile, log2 units (-inf: no row)
    __shared__ __align__(16) float ndelta_s[BQ];   // -Delta of the current query tile
    uint64_t *kv_full = &bars[0];
    uint64_t *stage_full = &bars[1];   // [2]
    uint64_t *stage_empty = &bars[3];  // [2]
    uint64_t *s_full = &bars[5];       // S^T, dP^T in TMEM
    uint64_t *ds_ready = &bars[6];     // dS in shared memory
    uint64_t *dq_full = &bars[7];      // dQ_i in TMEM
    uint64_t *dq_free = &bars[8];      // dQ_i read out of TMEM
    uint64_t *ds_free = &bars[9];      // the dQ staging no longer reads the dS buffer
    uint64_t *acc_full = &bars[10];
    uint64_t *mma_drain = &bars[11];
    uint64_t *p_ready = &bars[12];     // [BQ / 32]: P^T, dS^T (bf16) of 32 queries in TMEM
    const Abort ab{&abort_word, &g_status_bwd};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t BH = p.B * p.H;
    const int64_t N = p.N;
    // heaviest causal tiles first: key tile j sees query tiles j..nq-1
    const int64_t jt = (int64_t)blockIdx.x / BH;
    const int64_t bh = (int64_t)blockIdx.x % BH;
    const int64_t b = bh / p.H;
    const int64_t k0 = jt * BK;
    int64_t L = N;
    if (p.kv_len) {
        L = p.kv_len[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    const int64_t nq = (N + BQ - 1) / BQ;
    const int64_t i0 = p.causal ? jt : 0;
    const int n_iter = (k0 < L) ? (int)(nq - i0) : 0;

    if (threadIdx.x == 0) {
        ptx::mbar_init(kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&stage_full[s], 1);
            ptx::mbar_init(&stage_empty[s], 1);
        }
        ptx::mbar_init(s_full, 1);
        for (int c = 0; c < BQ / 32; ++c) ptx::mbar_init(&p_ready[c], 128);
        ptx::mbar_init(ds_ready, 128);
        ptx::mbar_init(dq_full, 1);
        ptx::mbar_init(dq_free, 128);
        ptx::mbar_init(ds_free, 1);
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(mma_drain, 1);
        abort_word = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_slot, Lay::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // Registers: the TMA / MMA warpgroup needs few; the two row warpgroups
    // hold a 64-column slice of S^T and dP^T, or a 128-column dQ row.
    // 128*112 + 2*128*192 fits in the 384*168 registers of the launch.
    if (warp < kWorkWarp0) {
    ptx::regs_dec<112>();
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0 && n_iter > 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            ptx::mbar_arrive_expect_tx(kv_full, 2 * Lay::kTileBytes);
            for (int c = 0; c < Lay::kChunks; ++c) {
                ptx::tma_load_3d(smem + Lay::kKOff + c * Lay::kChunkBytes, &tm_k, kv_full, c * 64,
                                 (int32_t)k0, (int32_t)bh);
                ptx::tma_load_3d(smem + Lay::kVOff + c * Lay::kChunkBytes, &tm_v, kv_full, c * 64,
                                 (int32_t)k0, (int32_t)bh);
            }
            uint32_t issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it & 1;
                if (it >= 2 &&
                    !wait_bounded(&stage_empty[s], ((it >> 1) - 1) & 1, p.wait_limit_ns, kSiteSlotEmpty, ab))
                    break;
                const int32_t qrow = (int32_t)((i0 + it) * BQ);
                uint8_t *st = smem + Lay::kStageOff + s * Lay::kStageBytes;
                ptx::mbar_arrive_expect_tx(&stage_full[s], 2 * Lay::kTileBytes);
                for (int c = 0; c < Lay::kChunks; ++c) {
                    ptx::tma_load_3d(st + c * Lay::kChunkBytes, &tm_q, &stage_full[s], c * 64, qrow, (int32_t)bh);
                    ptx::tma_load_3d(st + Lay::kTileBytes + c * Lay::kChunkBytes, &tm_do, &stage_full[s],
                                     c * 64, qrow, (int32_t)bh);
                }
                issued = (uint32_t)it + 1;
            }
            // Drain: every copy has landed before the CTA exits.
            wait_bounded(kv_full, 0, p.wait_limit_ns, kSiteDrain, ab, false);
            for (uint32_t it = issued >= 2 ? issued - 2 : 0; it < issued; ++it)
                wait_bounded(&stage_full[it & 1], (it >> 1) & 1, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0 && n_iter > 0) {
            const uint32_t base = ptx::smem_u32(smem);
            // K-major operands (rows of 128-byte swizzled chunks)
            const uint64_t dK_km = make_sdesc(base + Lay::kKOff, 16, 1024);
            const uint64_t dV_km = make_sdesc(base + Lay::kVOff, 16, 1024);
            // MN-major operands: 8 rows of 128 B per 1024 B group, 64-column
            // chunks one box (16 KiB) apart; a K-step of 16 rows is 2 KiB
            const uint64_t dK_mn = make_sdesc(base + Lay::kKOff, Lay::kChunkBytes, 1024);
            const uint64_t dS_mn = make_sdesc(base + Lay::kDSOff, Lay::kChunkBytes, 1024);
            constexpr uint32_t id_st = make_idesc(BK, BQ, 0, 0, kF16);   // S^T, dP^T: 128 keys x 128 queries
            constexpr uint32_t id_acc = make_idesc(BK, D, 0, 1, kF16);   // dV, dK: A in TMEM, B MN-major
            constexpr uint32_t id_dq = make_idesc(BQ, D, 1, 1, kF16);    // dQ: A = dS MN-major, B = K MN-major

            auto issue_dpt = [&](int stage) {   // dP^T = V_j dO_i^T
                const uint64_t dO_km = make_sdesc(base + Lay::kStageOff + stage * Lay::kStageBytes + Lay::kTileBytes,
                                                  16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * Lay::kChunkBytes + (k % 4) * 32) >> 4);
                    ptx::mma_ss(tmem + Lay::kColDPT, dV_km + off, dO_km + off, id_st, k > 0);
                }
            };
            // dP^T of a query tile is issued right after dQ of the one before:
            // its columns are free once dK has read dS^T and the key-row
            // threads have copied dS out (ds_ready), while S^T waits for the
            // dQ rows to leave TMEM.
            bool ok = wait_bounded(kv_full, 0, p.wait_limit_ns, kSiteQFull, ab) &&
                      wait_bounded(&stage_full[0], 0, p.wait_limit_ns, kSiteSlotFull, ab);
            if (ok) {
                ptx::tc_fence_after();
                issue_dpt(0);
            }
            for (int it = 0; it < n_iter && ok; ++it) {
                const int s = it & 1;
                const uint32_t st = base + Lay::kStageOff + s * Lay::kStageBytes;
                const uint64_t dQ_km = make_sdesc(st, 16, 1024);
                const uint64_t dQ_mn = make_sdesc(st, Lay::kChunkBytes, 1024);
                const uint64_t dO_mn = make_sdesc(st + Lay::kTileBytes, Lay::kChunkBytes, 1024);
                // dQ_{i-1} has left the S^T columns
                if (it > 0 && !wait_bounded(dq_free, (it - 1) & 1, p.wait_limit_ns, kSitePFull, ab)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * Lay::kChunkBytes + (k % 4) * 32) >> 4);
                    ptx::mma_ss(tmem + Lay::kColST, dK_km + off, dQ_km + off, id_st, k > 0);
                }
                ptx::mma_commit(s_full);
                // dV += P^T dO_i and dK += dS^T Q_i, 32 queries (two K-steps)
                // at a time as the key-row threads finish them
                bool got = true;
#pragma unroll
                for (int c = 0; c < BQ / 32; ++c) {
                    if (!(got = wait_bounded(&p_ready[c], it & 1, p.wait_limit_ns, kSitePFull, ab))) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int k = 2 * c; k < 2 * c + 2; ++k) {
                        const uint64_t off = (uint64_t)((k * 2048) >> 4);
                        ptx::mma_ts(tmem + Lay::kColDV, tmem + Lay::kColST + k * 8, dO_mn + off, id_acc,
                                    (it > 0 || k > 0) ? 1u : 0u);
                        ptx::mma_ts(tmem + Lay::kColDK, tmem + Lay::kColDPT + k * 8, dQ_mn + off, id_acc,
                                    (it > 0 || k > 0) ? 1u : 0u);
                    }
                }
                if (!got) break;
                ptx::mma_commit(&stage_empty[s]);     // Q_i, dO_i are no longer read
                if (!wait_bounded(ds_ready, it & 1, p.wait_limit_ns, kSitePFull, ab)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t off = (uint64_t)((k * 2048) >> 4);
                    ptx::mma_ss(tmem + Lay::kColST, dS_mn + off, dK_mn + off, id_dq, k > 0);
                }
                ptx::mma_commit(dq_full);
                if (it + 1 == n_iter) {
                    ptx::mma_commit(acc_full);
                } else {
                    const int s1 = (it + 1) & 1;
                    if (!wait_bounded(&stage_full[s1], ((it + 1) >> 1) & 1, p.wait_limit_ns, kSiteSlotFull, ab)) break;
                    ptx::tc_fence_after();
                    issue_dpt(s1);
                }
            }
            ptx::mma_commit(mma_drain);
            wait_bounded(mma_drain, 0, p.wait_limit_ns, kSiteDrain, ab, false);
        }
    }
    } else if (warp < kDQWarp0) {
        ptx::regs_inc<192>();
        // ================= key rows: P^T, dS^T =================
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;                      // TMEM lane: key t
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int64_t key = k0 + t;
        const bool key_ok = key < L;
        const float sl2 = p.scale_log2;
        const uint32_t ds_base = ptx::smem_u32(smem + Lay::kDSOff);
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int64_t q0 = (i0 + it) * BQ;
            // this query tile's -LSE (log2 units) and -Delta, shared by all key rows
            ptx::bar_sync(1, 128);
            {
                const int64_t qr = q0 + t;
                nlse2_s[t] = qr < N ? p.lse[bh * N + qr] * -1.4426950408889634f : -INFINITY;
                ndelta_s[t] = qr < N ? -p.delta[bh * N + qr] : 0.f;
            }
            ptx::bar_sync(1, 128);
            // all 128 threads agree on going on, so the named barriers stay matched
            ok = ptx::bar_and(1, 128, wait_bounded(s_full, it & 1, p.wait_limit_ns, kSiteSFull, ab));
            if (!ok) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BQ / 32; ++c) {
                uint32_t sv[32], dpv[32];
                ptx::tmem_ld32(tmem + lane_off + Lay::kColST + c * 32, sv);
                ptx::tmem_ld32(tmem + lane_off + Lay::kColDPT + c * 32, dpv);
                ptx::tmem_wait_ld();
                // this chunk's 32 -LSE / -Delta values as packed pairs (broadcast
                // smem reads) and the first visible query: causal hides q < key,
                // padding hides the row
                uint64_t nl2[16], nd2[16];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const ulonglong2 a2 = *reinterpret_cast<const ulonglong2 *>(&nlse2_s[c * 32 + 2 * e]);
                    const ulonglong2 d2 = *reinterpret_cast<const ulonglong2 *>(&ndelta_s[c * 32 + 2 * e]);
                    nl2[e] = a2.x; nl2[e + 1] = a2.y;
                    nd2[e] = d2.x; nd2[e + 1] = d2.y;
                }
                int e_min = 0;
                if (!key_ok) {
                    e_min = 32;
                } else if (p.causal) {
                    const int64_t d0 = key - (q0 + c * 32);
                    e_min = d0 <= 0 ? 0 : (d0 >= 32 ? 32 : (int)d0);
                }
                uint32_t pw[16], dsw[16];
                const uint64_t sl2_2 = ptx::pack2(sl2, sl2);
                if (__all_sync(0xffffffffu, e_min == 0)) {
                    // every query of the chunk sees every key of the warp: packed math
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1, d0, d1;
                        ptx::unpack2(ptx::fma2(ptx::pack2(u2f(sv[2 * e]), u2f(sv[2 * e + 1])), sl2_2, nl2[e]), x0, x1);
                        const float p0 = ptx::ex2_approx(x0);
                        const float p1 = ptx::ex2_approx(x1);
                        ptx::unpack2(ptx::mul2(ptx::pack2(p0, p1),
                                               ptx::add2(ptx::pack2(u2f(dpv[2 * e]), u2f(dpv[2 * e + 1])), nd2[e])),
                                     d0, d1);
                        pw[e] = ptx::pack16x2<kF16>(p0, p1);
                        dsw[e] = ptx::pack16x2<kF16>(d0, d1);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float nla, nlb, nda, ndb;
                        ptx::unpack2(nl2[e], nla, nlb);
                        ptx::unpack2(nd2[e], nda, ndb);
                        const float pa = 2 * e >= e_min ? ptx::ex2_approx(fmaf(u2f(sv[2 * e]), sl2, nla)) : 0.f;
                        const float pb = 2 * e + 1 >= e_min ? ptx::ex2_approx(fmaf(u2f(sv[2 * e + 1]), sl2, nlb)) : 0.f;
                        pw[e] = ptx::pack16x2<kF16>(pa, pb);
                        dsw[e] = ptx::pack16x2<kF16>(pa * (u2f(dpv[2 * e]) + nda), pb * (u2f(dpv[2 * e + 1]) + ndb));
                    }
                }
                ptx::tmem_st16(tmem + lane_off + Lay::kColST + c * 16, pw);
                ptx::tmem_st16(tmem + lane_off + Lay::kColDPT + c * 16, dsw);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&p_ready[c]);   // the products over these 32 queries may start
            }

            // dS (row t = key t) into the MN-major, 128-byte-swizzled A operand
            // of dQ = dS K, once the staging of dQ_{i-1} has left the buffer;
            // the bf16 pairs are read back from the dS^T columns of TMEM.
            if (it > 0) {
                ok = ptx::bar_and(1, 128, wait_bounded(ds_free, (it - 1) & 1, p.wait_limit_ns, kSitePFull, ab));
                if (!ok) break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int h = 0; h < BQ / 64; ++h) {
                uint32_t dsv[32];
                ptx::tmem_ld32(tmem + lane_off + Lay::kColDPT + h * 32, dsv);
                ptx::tmem_wait_ld();
                // 32 words = 64 queries = 8 units of 8 queries
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t unit = (uint32_t)u ^ (uint32_t)(t & 7);
                    const uint32_t addr = ds_base + (uint32_t)h * Lay::kChunkBytes + (uint32_t)t * 128u + (unit << 4);
                    ptx::st_shared_v4(addr, dsv[4 * u], dsv[4 * u + 1], dsv[4 * u + 2], dsv[4 * u + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ds_ready);
        }

        // ---- dK (times scale) and dV of this key tile ------------------------
        bool have = ok && n_iter > 0;
        if (n_iter > 0)
            have = ptx::bar_and(1, 128, have && wait_bounded(acc_full, 0, p.wait_limit_ns, kSiteOFinal, ab));
        if (have || n_iter == 0) {
            ptx::tc_fence_after();
            const int Dv = (int)p.D;                            // real columns (a multiple of 8, <= D)
            uint16_t *dk_row = static_cast<uint16_t *>(p.dk) + (bh * N + key) * Dv;
            uint16_t *dv_row = static_cast<uint16_t *>(p.dv) + (bh * N + key) * Dv;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which ? Lay::kColDK : Lay::kColDV;
                const float mul = which ? p.scale : 1.f;
                uint16_t *dst_row = which ? dk_row : dv_row;
#pragma unroll 1
                for (int c = 0; c < D / 32 && c * 32 < Dv; ++c) {
                    uint32_t v[32];
                    if (n_iter > 0) {
                        ptx::tmem_ld32(tmem + lane_off + col + c * 32, v);
                        ptx::tmem_wait_ld();
                    }
                    if (key < N) {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = n_iter > 0 ? ptx::pack16x2<kF16>(u2f(v[2 * e]) * mul, u2f(v[2 * e + 1]) * mul) : 0u;
                        uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (c * 32 + 8 * e < Dv)
                                dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
            }
        }
    } else {
        ptx::regs_inc<192>();
        // ================= query rows: dQ_i into the fp32 accumulator =================
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;                      // TMEM lane: query q0 + t
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float *stage = reinterpret_cast<float *>(smem + Lay::kDSOff);
        const int Dv = (int)p.D;                                // real columns (a multiple of 8, <= D)
        for (int it = 0; it < n_iter; ++it) {
            const int64_t q0 = (i0 + it) * BQ;
            if (!ptx::bar_and(2, 128, wait_bounded(dq_full, it & 1, p.wait_limit_ns, kSiteOFinal, ab))) break;
            ptx::tc_fence_after();
            // dQ_i goes to registers first, so that TMEM is handed back to the
            // next S^T at once.  Each 32-column chunk is then staged in the dS
            // buffer (free: dQ = dS K has read it) as a 128-row x 128-byte box
            // with the 16-byte units of row r XOR-swizzled by (r & 7) -- the
            // shared-memory form of a 128-byte-swizzled TMA box -- and one
            // thread hands it to the TMA engine, which adds it into the fp32
            // accumulator (rows at or past N are clipped by the tensor map).
            uint32_t dqv[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tmem + lane_off + Lay::kColST + c * 32, dqv[c]);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(dq_free);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if (c * 32 >= Dv) break;                 // zero padding past the real columns
                float *buf = stage + (c & 1) * (BQ * 32);
                if (c >= 2) {
                    // the reduce that read this buffer two chunks ago is done
                    if (t == 0) ptx::bulk_wait_group_read<1>();
                    ptx::bar_sync(2, 128);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    *reinterpret_cast<uint4 *>(buf + t * 32 + ((e ^ (t & 7)) << 2)) =
                        make_uint4(dqv[c][4 * e], dqv[c][4 * e + 1], dqv[c][4 * e + 2], dqv[c][4 * e + 3]);
                ptx::fence_proxy_async_smem();
                ptx::bar_sync(2, 128);
                if (t == 0) {
                    ptx::tma_reduce_add_3d(&tm_dq, buf, c * 32, (int32_t)q0, (int32_t)bh);
                    ptx::bulk_commit_group();
                }
            }
            // the buffer is the next tile's dS: hand it back once read
            if (t == 0) {
                ptx::bulk_wait_group_read<0>();
                ptx::mbar_arrive(ds_free);
            }
        }
        // every reduce-add issued here has reached global memory
        if (t == 0) ptx::bulk_wait_group_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// Delta = rowsum(dO * O) per query row (over the D real columns), and the
// zeroed fp32 dQ accumulator.  One warp per row.
template <bool kF16>
__device__ __forceinline__ float f16_to_f32(uint16_t x)
{
    if constexpr (kF16)
        return __half2float(__ushort_as_half(x));
    else
        return __uint_as_float((uint32_t)x << 16);
}

template <bool kF16>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ d_o,
                float *__restrict__ delta, float *__restrict__ dq_acc, int64_t rows, int D)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    float s = 0.f;
    for (int c = lane; c < D; c += 32) {
        const int64_t idx = row * D + c;
        s = fmaf(f16_to_f32<kF16>(o[idx]), f16_to_f32<kF16>(d_o[idx]), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) delta[row] = s;
    for (int c = lane; c < D; c += 32) dq_acc[row * D + c] = 0.f;
}

// dQ = scale * accumulator, rounded to bf16 / fp16 (two elements per thread).
template <bool kF16>
__global__ void __launch_bounds__(256)
bwd_dq_kernel(const float *__restrict__ dq_acc, uint16_t *__restrict__ dq, float scale, int64_t n2)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n2) return;
    const float2 v = reinterpret_cast<const float2 *>(dq_acc)[i];
    reinterpret_cast<uint32_t *>(dq)[i] = ptx::pack16x2<kF16>(v.x * scale, v.y * scale);
}

template <int D, bool kF16>
cudaError_t launch_bwd_d(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tdo, const CUtensorMap &tdq,
                         cudaStream_t stream)
{
    using Lay = BwdLayout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Lay::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = p.B * p.H * p.N;
    bwd_prep_kernel<kF16><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const uint16_t *>(p.o), static_cast<const uint16_t *>(p.d_o), p.delta, p.dq_acc, rows,
        (int)p.D);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ctas = p.B * p.H * ((p.N + BK - 1) / BK);
    bwd_kernel<D, kF16><<<(unsigned)ctas, kThreads, Lay::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n2 = rows * p.D / 2;
    bwd_dq_kernel<kF16><<<(unsigned)((n2 + 255) / 256), 256, 0, stream>>>(p.dq_acc, static_cast<uint16_t *>(p.dq),
                                                                  p.scale, n2);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_do, const CUtensorMap &tm_dq,
                            cudaStream_t stream)
{
    // D a multiple of 8 below 128 runs at the next of 64 / 128: the TMA boxes
    // fill the columns past D with zeros, which adds nothing to any product,
    // and only the D real columns of dQ, dK and dV are written.
    if (p.D % 8 != 0 || p.D <= 0 || p.D > 128) return cudaErrorInvalidValue;
    if (p.D <= 64)
        return p.f16 ? launch_bwd_d<64, true>(p, tm_q, tm_k, tm_v, tm_do, tm_dq, stream)
                     : launch_bwd_d<64, false>(p, tm_q, tm_k, tm_v, tm_do, tm_dq, stream);
    return p.f16 ? launch_bwd_d<128, true>(p, tm_q, tm_k, tm_v, tm_do, tm_dq, stream)
                 : launch_bwd_d<128, false>(p, tm_q, tm_k, tm_v, tm_do, tm_dq, stream);
}

cudaError_t read_and_clear_status_bwd(uint32_t *out)
{
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_bwd, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_bwd, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace fa
