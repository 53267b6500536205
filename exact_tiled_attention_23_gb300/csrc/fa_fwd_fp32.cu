// fa_fwd_fp32.cu -- fp32 attention forward on the CUDA cores.
//
// A CTA of four warps owns four consecutive query rows of one head, one row
// per warp.  Keys are visited in tiles of 32 that the CTA stages in shared
// memory by asynchronous copies, double-buffered so that the next tile loads
// while this one is used (K rows padded to D+1 floats so that lanes reading
// different keys hit different banks).  In a tile, lane t forms the full dot
// product of its warp's row with key (tile start + t), the warp takes the
// tile's max and sum by shuffles, and every lane keeps D/32 columns of the
// running numerator.  The running state
// (m, l, acc) follows the online softmax of "vectorized-flash-attention-
// kernel", Core algorithm step 3: a chunk that raises the max rescales l and
// acc by exp(m_old - m_new).  A row whose mask hides every key writes exact
// zeros and LSE = -inf ("js-flash-attention-tiled-online-softmax-exactness",
// Root causes 2).  All arithmetic is fp32 multiply-add (no TF32); exp and log
// are the CUDA fp32 functions.
#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr int kRows = 4;      // query rows (= warps) per CTA
constexpr int kKeyTile = 32;  // keys staged per tile (= one chunk of a warp)
constexpr int kMaxD = 256;

// 4-byte asynchronous global -> shared copy (no register staging), so that
// every element of a tile is in flight at once.
__device__ __forceinline__ void cp_async4(float *dst, const float *src)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(kPending) : "memory"); }

__host__ __device__ constexpr size_t smem_floats(int D)
{
    // two K tiles [kKeyTile][D+1], two V tiles [kKeyTile][D], Q rows [kRows][D]
    return 2 * (size_t)kKeyTile * (D + 1) + 2 * (size_t)kKeyTile * D + (size_t)kRows * D;
}

template <int DC>   // DC = ceil(D / 32) output columns per lane
__global__ void __launch_bounds__(kRows * 32)
fwd_fp32_kernel(FwdParams p)
{
    extern __shared__ float sm[];
    const int64_t N = p.N;
    const int D = (int)p.D;
    const int ks_stride = D + 1;
    float *Ks = sm;                                  // [2][kKeyTile][D+1]
    float *Vs = Ks + 2 * kKeyTile * ks_stride;       // [2][kKeyTile][D]
    float *Qs = Vs + 2 * kKeyTile * D;               // [kRows][D]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t row_blocks = (N + kRows - 1) / kRows;
    const int64_t head = (int64_t)blockIdx.x / row_blocks;       // b * H + h
    const int64_t r0 = ((int64_t)blockIdx.x % row_blocks) * kRows;
    const int64_t row = r0 + warp;
    const int64_t b = head / p.H;

    int64_t L = N;
    if (p.kv_len) {
        L = p.kv_len[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    // keys this row sees, and the most any row of the CTA sees
    int64_t nkeys = row < N ? L : 0;
    if (p.causal && row + 1 < nkeys) nkeys = row + 1;
    int64_t ncta = L;
    if (p.causal) {
        const int64_t last = (r0 + kRows < N ? r0 + kRows : N);   // one past the CTA's last row
        if (last < ncta) ncta = last;
    }
    const int ntiles = (int)((ncta + kKeyTile - 1) / kKeyTile);

    const float *Q = static_cast<const float *>(p.q) + head * N * D;
    const float *K = static_cast<const float *>(p.k) + head * N * D;
    const float *V = static_cast<const float *>(p.v) + head * N * D;

    // keys [kt, kt + cnt) into buffer `buf`
    auto issue_tile = [&](int buf, int64_t kt) {
        const int cnt = (int)((ncta - kt) < kKeyTile ? (ncta - kt) : kKeyTile);
        const float *Kt = K + kt * D;
        const float *Vt = V + kt * D;
        float *Kb = Ks + buf * kKeyTile * ks_stride;
        float *Vb = Vs + buf * kKeyTile * D;
        for (int i = tid; i < cnt * D; i += kRows * 32) {
            const int j = i / D, d = i - j * D;
            cp_async4(Kb + j * ks_stride + d, Kt + i);
            cp_async4(Vb + i, Vt + i);
        }
    };

    const int q_rows = (int)((N - r0) < kRows ? (N - r0) : kRows);
    for (int i = tid; i < q_rows * D; i += kRows * 32) cp_async4(Qs + i, Q + r0 * D + i);
    if (ntiles > 0) issue_tile(0, 0);
    cp_async_commit();

    float m = -INFINITY, l = 0.f;
    float acc[DC];
#pragma unroll
    for (int c = 0; c < DC; ++c) acc[c] = 0.f;
    const float *q = Qs + warp * D;

    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) {
            issue_tile((t + 1) & 1, (int64_t)(t + 1) * kKeyTile);   // prefetch the next tile
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();   // tile t (and Q) visible to every warp
        const int64_t base = (int64_t)t * kKeyTile;
        if (base < nkeys) {
            const float *Kb = Ks + (t & 1) * kKeyTile * ks_stride;
            const float *Vb = Vs + (t & 1) * kKeyTile * D;
            const int64_t j = base + lane;
            float s = -INFINITY;
            if (j < nkeys) {
                const float *k = Kb + lane * ks_stride;
                float dot = 0.f;
#pragma unroll 8
                for (int d = 0; d < D; ++d) dot = fmaf(q[d], k[d], dot);
                s = p.scale * dot;
            }
            float cmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
            const float m_new = fmaxf(m, cmax);          // finite: key `base` is visible
            const float corr = expf(m - m_new);          // m = -inf on the first chunk -> 0
            const float pj = (j < nkeys) ? expf(s - m_new) : 0.f;
            float psum = pj;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l = l * corr + psum;
#pragma unroll
            for (int c = 0; c < DC; ++c) acc[c] *= corr;
            const int n = (nkeys - base) < kKeyTile ? (int)(nkeys - base) : kKeyTile;
            for (int u = 0; u < n; ++u) {
                const float pt = __shfl_sync(0xffffffffu, pj, u);
                const float *v = Vb + u * D;
#pragma unroll
                for (int c = 0; c < DC; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) acc[c] = fmaf(pt, v[d], acc[c]);
                }
            }
            m = m_new;
        }
        __syncthreads();   // every warp is done with buffer t & 1 before it is refilled
    }
    cp_async_wait<0>();    // no copy outlives the CTA (a CTA with no keys still loaded Q)

    if (row >= N) return;
    float *O = static_cast<float *>(p.o) + (head * N + row) * D;
    const bool empty = (nkeys <= 0);
    const float inv = empty ? 0.f : 1.f / l;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        const int d = lane + 32 * c;
        if (d < D) O[d] = empty ? 0.f : acc[c] * inv;
    }
    if (p.lse && lane == 0) p.lse[head * N + row] = empty ? -INFINITY : m + logf(l);
}

template <int DC>
cudaError_t launch_dc(const FwdParams &p, cudaStream_t stream)
{
    const size_t smem = sizeof(float) * smem_floats((int)p.D);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fwd_fp32_kernel<DC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(sizeof(float) * smem_floats(kMaxD)));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t blocks = p.B * p.H * ((p.N + kRows - 1) / kRows);
    fwd_fp32_kernel<DC><<<(unsigned)blocks, kRows * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp32(const FwdParams &p, cudaStream_t stream)
{
    const int dc = (int)((p.D + 31) / 32);
    switch (dc) {
    case 1: return launch_dc<1>(p, stream);
    case 2: return launch_dc<2>(p, stream);
    case 3: return launch_dc<3>(p, stream);
    case 4: return launch_dc<4>(p, stream);
    case 5: return launch_dc<5>(p, stream);
    case 6: return launch_dc<6>(p, stream);
    case 7: return launch_dc<7>(p, stream);
    case 8: return launch_dc<8>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
