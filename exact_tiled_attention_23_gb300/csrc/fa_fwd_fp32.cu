// fa_fwd_fp32.cu -- fp32 attention forward on the CUDA cores.
//
// One warp owns one query row.  Keys are visited in chunks of 32: lane t
// forms the full dot product of the row with key (chunk + t), the warp takes
// the chunk's max and sum by shuffles, and every lane keeps D/32 columns of
// the running numerator.  The running state (m, l, acc) follows the online
// softmax of "vectorized-flash-attention-kernel", Core algorithm step 3: a
// chunk that raises the max rescales l and acc by exp(m_old - m_new).  A row
// whose mask hides every key skips the loop and writes exact zeros and
// LSE = -inf ("js-flash-attention-tiled-online-softmax-exactness", Root
// causes 2).  All arithmetic is fp32 multiply-add (no TF32), exp and log
// are the CUDA fp32 functions.
#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kMaxD = 256;

template <int DC>   // DC = ceil(D / 32) columns per lane
__global__ void __launch_bounds__(kWarpsPerCta * 32)
fwd_fp32_kernel(FwdParams p)
{
    __shared__ float q_sm[kWarpsPerCta][kMaxD];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t N = p.N, D = p.D;
    const int64_t row_blocks = (N + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t head = (int64_t)blockIdx.x / row_blocks;       // b * H + h
    const int64_t row = ((int64_t)blockIdx.x % row_blocks) * kWarpsPerCta + warp;
    if (row >= N) return;
    const int64_t b = head / p.H;

    int64_t L = N;
    if (p.kv_len) {
        L = p.kv_len[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    int64_t nkeys = L;
    if (p.causal && row + 1 < nkeys) nkeys = row + 1;

    const float *Q = static_cast<const float *>(p.q) + (head * N + row) * D;
    const float *K = static_cast<const float *>(p.k) + head * N * D;
    const float *V = static_cast<const float *>(p.v) + head * N * D;
    float *O = static_cast<float *>(p.o) + (head * N + row) * D;

    for (int64_t d = lane; d < D; d += 32) q_sm[warp][d] = Q[d];
    __syncwarp();

    float m = -INFINITY, l = 0.f;
    float acc[DC];
#pragma unroll
    for (int c = 0; c < DC; ++c) acc[c] = 0.f;

    for (int64_t base = 0; base < nkeys; base += 32) {
        const int64_t j = base + lane;
        float s = -INFINITY;
        if (j < nkeys) {
            const float *k = K + j * D;
            float dot = 0.f;
            for (int64_t d = 0; d < D; ++d) dot = fmaf(q_sm[warp][d], k[d], dot);
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
        const int cnt = (nkeys - base) < 32 ? (int)(nkeys - base) : 32;
        for (int t = 0; t < cnt; ++t) {
            const float pt = __shfl_sync(0xffffffffu, pj, t);
            const float *v = V + (base + t) * D;
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const int64_t d = lane + 32 * c;
                if (d < D) acc[c] = fmaf(pt, v[d], acc[c]);
            }
        }
        m = m_new;
    }

    const bool empty = (nkeys <= 0);
    const float inv = empty ? 0.f : 1.f / l;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        const int64_t d = lane + 32 * c;
        if (d < D) O[d] = empty ? 0.f : acc[c] * inv;
    }
    if (p.lse && lane == 0) p.lse[head * N + row] = empty ? -INFINITY : m + logf(l);
}

template <int DC>
cudaError_t launch_dc(const FwdParams &p, cudaStream_t stream)
{
    const int64_t blocks = p.B * p.H * ((p.N + kWarpsPerCta - 1) / kWarpsPerCta);
    fwd_fp32_kernel<DC><<<(unsigned)blocks, kWarpsPerCta * 32, 0, stream>>>(p);
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
