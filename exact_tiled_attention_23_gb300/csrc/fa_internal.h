// fa_internal.h -- declarations shared by the host launcher and the kernels
// of the attention library (not part of the public C ABI).
#pragma once

#include "fa.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

// The tensor-core forward's kernel for a problem of these sizes, as fa_fwd /
// fa_fwd_f16 choose it: 1 = one query tile per CTA, 2 = two tiles per CTA,
// 3 = one tile per CTA with each row's keys split between two softmax
// warpgroups.
int fwd16_tiles(int B, int H, int N, int D);

// fa_fwd (f16: fa_fwd_f16) with the kernel fixed by `tiles` (1, 2 or 3), for
// callers that split one problem into several launches and want every part
// computed as one whole call would compute it: the kernels agree only to
// rounding, not bit for bit.
fa_status fwd16_with_tiles(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                           int N, int D, int causal, float scale, const int32_t *kv_len, bool f16, int tiles,
                           void *stream);

// Device-side status word.  Kernels OR an error code into the low byte and
// record the site of the first give-up in the upper bits; the host reads and
// clears it in fa_device_status.
enum : uint32_t {
    kStatusTimeout = 0x1u,
};

// Site codes of the bounded waits (upper 24 bits of the status word).
enum WaitSite : uint32_t {
    kSiteQFull = 1,
    kSiteSlotFull = 2,
    kSiteSlotEmpty = 3,
    kSiteSFull = 4,
    kSitePFull = 5,
    kSiteOFinal = 6,
    kSiteDrain = 7,
};

// Arguments common to both forward kernels.  Pointers are device pointers.
struct FwdParams {
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;               // may be null
    const int32_t *kv_len;    // may be null (= N)
    int64_t B, H, N, D;
    int causal;
    int f16;                  // 16-bit operand type of the tensor-core path: 0 = bf16, 1 = fp16
    float scale;              // natural-log scale applied to Q K^T
    float scale_log2;         // scale * log2(e)
    uint64_t wait_limit_ns;   // bounded-wait budget of every mbarrier wait
    // split-KV only: key blocks of every query item are divided into
    // num_splits contiguous ranges; range s writes its normalised partial
    // output part_o[s][B*H*N][D] (fp32) and part_lse[s][B*H*N].
    int num_splits;
    float *part_o;
    float *part_lse;
    // split-row kernel only: heads per group of its CTA order (>= 1; the
    // launcher sets it)
    int head_group;
};

// Arguments of the backward pass (bf16 or fp16 tensors, fp32 LSE and workspace).
struct BwdParams {
    const void *q, *k, *v, *o, *d_o;
    const float *lse;
    void *dq, *dk, *dv;
    const int32_t *kv_len;    // may be null (= N)
    int64_t B, H, N, D;
    int causal;
    int f16;                  // 16-bit type of Q, K, V, O, dO and the gradients: 0 = bf16, 1 = fp16
    float scale;
    float scale_log2;
    uint64_t wait_limit_ns;
    float *delta;             // workspace: rowsum(dO * O), [B*H*N]
    float *dq_acc;            // workspace: fp32 dQ accumulator, [B*H*N*D]
};

// Launchers (return the CUDA error of the launch).
cudaError_t launch_fwd_fp32(const FwdParams &p, cudaStream_t stream);
cudaError_t launch_fwd_bf16(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream);

// One 128-row query tile per CTA: head dimension 256, and grids too small for
// the two-tile kernel to fill the GPU.
cudaError_t launch_fwd_onetile(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream);

// One 128-row query tile per CTA, each row's keys split between two softmax
// warpgroups with separate online-softmax states, merged in the epilogue
// (D <= 128).
cudaError_t launch_fwd_halves(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t stream);

// Split-KV forward: partial kernel over key-block ranges, then the merge.
cudaError_t launch_fwd_bf16_split(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                  const CUtensorMap &tm_v, cudaStream_t stream);

// Backward: Delta / accumulator preparation, the tensor-core kernel, dQ.
cudaError_t launch_bwd_bf16(const BwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_do, const CUtensorMap &tm_dq,
                            cudaStream_t stream);

// Read-and-clear of the device status word (synchronises `stream` first).
cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *out);
// The backward kernels' status word (call after read_and_clear_status).
cudaError_t read_and_clear_status_bwd(uint32_t *out);
// The one-tile forward kernel's status word (call after read_and_clear_status).
cudaError_t read_and_clear_status_onetile(uint32_t *out);
// The split-row forward kernel's status word (call after read_and_clear_status).
cudaError_t read_and_clear_status_halves(uint32_t *out);

}  // namespace fa
