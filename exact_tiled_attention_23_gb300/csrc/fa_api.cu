// fa_api.cu -- the C ABI of the attention library: argument checks, the TMA
// tensor maps, and the kernel launches.  Declared in include/fa.h.
//
// Every check that can fail runs before any CUDA call, so a rejected call has
// no side effect.  The library allocates no device memory.
#include "fa.h"
#include "fa_internal.h"

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

uint32_t g_last_detail = 0;

// Default bounded-wait budget: far above any legitimate wait (one key block
// takes microseconds), short enough that a stuck kernel ends on its own.
uint64_t wait_limit_ns()
{
    static uint64_t v = [] {
        const char *e = std::getenv("FA_WAIT_LIMIT_MS");
        double ms = e ? std::atof(e) : 4000.0;
        if (!(ms > 0)) ms = 4000.0;
        return (uint64_t)(ms * 1e6);
    }();
    return v;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The tensor-core forward kernel that FA_FWD_TILES asks for: "1" (one query
// tile per CTA), "2" (two tiles per CTA) or "3" (one tile, split rows), else
// 0 (the automatic choice).  Read on every call, so that a process can
// compare the kernels.
int forced_tiles()
{
    const char *e = std::getenv("FA_FWD_TILES");
    if (!e) return 0;
    if (e[0] >= '1' && e[0] <= '3' && e[1] == 0) return e[0] - '0';
    return 0;
}

// SMs of the current device (148 if it cannot be read).
int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    return sms;
}

// Head dimensions of the tensor-core kernels that zero-pad to 64 / 128 (the
// forward, its split-KV form and the backward): multiples of 8 (a TMA row
// stride must be a multiple of 16 bytes) up to 128.
bool tc_fwd_head_dim(int D) { return D > 0 && D <= 128 && D % 8 == 0; }

fa_status check_common(const void *Q, const void *K, const void *V, const void *O, int B, int H,
                       int N, int D)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0) return FA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)B * H * N;
    if (rows == 0) return FA_OK;
    if (!Q || !K || !V || !O) return FA_ERR_INVALID_ARG;
    // element counts must stay addressable with 64-bit offsets and fit the grid
    if (rows > (int64_t)1 << 40 || (int64_t)B * H > INT32_MAX) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

float resolve_scale(float scale, int D)
{
    if (std::isnan(scale) || !(scale > 0.f) || std::isinf(scale)) return 1.0f / std::sqrt((float)D);
    return scale;
}

fa::FwdParams make_params(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                          int H, int N, int D, int causal, float scale, const int32_t *kv_len)
{
    fa::FwdParams p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.lse = LSE;
    p.kv_len = kv_len;
    p.B = B;
    p.H = H;
    p.N = N;
    p.D = D;
    p.causal = causal ? 1 : 0;
    p.scale = resolve_scale(scale, D);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.wait_limit_ns = wait_limit_ns();
    p.f16 = 0;
    p.num_splits = 1;
    p.part_o = nullptr;
    p.part_lse = nullptr;
    return p;
}

// 3-D map over a contiguous [B*H, N, D] array of 16-bit elements: box = 64
// columns x 128 rows of one head, 128-byte swizzle, zero fill outside [0, N)
// so a box never reads the next head's rows.
bool encode_map16(CUtensorMap *m, const void *base, int64_t BH, int64_t N, int64_t D,
                  CUtensorMapDataType dtype)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dtype, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over the fp32 dQ accumulator [B*H, N, D]: box = 32 columns (128 B)
// x 128 rows, 128-byte swizzle; rows past N are clipped by reduce-adds.
bool encode_dq_acc_map(CUtensorMap *m, const void *base, int64_t BH, int64_t N, int64_t D)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)N * D * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_map(CUtensorMap *m, const void *base, int64_t BH, int64_t N, int64_t D)
{
    return encode_map16(m, base, BH, N, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// The kernel the tensor-core forward runs for a problem (measured on GB300):
//   1: one 128-row query tile per CTA -- D = 256, and grids of D <= 64 whose
//      twice as many one-tile CTAs still fit in one wave (one CTA per SM);
//   3: one tile per CTA, each row's keys split between two softmax
//      warpgroups -- 64 < D <= 128 with long rows (N >= 8192), where it runs
//      ahead of the two-tile kernel, or with such small grids;
//   2: two tiles per CTA (work item: 256 query rows of one head) otherwise,
//      where it runs ahead: D <= 64, and shorter rows (whose per-tile ramp the
//      two-tile kernel amortises over twice the rows).
int choose_tiles(int B, int H, int N, int D)
{
    const int64_t items = (int64_t)B * H * (((int64_t)N + 255) / 256);
    const int forced = forced_tiles();
    if (D == 256) return 1;
    if (forced != 0) return forced;
    const bool small_grid = 2 * items <= sm_count();
    if (D > 64) return (small_grid || N >= 8192) ? 3 : 2;
    return small_grid ? 1 : 2;
}

// Shared checks and launch of the single-pass tensor-core kernel.  tiles: the
// kernel (1, 2 or 3), or 0 for choose_tiles on this call's sizes.
fa_status fwd16(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                int N, int D, int causal, float scale, const int32_t *kv_len, void *stream, bool f16,
                int tiles = 0)
{
    fa_status st = check_common(Q, K, V, O, B, H, N, D);
    if (st != FA_OK) return st;
    if ((int64_t)B * H * N == 0) return FA_OK;
    if (!tc_fwd_head_dim(D) && D != 256) return FA_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return FA_ERR_INVALID_ARG;
    if (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return FA_ERR_INVALID_ARG;
    if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
    if (tiles == 0) tiles = choose_tiles(B, H, N, D);
    if (tiles < 1 || tiles > 3 || (tiles != 1 && D == 256)) return FA_ERR_INVALID_ARG;
    const bool one_tile = tiles != 2;
    // The grid is 1-D.
    const int64_t items = (int64_t)B * H * (((int64_t)N + 255) / 256);
    const int64_t ctas = one_tile ? (int64_t)B * H * (((int64_t)N + 127) / 128) : items;
    if (ctas > INT32_MAX) return FA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv, to;
    if (!encode_map16(&tq, Q, BH, N, D, dt) || !encode_map16(&tk, K, BH, N, D, dt) ||
        !encode_map16(&tv, V, BH, N, D, dt) || !encode_map16(&to, O, BH, N, D, dt))
        return FA_ERR_CUDA;
    fa::FwdParams p = make_params(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len);
    p.f16 = f16 ? 1 : 0;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = tiles == 1   ? fa::launch_fwd_onetile(p, tq, tk, tv, to, cs)
                    : tiles == 3 ? fa::launch_fwd_halves(p, tq, tk, tv, to, cs)
                                 : fa::launch_fwd_bf16(p, tq, tk, tv, to, cs);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Shared checks and launches of the backward (bf16 or fp16 tensors).
fa_status bwd16(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                int causal, float scale, const int32_t *kv_len, void *workspace,
                size_t workspace_bytes, void *stream, bool f16)
{
    fa_status st = check_common(Q, K, V, dQ, B, H, N, D);
    if (st != FA_OK) return st;
    if ((int64_t)B * H * N == 0) return FA_OK;
    if (!O || !dO || !LSE || !dK || !dV || !workspace) return FA_ERR_INVALID_ARG;
    if (!tc_fwd_head_dim(D)) return FA_ERR_UNSUPPORTED;
    const void *ptrs16[] = {Q, K, V, O, dO, dQ, dK, dV, workspace};
    for (const void *ptr : ptrs16)
        if (!aligned16(ptr)) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(LSE) & 3u) || (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)))
        return FA_ERR_INVALID_ARG;
    if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, D)) return FA_ERR_INVALID_ARG;
    const int64_t ctas = (int64_t)B * H * (((int64_t)N + 127) / 128);
    if (ctas > INT32_MAX) return FA_ERR_INVALID_ARG;

    const int64_t BH = (int64_t)B * H;
    CUtensorMap tq, tk, tv, tdo, tdq;
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_map16(&tq, Q, BH, N, D, dt) || !encode_map16(&tk, K, BH, N, D, dt) ||
        !encode_map16(&tv, V, BH, N, D, dt) || !encode_map16(&tdo, dO, BH, N, D, dt) ||
        !encode_dq_acc_map(&tdq, workspace, BH, N, D))
        return FA_ERR_CUDA;
    fa::BwdParams p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.d_o = dO;
    p.lse = LSE;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.kv_len = kv_len;
    p.B = B;
    p.H = H;
    p.N = N;
    p.D = D;
    p.causal = causal ? 1 : 0;
    p.f16 = f16 ? 1 : 0;
    p.scale = resolve_scale(scale, D);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.wait_limit_ns = wait_limit_ns();
    p.dq_acc = static_cast<float *>(workspace);
    p.delta = p.dq_acc + (size_t)BH * N * D;
    cudaError_t e = fa::launch_bwd_bf16(p, tq, tk, tv, tdo, tdq, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace fa {

int fwd16_tiles(int B, int H, int N, int D) { return choose_tiles(B, H, N, D); }

fa_status fwd16_with_tiles(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                           int N, int D, int causal, float scale, const int32_t *kv_len, bool f16, int tiles,
                           void *stream)
{
    return fwd16(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream, f16, tiles);
}

}  // namespace fa

extern "C" {

fa_status fa_fwd_f16(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                     int N, int D, int causal, float scale, const int32_t *kv_len, void *stream)
{
    return fwd16(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream, true);
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                 int N, int D, int causal, float scale, const int32_t *kv_len, void *stream)
{
    return fwd16(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream, false);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0 || num_splits < 0 || num_splits > FA_MAX_SPLITS) return 0;
    if (num_splits == 0) num_splits = fa_fwd_splitkv_auto_splits(B, H, N, D);
    return (size_t)num_splits * (size_t)B * (size_t)H * (size_t)N * ((size_t)D + 1) * sizeof(float);
}

int fa_fwd_kernel_choice(int B, int H, int N, int D)
{
    if (!tc_fwd_head_dim(D) && D != 256) return 0;
    return choose_tiles(B < 0 ? 0 : B, H < 0 ? 0 : H, N < 0 ? 0 : N, D);
}

int fa_fwd_splitkv_auto_splits(int B, int H, int N, int D)
{
    if (B <= 0 || H <= 0 || N <= 0) return 1;
    const int sms = sm_count();
    const int64_t items = (int64_t)B * H * (((int64_t)N + 255) / 256);
    // Measured on GB300: splitting pays only at D <= 64 with long rows (N >=
    // 4096) whose single-pass grid (2 * items one-tile CTAs) leaves SMs idle.
    // At 64 < D <= 128 the split-row kernel runs these problems faster, and
    // below N = 4096 the merge launch costs more than the shorter ranges save.
    if (D > 64 || N < 4096 || 2 * items >= sms) return 1;
    // one CTA per SM (shared memory), so fill one wave without a ragged second
    // one, and keep at least two key blocks in every range
    const int64_t blocks = ((int64_t)N + 127) / 128;
    int64_t s = items >= sms ? 1 : sms / items;
    if (s > blocks / 2) s = blocks / 2;
    if (s > FA_MAX_SPLITS) s = FA_MAX_SPLITS;
    return s < 1 ? 1 : (int)s;
}

fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                         int H, int N, int D, int causal, float scale, const int32_t *kv_len,
                         int num_splits, void *workspace, size_t workspace_bytes, void *stream)
{
    fa_status st = check_common(Q, K, V, O, B, H, N, D);
    if (st != FA_OK) return st;
    if ((int64_t)B * H * N == 0) return FA_OK;
    if (!tc_fwd_head_dim(D)) return FA_ERR_UNSUPPORTED;
    if (num_splits < 0 || num_splits > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return FA_ERR_INVALID_ARG;
    if (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return FA_ERR_INVALID_ARG;
    if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return FA_ERR_INVALID_ARG;
    if (num_splits == 0) num_splits = fa_fwd_splitkv_auto_splits(B, H, N, D);
    if (workspace_bytes < fa_fwd_splitkv_workspace_bytes(B, H, N, D, num_splits)) return FA_ERR_INVALID_ARG;
    // One range is the whole key sequence: the single-pass kernel computes
    // it directly, without the partial pass and the merge.
    if (num_splits == 1) return fwd16(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len, stream, false);
    const int64_t items = (int64_t)B * H * (((int64_t)N + 255) / 256);
    if (items * num_splits > INT32_MAX) return FA_ERR_INVALID_ARG;

    const int64_t BH = (int64_t)B * H;
    CUtensorMap tq, tk, tv;
    if (!encode_bf16_map(&tq, Q, BH, N, D) || !encode_bf16_map(&tk, K, BH, N, D) ||
        !encode_bf16_map(&tv, V, BH, N, D))
        return FA_ERR_CUDA;
    fa::FwdParams p = make_params(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len);
    p.num_splits = num_splits;
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = p.part_o + (size_t)num_splits * BH * N * D;
    cudaError_t e = fa::launch_fwd_bf16_split(p, tq, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp32(const float *Q, const float *K, const float *V, float *O, float *LSE, int B,
                      int H, int N, int D, int causal, float scale, const int32_t *kv_len,
                      void *stream)
{
    fa_status st = check_common(Q, K, V, O, B, H, N, D);
    if (st != FA_OK) return st;
    if ((int64_t)B * H * N == 0) return FA_OK;
    if (D > 256) return FA_ERR_UNSUPPORTED;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                          reinterpret_cast<uintptr_t>(LSE) | reinterpret_cast<uintptr_t>(kv_len);
    if (mis & 3u) return FA_ERR_INVALID_ARG;
    const int64_t blocks = (int64_t)B * H * (((int64_t)N + 3) / 4);
    if (blocks > INT32_MAX) return FA_ERR_INVALID_ARG;
    const fa::FwdParams p = make_params(Q, K, V, O, LSE, B, H, N, D, causal, scale, kv_len);
    cudaError_t e = fa::launch_fwd_fp32(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int D)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0) return 0;
    return (size_t)B * (size_t)H * (size_t)N * ((size_t)D + 1) * sizeof(float);
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                 int causal, float scale, const int32_t *kv_len, void *workspace,
                 size_t workspace_bytes, void *stream)
{
    return bwd16(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, causal, scale, kv_len, workspace,
                 workspace_bytes, stream, false);
}

fa_status fa_bwd_f16(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                     int causal, float scale, const int32_t *kv_len, void *workspace,
                     size_t workspace_bytes, void *stream)
{
    return bwd16(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, causal, scale, kv_len, workspace,
                 workspace_bytes, stream, true);
}

const char *fa_status_string(fa_status s)
{
    switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_UNKNOWN_STATUS";
}

fa_status fa_device_status(void *stream)
{
    uint32_t v = 0, vb = 0, vd = 0, vh = 0;
    if (fa::read_and_clear_status(static_cast<cudaStream_t>(stream), &v) != cudaSuccess ||
        fa::read_and_clear_status_bwd(&vb) != cudaSuccess || fa::read_and_clear_status_onetile(&vd) != cudaSuccess ||
        fa::read_and_clear_status_halves(&vh) != cudaSuccess)
        return FA_ERR_CUDA;
    v |= vb | vd | vh;
    if (v) {
        g_last_detail = v;
        if (v & fa::kStatusTimeout) return FA_ERR_TIMEOUT;
    }
    return FA_OK;
}

uint32_t fa_last_error_detail(void) { return g_last_detail; }

}  // extern "C"
