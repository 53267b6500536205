/*
 * fa.h -- C ABI of the exact tiled attention forward pass for GB300 (sm_103a).
 *
 * The library computes, for every batch b and head h,
 *
 *     O   = softmax(scale * Q K^T + mask) V
 *     LSE = log-sum-exp of each row of (scale * Q K^T + mask), natural log
 *
 * block by block with the online-softmax running max m and running sum l,
 * rescaled by exp(m_old - m_new) whenever a key block raises the max, and
 * without ever writing the N x N score matrix to device memory
 * ("vectorized-flash-attention-kernel", Core algorithm and Key design
 * decisions 1-3; "FlashAttention" module F08, Paper).  The mask hides key j
 * from query i when j >= kv_len[b] (key padding), and, if `causal`, when
 * j > i ("kvRow > qRow -> -inf", Core algorithm step 2).
 *
 * Layout (all arguments): Q, K, V and O are contiguous row-major
 * [B, H, N, D] arrays; LSE is a contiguous [B, H, N] float array; kv_len is
 * an int32 array of B entries.  Every pointer is DEVICE memory owned by the
 * caller unless stated otherwise (fa_fwd_from_host takes host arrays); no
 * call allocates device memory or keeps a pointer after it returns.  The
 * library's own state is: device-side status words (see fa_device_status); a
 * cached driver entry point; the fixed scratch array of
 * fa_fwd_splitkv_noalloc (FA_NOALLOC_SCRATCH_BYTES of device memory, held from
 * the time the library's code is loaded on a device); and, per device that
 * calls fa_fwd_from_host, four streams and a set of events, created by the
 * first such call and kept for the life of the process.
 *
 * Calls are asynchronous: they validate their arguments on the host, enqueue
 * one kernel on `stream` (a cudaStream_t; NULL = the legacy default stream)
 * and return.  Results are ready when the stream reaches that point.  Input
 * and output buffers must not overlap.
 *
 * Numerical contract:
 *   - rows whose mask hides every key (kv_len[b] == 0) get O = +0.0 exactly
 *     and LSE = -inf, never NaN ("js-flash-attention-tiled-online-softmax-
 *     exactness", Root causes 2);
 *   - query rows at or past kv_len[b] are still computed over the keys
 *     j < kv_len[b] (padding hides keys, not queries);
 *   - kv_len entries outside [0, N] are clamped to that range on the device;
 *   - input range: the 16-bit paths keep each key block's weights p against a
 *     reference that moves only when a block's sum of p would pass 2^64
 *     (bf16) or 2^15 (fp16), so the fp32 output accumulator holds up to
 *     N * 2^64 * max|V|; O is finite for bf16 |V| < 2^32 (any N < 2^31) and
 *     for every fp16 V.  Q and K may take any finite values.
 */
#ifndef EXACT_TILED_ATTENTION_FA_H
#define EXACT_TILED_ATTENTION_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment, overflow */
    FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head dim, device)        */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed                   */
    FA_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up (fa_device_status) */
} fa_status;

/*
 * fa_fwd -- bf16 attention forward on the tensor cores (tcgen05, TMEM, TMA).
 *
 *   Q, K, V  const bf16 [B,H,N,D] device pointers, 16-byte aligned.
 *   O        bf16 [B,H,N,D] device pointer, 16-byte aligned; each element is
 *            the fp32 result rounded to nearest-even.
 *   LSE      float [B,H,N] device pointer, or NULL to skip it (the saved row
 *            statistic a recomputing backward needs: "vectorized-flash-
 *            attention-kernel", Key design decisions 4).
 *   B, H, N  batch, heads, sequence length; any value >= 0.  B*H*N == 0
 *            returns FA_OK without a launch.
 *   D        head dimension: a multiple of 8 from 8 to 128, or 256 (the
 *            pages run D = 16 in "vectorized-flash-attention-kernel",
 *            Evidence & signatures, and d = 32 in "js-flash-attention-tiled-
 *            online-softmax-exactness", Verification).  Other values give
 *            FA_ERR_UNSUPPORTED.  Below 128 the tensor cores run at D
 *            rounded up to 64 or 128 with zero-filled columns, which leave
 *            every score unchanged; only the D real columns of O are
 *            written.
 *   causal   nonzero: key j is hidden from query i when j > i.
 *   scale    softmax scale; NaN or <= 0 selects the default 1/sqrt(D)
 *            ("vectorized-flash-attention-kernel", Constructor options).
 *   kv_len   const int32 [B] device pointer of key lengths, or NULL (= N).
 *   stream   cudaStream_t to enqueue on.
 *
 * Three kernels serve this call.  One gives every CTA two 128-row query
 * tiles (D <= 128).  One gives it one tile (any D here): D = 256, and D <= 64
 * on grids whose one-tile CTAs (2 * B * H * ceil(N/256)) fit in one wave of
 * the GPU's SMs.  The third gives it one tile and splits each row's keys
 * between two softmax warpgroups, whose partial softmax states it merges at
 * the end (D <= 128): 64 < D <= 128 with N >= 8192 or on such small grids.
 * The environment variable FA_FWD_TILES = "1", "2" or "3", read on every
 * call, forces one of them (D = 256 always runs the one-tile kernel).  The
 * kernels agree to rounding, not bit for bit.
 *
 * Accumulation is fp32 (scores, running sums, O); P is rounded to bf16 for
 * the second product, and O is divided by the sum of those rounded weights
 * (the LSE uses the sum of the unrounded ones), so O is a convex combination
 * of V rows whatever the rounding.  Returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED from
 * host-side checks before anything is enqueued, FA_ERR_CUDA if the launch
 * fails.
 */
fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                 int B, int H, int N, int D, int causal, float scale,
                 const int32_t *kv_len, void *stream);

/*
 * fa_fwd_f16 -- fp16 attention forward on the tensor cores ("FlashAttention"
 * module F08, Exercises: the backward exercise's "fp16" variant of the same
 * tiles).  Same arguments, layout and limits as fa_fwd with IEEE half Q, K,
 * V and O (O rounded to nearest even); LSE stays fp32.  P is rounded to fp16
 * for the second product; the reference max is raised whenever a key
 * block's sum of p would pass 2^15, so P stays inside the fp16 range.
 */
fa_status fa_fwd_f16(const void *Q, const void *K, const void *V, void *O, float *LSE,
                     int B, int H, int N, int D, int causal, float scale,
                     const int32_t *kv_len, void *stream);

/*
 * fa_fwd_fp32 -- fp32 attention forward (fp32 multiply-add on the CUDA cores,
 * no TF32).  Same argument meaning as fa_fwd with float Q, K, V, O; any head
 * dimension 1 <= D <= 256; pointers need only float alignment.
 */
fa_status fa_fwd_fp32(const float *Q, const float *K, const float *V, float *O, float *LSE,
                      int B, int H, int N, int D, int causal, float scale,
                      const int32_t *kv_len, void *stream);

/* The forward kernel fa_fwd and fa_fwd_f16 run for these sizes on the
 * current device: 1 = one 128-row query tile per CTA, 2 = two tiles per CTA,
 * 3 = one tile with each row's keys split between two softmax warpgroups
 * (FA_FWD_TILES, when set, decides as it does for those calls).  0 for a head
 * dimension the tensor-core kernels do not take.  No device work. */
int fa_fwd_kernel_choice(int B, int H, int N, int D);

/*
 * Split-KV forward ("FlashAttention" module F08, Paper and Math: partial
 * softmax states merge associatively).  Same computation and arguments as
 * fa_fwd, for sequences too short to fill the GPU with query tiles: the key
 * blocks of every (batch, head, 256-query-row) item are divided into
 * `num_splits` contiguous ranges processed by separate CTAs.  Each range
 * writes its normalised fp32 partial output and partial LSE to `workspace`,
 * and a second kernel on the same stream merges them:
 *     m = max_s LSE_s,  w_s = exp(LSE_s - m),
 *     O = sum_s w_s O_s / sum_s w_s,  LSE = m + ln sum_s w_s.
 * Ranges that see no key have LSE_s = -inf and weight 0.
 *
 *   num_splits       1..FA_MAX_SPLITS, or 0 for fa_fwd_splitkv_auto_splits().
 *                    With 1 split (given or chosen) the single-pass kernel
 *                    of fa_fwd runs and the workspace is not touched.
 *   workspace        caller-owned device memory, 16-byte aligned, of at least
 *                    fa_fwd_splitkv_workspace_bytes(B,H,N,D,num_splits)
 *                    bytes; its contents on entry do not matter, it is fully
 *                    rewritten, and it must not be used by another call that
 *                    may run at the same time.
 * D is a multiple of 8 up to 128 (256 gives FA_ERR_UNSUPPORTED here).
 * Returns FA_ERR_INVALID_ARG for a missing, misaligned or too small
 * workspace or a split count out of range; otherwise as fa_fwd.
 */
#define FA_MAX_SPLITS 64

fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int B, int H, int N, int D, int causal, float scale,
                         const int32_t *kv_len, int num_splits, void *workspace,
                         size_t workspace_bytes, void *stream);

/* Bytes of workspace fa_fwd_splitkv needs: num_splits * B*H*N * (D + 1) * 4
 * (0 for invalid sizes); num_splits 0 means the automatic choice. */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits);

/* The split count fa_fwd_splitkv uses for num_splits = 0 on the current
 * device.  1 unless D <= 64, N >= 4096 and fa_fwd's grid (2 * B * H *
 * ceil(N/256) one-tile CTAs) leaves SMs idle: there, as many ranges as fill
 * one wave of CTAs (one per SM), at least two key blocks per range, at most
 * FA_MAX_SPLITS.  (Measured on GB300: elsewhere the split path is not faster
 * than fa_fwd.) */
int fa_fwd_splitkv_auto_splits(int B, int H, int N, int D);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a library service.
 *
 * Some callers cannot call cudaMalloc or any allocator: code inside a
 * framework's allocation-free region, a plugin that is only handed its input
 * and output buffers, or a real-time loop where an allocation could block.
 * This entry point takes no workspace.  It uses a fixed scratch array of
 * FA_NOALLOC_SCRATCH_BYTES bytes that the library keeps in device memory.
 * A device holds that array from the time the library's code is loaded on
 * it (with CUDA's lazy module loading, the first call of this entry point
 * there at the latest) until the process exits.  The call itself allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments are those of fa_fwd_splitkv without the workspace.  The caller
 * still passes the inputs and outputs.
 *
 * Limits and behaviour:
 *   - A problem whose fa_fwd_splitkv_workspace_bytes(B,H,N,D,num_splits)
 *     exceeds FA_NOALLOC_SCRATCH_BYTES is rejected with FA_ERR_UNSUPPORTED
 *     before anything is enqueued.  Fewer splits, or fa_fwd, are the
 *     alternatives.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and later calls on
 *     that device reuse it.  Make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset of a device this entry point must not be called on it
 *     again, because the array may then sit at another address.
 *   - All calls share the one array, and it keeps the last call's contents.
 *     Each call rewrites every part it reads, so nothing needs clearing.
 *   - Two calls whose kernels overlap on the GPU (different streams, or
 *     different host threads without ordering) race on the array and give
 *     wrong results.  Order them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)

fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                 int B, int H, int N, int D, int causal, float scale,
                                 const int32_t *kv_len, int num_splits, void *stream);

/*
 * fa_fwd_from_host -- fa_fwd (or fa_fwd_f16) over inputs and outputs in host
 * memory, with the host<->device copies overlapped with the computation.  The
 * paper has no counterpart: this is a library service for callers whose data
 * starts and ends on the host.
 *
 * The (batch, head) slices are split into `groups` groups, none spanning two
 * batches.  Group c is copied to the device on a library-owned copy stream,
 * computed on one of two library-owned compute streams (alternating, so that
 * consecutive groups' kernels can share the SMs) while group c+1 is copied
 * in, and copied back on a second copy stream.  On a
 * Grace-Blackwell node the copies of a long-context problem take longer than
 * the attention, so the overlap shortens the whole call.
 *
 *   Q_host, K_host, V_host  const [B,H,N,D] host arrays (bf16, or fp16 if f16
 *                           is nonzero).  Page-locked memory lets the copies
 *                           run asynchronously.
 *   O_host                  [B,H,N,D] host array for O.
 *   LSE_host                float [B,H,N] host array, or NULL to skip LSE.
 *   Q_dev, K_dev, V_dev, O_dev  caller-owned device buffers of the same
 *                           shape, 16-byte aligned.  The inputs are copied
 *                           into them, and O is computed there.
 *   LSE_dev                 float [B,H,N] device buffer; required when
 *                           LSE_host is given, else may be NULL.
 *   B,H,N,D, causal, scale, kv_len  as in fa_fwd (kv_len in device memory).
 *   groups                  1..FA_MAX_HOST_GROUPS, or 0 for
 *                           fa_fwd_from_host_auto_groups(B,H,N,D).
 *   stream                  the caller's stream.  The copies start after the
 *                           work already enqueued on it.  Work enqueued on it
 *                           afterwards starts only once O and LSE are back in
 *                           host memory.
 *
 * Returns as fa_fwd; all argument checks run before any CUDA call.  The first
 * call on a device creates that device's four streams and their events.
 * Calls on one device share them.  Calls from several host threads are safe:
 * each enqueues its whole sequence of copies, launches and event records
 * under a per-device lock, so the calls run one after another on the
 * library's streams.  If a CUDA call fails partway, the caller's stream
 * still waits for everything the call had enqueued before the failure, so
 * the buffers may be freed or reused once that stream reaches this point.
 */
#define FA_MAX_HOST_GROUPS 1024

fa_status fa_fwd_from_host(const void *Q_host, const void *K_host, const void *V_host, void *O_host,
                           float *LSE_host, void *Q_dev, void *K_dev, void *V_dev, void *O_dev,
                           float *LSE_dev, int B, int H, int N, int D, int causal, float scale,
                           const int32_t *kv_len, int f16, int groups, void *stream);

/* The group count fa_fwd_from_host uses for groups = 0 on the current
 * device: min(B*H, 8, 256-row work items / SMs), at least 1.  (Groups never
 * span batches, so a call may run more groups than asked for: at least B.) */
int fa_fwd_from_host_auto_groups(int B, int H, int N, int D);

/*
 * fa_bwd -- backward pass of fa_fwd by recomputation ("FlashAttention"
 * module F08, Math: backward via recomputation and the identity
 * rowsum(dP*P) = rowsum(dO*O); "vectorized-flash-attention-kernel", Key
 * design decisions 4: the saved row statistics rebuild P).  Computes the
 * gradients of sum(O * dO) for O = fa_fwd(Q, K, V, ...):
 *
 *     P = exp(scale*Q K^T + mask - LSE),  dV = P^T dO,  dP = dO V^T,
 *     Delta = rowsum(dO * O),  dS = P * (dP - Delta),
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 *   Q, K, V, O, dO  const bf16 [B,H,N,D]: the forward's inputs and output
 *                   and the upstream gradient; 16-byte aligned.
 *   LSE             const float [B,H,N]: the LSE fa_fwd returned.
 *   dQ, dK, dV      bf16 [B,H,N,D] outputs (fp32 accumulation, rounded to
 *                   nearest even); keys at or past kv_len get zero dK, dV.
 *   B,H,N,D, causal, scale, kv_len: as in the forward call; D a multiple
 *            of 8 up to 128 (zero-padded to 64 / 128 like the forward; 256
 *            gives FA_ERR_UNSUPPORTED).
 *   workspace       caller-owned device memory, 16-byte aligned, of at least
 *                   fa_bwd_workspace_bytes(B,H,N,D) bytes (an fp32 dQ
 *                   accumulator and Delta); fully rewritten by each call;
 *                   calls that may overlap need separate workspaces.
 * dQ is summed across key tiles by fp32 reduce-adds, so its last bits may
 * differ from run to run; dK and dV are deterministic.  Three kernels are
 * enqueued on `stream`.  Errors as fa_fwd, plus FA_ERR_INVALID_ARG for a
 * missing or too small workspace.
 */
fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                 int causal, float scale, const int32_t *kv_len, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * fa_bwd_f16 -- fa_bwd for the fp16 forward (fa_fwd_f16): IEEE half Q, K, V,
 * O, dO and dQ, dK, dV; LSE, the workspace and every accumulation stay fp32,
 * and P and dS are rounded to fp16 for the tensor-core products (P <= 1; dS
 * must stay inside the fp16 range, as in any fp16 training).  Same arguments,
 * limits and errors as fa_bwd.
 */
fa_status fa_bwd_f16(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                     int causal, float scale, const int32_t *kv_len, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Bytes of workspace fa_bwd needs: B*H*N*(D + 1)*4 (0 for invalid sizes). */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int D);

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(fa_status s);

/*
 * fa_device_status -- synchronise `stream`, then report and clear the
 * device-side status word.  Returns FA_ERR_TIMEOUT if a kernel of this
 * library gave up a bounded wait since the last call (its output is then
 * undefined), FA_ERR_CUDA if synchronising failed, FA_OK otherwise.
 *
 * Every wait of the tensor-core kernels on another part of the same CTA
 * gives up after a budget: 4 s by default, or the environment variable
 * FA_WAIT_LIMIT_MS (milliseconds, fractions allowed), read once per process.
 * A kernel that gives up still waits, with a budget of at least 1 s, for the
 * copies and MMAs it has in flight before it exits, so the CUDA context stays
 * usable.
 */
fa_status fa_device_status(void *stream);

/*
 * fa_last_error_detail -- the site code of the last device-side give-up that
 * fa_device_status saw (0 if none): a diagnostic for bug reports.
 */
uint32_t fa_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TILED_ATTENTION_FA_H */
