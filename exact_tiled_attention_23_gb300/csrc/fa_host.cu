// fa_host.cu -- the forward pass over inputs and outputs in host memory, with
// the host<->device copies pipelined against the computation.
//
// On a Grace-Blackwell node the host<->device copy of a long-context problem
// takes longer than the attention itself, so copying everything in, computing
// and copying out one after another leaves the GPU idle most of the time.
// This entry point splits the (batch, head) slices into groups and runs the
// copies and the computation side by side: group c+1 is copied in while group
// c is computed and group c-1 is copied out.  Consecutive groups are computed
// on two alternating streams, so that one group's kernel can fill the SMs
// that the other's longest work items (the last query tiles under a causal
// mask) leave idle.  The caller provides the device buffers, so the library
// still allocates no device memory; it keeps four streams and a ring of
// events per device.  Calls on one device from several host threads take
// turns: each enqueues its whole sequence under that device's lock, so no
// call's event records fall between another's records and waits.
#include "fa.h"
#include "fa_internal.h"

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr int kEventRing = 64;   // events are reused round-robin (see below)

struct CopyStreams {
    cudaStream_t h2d = nullptr;
    cudaStream_t d2h = nullptr;
    cudaStream_t comp[2] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t done = nullptr;
    cudaEvent_t comp_end[2] = {};
    cudaEvent_t in_ready[kEventRing] = {};
    cudaEvent_t out_ready[kEventRing] = {};
    bool ready = false;
    std::mutex enqueue;   // held by a call from its first record to its last wait
};

std::mutex g_mu;
CopyStreams g_copy[kMaxDevices];

// The current device's copy streams and events, created on first use.
fa_status copy_streams(CopyStreams **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    CopyStreams &cs = g_copy[dev];
    if (!cs.ready) {
        const unsigned flags = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&cs.comp[0], cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&cs.comp[1], cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&cs.start, flags) == cudaSuccess &&
                  cudaEventCreateWithFlags(&cs.done, flags) == cudaSuccess &&
                  cudaEventCreateWithFlags(&cs.comp_end[0], flags) == cudaSuccess &&
                  cudaEventCreateWithFlags(&cs.comp_end[1], flags) == cudaSuccess;
        for (int i = 0; ok && i < kEventRing; ++i)
            ok = cudaEventCreateWithFlags(&cs.in_ready[i], flags) == cudaSuccess &&
                 cudaEventCreateWithFlags(&cs.out_ready[i], flags) == cudaSuccess;
        if (!ok) return FA_ERR_CUDA;
        cs.ready = true;
    }
    *out = &cs;
    return FA_OK;
}

bool tc_head_dim(int D) { return (D > 0 && D <= 128 && D % 8 == 0) || D == 256; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int current_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    return sms;
}

}  // namespace

extern "C" int fa_fwd_from_host_auto_groups(int B, int H, int N, int D)
{
    (void)D;
    if (B <= 0 || H <= 0 || N <= 0) return 1;
    // Up to 8 groups of at least one wave of 256-row work items each.  The
    // copies set the pace (page-locked host memory moves at about 200 GB/s
    // per direction on a GB300 node), and what is not hidden is the first
    // group's copy-in and the last group's computation and copy-out: more
    // groups shorten those, while fewer, larger groups keep the kernels
    // efficient.  On B=1 H=32 N=16384 D=128 causal, 8 to 11 groups gave
    // the shortest time (2.42 ms, against 4.15 ms for one group).
    const int64_t items = (int64_t)B * H * (((int64_t)N + 255) / 256);
    int64_t g = items / (int64_t)current_sms();
    if (g > 8) g = 8;
    const int64_t bh = (int64_t)B * H;
    if (g > bh) g = bh;
    return g < 1 ? 1 : (int)g;
}

extern "C" fa_status fa_fwd_from_host(const void *Q_host, const void *K_host, const void *V_host,
                                      void *O_host, float *LSE_host, void *Q_dev, void *K_dev, void *V_dev,
                                      void *O_dev, float *LSE_dev, int B, int H, int N, int D, int causal,
                                      float scale, const int32_t *kv_len, int f16, int groups, void *stream)
{
    // ---- checks: all before any CUDA call --------------------------------
    if (B < 0 || H < 0 || N < 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (groups < 0 || groups > FA_MAX_HOST_GROUPS) return FA_ERR_INVALID_ARG;
    if ((int64_t)B * H * N == 0) return FA_OK;
    if (!Q_host || !K_host || !V_host || !O_host || !Q_dev || !K_dev || !V_dev || !O_dev)
        return FA_ERR_INVALID_ARG;
    if (LSE_host && !LSE_dev) return FA_ERR_INVALID_ARG;
    if (!tc_head_dim(D)) return FA_ERR_UNSUPPORTED;
    if (!aligned(Q_dev, 16) || !aligned(K_dev, 16) || !aligned(V_dev, 16) || !aligned(O_dev, 16))
        return FA_ERR_INVALID_ARG;
    if ((LSE_dev && !aligned(LSE_dev, 4)) || (kv_len && !aligned(kv_len, 4))) return FA_ERR_INVALID_ARG;
    if ((int64_t)B * H * N > ((int64_t)1 << 40)) return FA_ERR_INVALID_ARG;

    CopyStreams *cs = nullptr;
    fa_status st = copy_streams(&cs);
    if (st != FA_OK) return st;
    if (groups == 0) groups = fa_fwd_from_host_auto_groups(B, H, N, D);
    // Groups never span two batches, so each one is a call with B = 1 and
    // its batch's key length.  Split every batch's H heads into gpb groups.
    int gpb = (groups + B - 1) / B;
    if (gpb > H) gpb = H;
    const int hc_max = (H + gpb - 1) / gpb;

    const cudaStream_t user = static_cast<cudaStream_t>(stream);
    const size_t es = 2;                                   // bf16 / fp16 element size
    const size_t head_elems = (size_t)N * (size_t)D;
    auto h2d = [&](void *dst, const void *src, size_t off, size_t n) {
        return cudaMemcpyAsync(static_cast<char *>(dst) + off, static_cast<const char *>(src) + off, n,
                               cudaMemcpyHostToDevice, cs->h2d);
    };
    auto d2h = [&](void *dst, const void *src, size_t off, size_t n) {
        return cudaMemcpyAsync(static_cast<char *>(dst) + off, static_cast<const char *>(src) + off, n,
                               cudaMemcpyDeviceToHost, cs->d2h);
    };
#define FA_TRY(x)                                  \
    do {                                           \
        if ((x) != cudaSuccess) return FA_ERR_CUDA; \
    } while (0)

    // Every group runs the kernel fa_fwd would run for the whole problem, so
    // that the result is fa_fwd's exactly (the kernels agree only to rounding).
    const int tiles = fa::fwd16_tiles(B, H, N, D);

    std::lock_guard<std::mutex> turn(cs->enqueue);
    // Events are reused round-robin.  That is safe because each record is
    // followed, in host order, by the wait that consumes it: a wait takes
    // the work of the most recent record at the time it is enqueued.
    auto enqueue_groups = [&]() -> fa_status {
        // Earlier work on the caller's stream may still use the buffers.
        FA_TRY(cudaEventRecord(cs->start, user));
        FA_TRY(cudaStreamWaitEvent(cs->h2d, cs->start, 0));
        FA_TRY(cudaStreamWaitEvent(cs->d2h, cs->start, 0));
        FA_TRY(cudaStreamWaitEvent(cs->comp[0], cs->start, 0));
        FA_TRY(cudaStreamWaitEvent(cs->comp[1], cs->start, 0));
        int c = 0;
        for (int b = 0; b < B; ++b) {
            for (int h0 = 0; h0 < H; h0 += hc_max, ++c) {
                const int hc = (H - h0) < hc_max ? (H - h0) : hc_max;
                const size_t first = (size_t)b * H + (size_t)h0;        // first (b, h) slice of the group
                const size_t off = first * head_elems * es, bytes = (size_t)hc * head_elems * es;
                const size_t loff = first * (size_t)N * sizeof(float), lbytes = (size_t)hc * N * sizeof(float);
                cudaEvent_t in = cs->in_ready[c % kEventRing], outv = cs->out_ready[c % kEventRing];
                FA_TRY(h2d(Q_dev, Q_host, off, bytes));
                FA_TRY(h2d(K_dev, K_host, off, bytes));
                FA_TRY(h2d(V_dev, V_host, off, bytes));
                FA_TRY(cudaEventRecord(in, cs->h2d));
                cudaStream_t comp = cs->comp[c & 1];
                FA_TRY(cudaStreamWaitEvent(comp, in, 0));
                char *qd = static_cast<char *>(Q_dev) + off;
                char *kd = static_cast<char *>(K_dev) + off;
                char *vd = static_cast<char *>(V_dev) + off;
                char *od = static_cast<char *>(O_dev) + off;
                float *ld = LSE_dev ? LSE_dev + first * (size_t)N : nullptr;
                const int32_t *kl = kv_len ? kv_len + b : nullptr;
                const fa_status gs =
                    fa::fwd16_with_tiles(qd, kd, vd, od, ld, 1, hc, N, D, causal, scale, kl, f16 != 0, tiles, comp);
                if (gs != FA_OK) return gs;
                FA_TRY(cudaEventRecord(outv, comp));
                FA_TRY(cudaStreamWaitEvent(cs->d2h, outv, 0));
                FA_TRY(d2h(O_host, O_dev, off, bytes));
                if (LSE_host) FA_TRY(d2h(LSE_host, LSE_dev, loff, lbytes));
            }
        }
        return FA_OK;
    };
    st = enqueue_groups();
    // Whether or not every group was enqueued, the caller's stream goes on
    // only after everything this call put on the library's streams: the
    // copy-out stream waits for the end of both compute streams (on success
    // it has already waited for every group's computation), and the caller's
    // stream waits for the copy-out stream.  So a caller that frees or reuses
    // the buffers after an error does not race with work still in flight.
    const bool fenced = cudaEventRecord(cs->comp_end[0], cs->comp[0]) == cudaSuccess &&
                        cudaEventRecord(cs->comp_end[1], cs->comp[1]) == cudaSuccess &&
                        cudaStreamWaitEvent(cs->d2h, cs->comp_end[0], 0) == cudaSuccess &&
                        cudaStreamWaitEvent(cs->d2h, cs->comp_end[1], 0) == cudaSuccess &&
                        cudaEventRecord(cs->done, cs->d2h) == cudaSuccess &&
                        cudaStreamWaitEvent(user, cs->done, 0) == cudaSuccess;
    if (st != FA_OK) return st;
#undef FA_TRY
    return fenced ? FA_OK : FA_ERR_CUDA;
}
