// lla_fwd_host: the forward on inputs and outputs in host memory.
//
// The (batch, head) pairs are independent and each pair's rows are one
// contiguous span of every tensor, so the call cuts them into groups (half
// size at both ends) and pipelines three stages over two device slots: the copy of group j+1's
// inputs (host -> device), the forward of group j, and the copy of group
// j-1's output (device -> host) run at the same time on a copy-in stream,
// the caller's stream and a copy-out stream.  The two copy directions use
// separate copy engines, so the transfer time approaches the larger of the
// two directions instead of their sum.
//
// The two internal streams and the ordering events are created once per
// device on the first call (with that device current) and kept until exit
// (a creation that fails is undone and tried again by the next call); a
// mutex per device serialises the enqueueing of concurrent calls.  The
// call is ordered on the caller's stream: work already on it completes
// before any copy starts, and the caller's stream waits for the last output
// copy.  Host buffers should be pinned (page-locked) for the copies to run
// asynchronously; pageable buffers still give correct results.
#include <mutex>

#include "lla_common.cuh"

namespace {

constexpr int kMaxDevices = 64;

struct Pipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr;
    cudaEvent_t in_ready[2] = {nullptr, nullptr}, comp_done[2] = {nullptr, nullptr},
                out_done[2] = {nullptr, nullptr};
    bool ready = false;
    std::mutex mu;  // guards the set-up and serialises the enqueueing
};

Pipe g_pipe[kMaxDevices];

void destroy_pipe(Pipe *p)
{
    cudaEvent_t *evs[] = {&p->entry, &p->done, &p->in_ready[0], &p->in_ready[1], &p->comp_done[0],
                          &p->comp_done[1], &p->out_done[0], &p->out_done[1]};
    for (cudaEvent_t *ev : evs)
        if (*ev) {
            cudaEventDestroy(*ev);
            *ev = nullptr;
        }
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    p->h2d = p->d2h = nullptr;
}

// The current device's pipe with p->mu held (streams and events created on
// first use); nullptr if they cannot be created.
Pipe *lock_pipe_for_current_device(std::unique_lock<std::mutex> *lock)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    Pipe *p = &g_pipe[dev];
    *lock = std::unique_lock<std::mutex>(p->mu);
    if (!p->ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&p->entry, &p->done, &p->in_ready[0], &p->in_ready[1], &p->comp_done[0],
                              &p->comp_done[1], &p->out_done[0], &p->out_done[1]};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            destroy_pipe(p);
            cudaGetLastError();
            return nullptr;
        }
        p->ready = true;
    }
    return p;
}

size_t dt_size(lla_dtype dt) { return dt == LLA_BF16 ? 2 : 4; }

int resolve_group(long long BH, int group)
{
    if (group > 0) return (int)(group < BH ? group : BH);
    const long long g = (BH + 7) / 8;
    return (int)(g > 0 ? g : 1);
}

struct Spans {  // bytes of one (batch, head) pair in each tensor
    size_t q, k, v, g, lam, out;
};

Spans spans(int T, int dk, int dv, lla_dtype in_dt, lla_dtype out_dt)
{
    const int L = lla_num_levels(T);
    Spans s;
    s.q = (size_t)T * dk * dt_size(in_dt);
    s.k = s.q;
    s.v = (size_t)T * dv * dt_size(in_dt);
    s.g = (size_t)T * 4;
    s.lam = (size_t)T * L * 4;
    s.out = (size_t)T * dv * dt_size(out_dt);
    return s;
}

size_t slot_bytes(const Spans &s, int group)
{
    using lla::align_up;
    return align_up(s.q * group, 256) + align_up(s.k * group, 256) + align_up(s.v * group, 256) +
           align_up(s.g * group, 256) + align_up(s.lam * group, 256) + align_up(s.out * group, 256);
}

}  // namespace

extern "C" {

size_t lla_fwd_host_workspace_bytes(int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt,
                                    lla_dtype out_dt, int group)
{
    if (B < 0 || H < 0 || T < 0 || (long long)B * H * T == 0) return 0;
    if (lla_fwd_workspace_bytes(1, 1, T, dk, dv, chunk, in_dt) == 0) return 0;  // unsupported shape
    const int G = resolve_group((long long)B * H, group);
    const Spans s = spans(T, dk, dv, in_dt, out_dt);
    return 2 * slot_bytes(s, G) + lla::align_up(lla_fwd_workspace_bytes(1, G, T, dk, dv, chunk, in_dt), 256);
}

lla_status lla_fwd_host(const void *q, const void *k, const void *v, const float *g, const float *lambda,
                        void *out, int B, int H, int T, int dk, int dv, int chunk, lla_dtype in_dt,
                        lla_dtype out_dt, int group, void *workspace, size_t workspace_bytes,
                        int32_t *device_error, void *stream)
{
    // shapes, dtypes and the empty case exactly as lla_fwd decides them
    if (B < 0 || H < 0 || T < 0 || group < 0) return LLA_ERR_INVALID_ARGUMENT;
    if (out_dt != LLA_F32 && out_dt != LLA_BF16) return LLA_ERR_INVALID_ARGUMENT;
    if ((long long)B * H * T == 0)
        return lla_fwd(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt, out_dt, nullptr, 0,
                       device_error, stream);
    if (lla_fwd_workspace_bytes(1, 1, T, dk, dv, chunk, in_dt) == 0) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (in_dt == LLA_F32 && out_dt != LLA_F32) return LLA_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k || !v || !g || !lambda || !out) return LLA_ERR_INVALID_ARGUMENT;
    const size_t need = lla_fwd_host_workspace_bytes(B, H, T, dk, dv, chunk, in_dt, out_dt, group);
    if (workspace_bytes < need) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0) return LLA_ERR_INVALID_ARGUMENT;
    std::unique_lock<std::mutex> lock;
    Pipe *p = lock_pipe_for_current_device(&lock);
    if (!p) return LLA_ERR_CUDA;
    const long long BH = (long long)B * H;
    const int G = resolve_group(BH, group);
    const Spans s = spans(T, dk, dv, in_dt, out_dt);
    const size_t sb = slot_bytes(s, G);
    char *ws = (char *)workspace;
    void *fws = ws + 2 * sb;
    const size_t fws_bytes = workspace_bytes - 2 * sb;
    cudaStream_t cs = (cudaStream_t)stream;
#define LLA_TRY(x)                                       \
    do {                                                 \
        if ((x) != cudaSuccess) return LLA_ERR_CUDA;     \
    } while (0)
    LLA_TRY(cudaEventRecord(p->entry, cs));
    LLA_TRY(cudaStreamWaitEvent(p->h2d, p->entry, 0));
    LLA_TRY(cudaStreamWaitEvent(p->d2h, p->entry, 0));
    // G pairs per group in the middle, half as many in the first and the last
    // group: the pipeline's fill (the first input copy, alone) and drain (the
    // last output copy, alone) are the transfer time it cannot overlap
    const int Gh = G > 1 ? G / 2 : 1;
    long long b0 = 0;
    for (long long j = 0; b0 < BH; j++) {
        const int sl = (int)(j & 1);
        const long long rem = BH - b0;
        long long nn;
        if (j == 0) nn = rem < Gh ? rem : Gh;
        else if (rem <= Gh) nn = rem;             // the last group
        else if (rem <= G + Gh) nn = rem - Gh;    // leaves a small last group
        else nn = G;
        const int n = (int)nn;
        char *base = ws + sl * sb;
        char *dq = base;
        char *dk_ = dq + lla::align_up(s.q * G, 256);
        char *dv_ = dk_ + lla::align_up(s.k * G, 256);
        char *dg = dv_ + lla::align_up(s.v * G, 256);
        char *dl = dg + lla::align_up(s.g * G, 256);
        char *dout = dl + lla::align_up(s.lam * G, 256);
        // inputs of group j into slot sl once group j-2 has finished with it
        LLA_TRY(cudaStreamWaitEvent(p->h2d, p->comp_done[sl], 0));
        LLA_TRY(cudaMemcpyAsync(dq, (const char *)q + b0 * s.q, n * s.q, cudaMemcpyHostToDevice, p->h2d));
        LLA_TRY(cudaMemcpyAsync(dk_, (const char *)k + b0 * s.k, n * s.k, cudaMemcpyHostToDevice, p->h2d));
        LLA_TRY(cudaMemcpyAsync(dv_, (const char *)v + b0 * s.v, n * s.v, cudaMemcpyHostToDevice, p->h2d));
        LLA_TRY(cudaMemcpyAsync(dg, (const char *)g + b0 * s.g, n * s.g, cudaMemcpyHostToDevice, p->h2d));
        LLA_TRY(cudaMemcpyAsync(dl, (const char *)lambda + b0 * s.lam, n * s.lam, cudaMemcpyHostToDevice,
                                p->h2d));
        LLA_TRY(cudaEventRecord(p->in_ready[sl], p->h2d));
        // the forward of group j, after its inputs and after group j-2's output copy
        LLA_TRY(cudaStreamWaitEvent(cs, p->in_ready[sl], 0));
        LLA_TRY(cudaStreamWaitEvent(cs, p->out_done[sl], 0));
        lla_status st = lla_fwd(dq, dk_, dv_, (const float *)dg, (const float *)dl, dout, 1, n, T, dk, dv,
                                chunk, in_dt, out_dt, fws, fws_bytes, device_error, stream);
        if (st != LLA_OK) return st;
        LLA_TRY(cudaEventRecord(p->comp_done[sl], cs));
        // its output back to the host
        LLA_TRY(cudaStreamWaitEvent(p->d2h, p->comp_done[sl], 0));
        LLA_TRY(cudaMemcpyAsync((char *)out + b0 * s.out, dout, n * s.out, cudaMemcpyDeviceToHost, p->d2h));
        LLA_TRY(cudaEventRecord(p->out_done[sl], p->d2h));
        b0 += n;
    }
    LLA_TRY(cudaEventRecord(p->done, p->d2h));
    LLA_TRY(cudaStreamWaitEvent(cs, p->done, 0));
#undef LLA_TRY
    return LLA_OK;
}

}  // extern "C"
