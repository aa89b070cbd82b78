// host_pipeline.cpp -- fa_fwd_host: the attention forward for q, k, v, o and lse held in
// host memory, with the host<->device copies overlapped with the kernel.
//
// The problem is cut along the flat (batch, KV head) axis into `chunks` runs.  KV heads
// [h0, h1) of one batch touch one contiguous range of k and v and, because consecutive query
// heads share a KV head, one contiguous range of q, o and lse; a run that crosses a batch
// boundary is split there.  Three streams per device carry the pipeline: chunk c's
// host->device copies, its kernels (the fa_fwd path on the sub-problem B = 1,
// Hq = group * (h1 - h0), Hkv = h1 - h0), then its device->host copies.  The two copy
// directions and the SMs thus work on three different chunks at once.  The pipeline starts
// after the work already enqueued on the caller's stream, and the caller's stream waits for
// the last copy back.  Streams and events are created on the first call for a device and
// reused; the device buffers are the caller's.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;
constexpr int kAutoChunks = 4;

struct Pipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, in[kMaxChunks] = {}, done[kMaxChunks] = {}, out = nullptr;
    std::mutex mu;
};
Pipe g_pipes[kMaxDevices];

bool init_pipe(Pipe &p)
{
    if (p.ready) return true;
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ev) != cudaSuccess || cudaEventCreateWithFlags(&p.out, ev) != cudaSuccess)
        return false;
    for (int i = 0; i < kMaxChunks; ++i)
        if (cudaEventCreateWithFlags(&p.in[i], ev) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.done[i], ev) != cudaSuccess)
            return false;
    p.ready = true;
    return true;
}

struct Range {
    const void *p;
    size_t n;
};

bool disjoint(Range a, Range b)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return x + a.n <= y || y + b.n <= x;
}

// Calls fn(b, h0, nkv) for every piece of KV heads [g0, g1) of the flat (B * Hkv) axis that
// lies inside one batch b, as heads [h0, h0 + nkv) of that batch.
template <class F> int for_each_run(long long g0, long long g1, int Hkv, F fn)
{
    for (long long a = g0; a < g1;) {
        const long long b = a / Hkv, h0 = a % Hkv;
        const long long h1 = (g1 - b * Hkv < Hkv) ? g1 - b * Hkv : Hkv;
        const int st = fn(b, h0, h1 - h0);
        if (st != FA_OK) return st;
        a = b * Hkv + h1;
    }
    return FA_OK;
}

int ok(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH; }

} // namespace

extern "C" int fa_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h, void *q_d,
                           void *k_d, void *v_d, void *o_d, float *lse_d, int B, int Hq, int Hkv, int Sq, int Sk,
                           int D, int causal, float scale, int dtype, int chunks, fa_stream_t stream)
{
    // ---- argument checks: no CUDA call before these pass
    if (dtype != 0 && dtype != 1) return FA_ERR_ARG;
    if (chunks < 0 || chunks > kMaxChunks) return FA_ERR_ARG;
    int st = fa::check_fwd_args(q_d, k_d, v_d, o_d, lse_d, B, Hq, Hkv, Sq, Sk, D, causal, scale, 0);
    if (st != FA_OK || B == 0 || Sq == 0) return st;
    if (!q_h || !k_h || !v_h || !o_h || !lse_h) return FA_ERR_NULL_PTR;
    const long long group = Hq / Hkv;
    const size_t qrow = (size_t)Sq * D * 2, krow = (size_t)Sk * D * 2, lrow = (size_t)Sq * 4;   // bytes per head
    const size_t nq = (size_t)B * Hq * qrow, nk = (size_t)B * Hkv * krow, nl = (size_t)B * Hq * lrow;
    {
        // Device buffers are written by the copies, host outputs by the copies back: each of
        // them must be disjoint from every other range (host inputs may share memory).
        const Range r[10] = {{q_d, nq}, {k_d, nk}, {v_d, nk}, {o_d, nq}, {lse_d, nl},
                             {o_h, nq}, {lse_h, nl}, {q_h, nq}, {k_h, nk}, {v_h, nk}};
        for (int i = 0; i < 7; ++i)
            for (int j = i + 1; j < 10; ++j)
                if (!disjoint(r[i], r[j])) return FA_ERR_ALIAS;
    }
    if ((st = fa::check_device()) != FA_OK) return st;

    const long long groups = (long long)B * Hkv;
    long long nc = chunks ? chunks : kAutoChunks;
    if (nc > groups) nc = groups;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
    Pipe &pp = g_pipes[dev];
    std::lock_guard<std::mutex> lock(pp.mu);   // one enqueue at a time per device: the events are shared
    if (!init_pipe(pp)) return FA_ERR_NO_DEVICE;
    cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);

    if ((st = ok(cudaEventRecord(pp.start, user))) != FA_OK) return st;
    for (cudaStream_t s : {pp.h2d, pp.comp, pp.d2h})
        if ((st = ok(cudaStreamWaitEvent(s, pp.start, 0))) != FA_OK) return st;

    // After a failure mid-way the caller's stream still waits for whatever was enqueued.
    auto drain = [&](int e) {
        for (cudaStream_t s : {pp.h2d, pp.comp, pp.d2h})
            if (cudaEventRecord(pp.out, s) == cudaSuccess) cudaStreamWaitEvent(user, pp.out, 0);
        return e;
    };
    auto cp = [](void *dst, const void *src, size_t off, size_t n, cudaMemcpyKind kind, cudaStream_t s) {
        return ok(cudaMemcpyAsync(static_cast<char *>(dst) + off, static_cast<const char *>(src) + off, n, kind, s));
    };
    for (long long c = 0; c < nc; ++c) {
        const long long g0 = groups * c / nc, g1 = groups * (c + 1) / nc;
        // inputs of chunk c
        st = for_each_run(g0, g1, Hkv, [&](long long b, long long h0, long long nkv) {
            const size_t qo = (size_t)(b * Hq + h0 * group) * qrow, ko = (size_t)(b * Hkv + h0) * krow;
            int e = cp(q_d, q_h, qo, (size_t)(nkv * group) * qrow, cudaMemcpyHostToDevice, pp.h2d);
            if (e == FA_OK) e = cp(k_d, k_h, ko, (size_t)nkv * krow, cudaMemcpyHostToDevice, pp.h2d);
            if (e == FA_OK) e = cp(v_d, v_h, ko, (size_t)nkv * krow, cudaMemcpyHostToDevice, pp.h2d);
            return e;
        });
        if (st != FA_OK) return drain(st);
        if ((st = ok(cudaEventRecord(pp.in[c], pp.h2d))) != FA_OK) return drain(st);
        if ((st = ok(cudaStreamWaitEvent(pp.comp, pp.in[c], 0))) != FA_OK) return drain(st);
        // attention on chunk c
        st = for_each_run(g0, g1, Hkv, [&](long long b, long long h0, long long nkv) {
            const size_t qo = (size_t)(b * Hq + h0 * group) * qrow, ko = (size_t)(b * Hkv + h0) * krow;
            const size_t lo = (size_t)(b * Hq + h0 * group) * lrow;
            char *qd = static_cast<char *>(q_d) + qo, *od = static_cast<char *>(o_d) + qo;
            char *kd = static_cast<char *>(k_d) + ko, *vd = static_cast<char *>(v_d) + ko;
            float *ld = reinterpret_cast<float *>(reinterpret_cast<char *>(lse_d) + lo);
            auto s = reinterpret_cast<fa_stream_t>(pp.comp);
            return fa_fwd_select(qd, kd, vd, od, ld, 1, (int)(nkv * group), (int)nkv, Sq, Sk, D, causal, scale, s,
                                 dtype, 0);
        });
        if (st != FA_OK) return drain(st);
        if ((st = ok(cudaEventRecord(pp.done[c], pp.comp))) != FA_OK) return drain(st);
        if ((st = ok(cudaStreamWaitEvent(pp.d2h, pp.done[c], 0))) != FA_OK) return drain(st);
        // outputs of chunk c
        st = for_each_run(g0, g1, Hkv, [&](long long b, long long h0, long long nkv) {
            const size_t qo = (size_t)(b * Hq + h0 * group) * qrow, lo = (size_t)(b * Hq + h0 * group) * lrow;
            int e = cp(o_h, o_d, qo, (size_t)(nkv * group) * qrow, cudaMemcpyDeviceToHost, pp.d2h);
            if (e == FA_OK) e = cp(lse_h, lse_d, lo, (size_t)(nkv * group) * lrow, cudaMemcpyDeviceToHost, pp.d2h);
            return e;
        });
        if (st != FA_OK) return drain(st);
    }
    // copies back run in order on one stream: the last one ends the call's work
    if ((st = ok(cudaEventRecord(pp.out, pp.d2h))) != FA_OK) return drain(st);
    return ok(cudaStreamWaitEvent(user, pp.out, 0));
}
