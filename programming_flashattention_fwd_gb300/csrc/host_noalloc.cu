// host_noalloc.cu -- fa_fwd_host_noalloc: fa_fwd_host for callers that cannot allocate device
// memory, with the staging area in a fixed array of device memory that belongs to the library.
//
// fa_fwd_host copies q, k, v from host memory into five device buffers (q, k, v in; o, lse
// out) and back.  Here those five buffers are slices of g_staging, each starting on a 256-byte
// boundary.  In host code the name g_staging stands for a host-side shadow of the array, not
// for its device address, so the address is looked up once per device with that device
// current (cudaGetSymbolAddress) and cached.  Nothing here allocates.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

// The staging area.  Each GPU on which this image is loaded holds it until the process exits.
static __device__ __align__(256) unsigned char g_staging[FA_HOST_NOALLOC_MAX_BYTES];

namespace {

constexpr size_t kCap = FA_HOST_NOALLOC_MAX_BYTES;
constexpr size_t kSliceAlign = 256;
constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;   // fa_fwd_host's limit, checked here too so that no CUDA call precedes it

std::mutex g_mu;
void *g_addr[kMaxDevices];       // device address of g_staging per device, once looked up

size_t round_up(size_t n) { return (n + kSliceAlign - 1) / kSliceAlign * kSliceAlign; }

bool disjoint(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x + na <= y || y + nb <= x;
}

// Device address of the staging area on the current device `dev`.  The first call per device
// does the look-up (which also loads this file's device image there, if it is not loaded yet).
int staging_on(int dev, unsigned char **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_staging) != cudaSuccess || !p) {
            cudaGetLastError();   // do not leave the error for the caller's next launch check
            return FA_ERR_NO_DEVICE;
        }
        g_addr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_addr[dev]);
    return FA_OK;
}

} // namespace

extern "C" int fa_fwd_host_noalloc(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                                   int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                                   int dtype, int chunks, fa_stream_t stream)
{
    // ---- argument checks: no CUDA call before these pass
    if (dtype != 0 && dtype != 1) return FA_ERR_ARG;
    if (chunks < 0 || chunks > kMaxChunks) return FA_ERR_ARG;
    // fa_fwd's checks of everything but the pointers: with all five pointers NULL they return
    // FA_ERR_NULL_PTR exactly when the sizes, heads, D, causal and scale are valid and the
    // problem is not empty (an empty problem is FA_OK, any other code is the argument error).
    int st = fa::check_fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, B, Hq, Hkv, Sq, Sk, D, causal, scale,
                                0);
    if (st != FA_ERR_NULL_PTR) return st;
    if (!q_h || !k_h || !v_h || !o_h || !lse_h) return FA_ERR_NULL_PTR;

    // Staging bytes.  First the unrounded total in double, where the products cannot overflow:
    // it is a lower bound, so above the cap the problem is too large.  Below it every size fits
    // in size_t, and the exact total with each slice rounded up decides.
    const double need = 2.0 * ((double)B * Hq * Sq * D * 2) + 2.0 * ((double)B * Hkv * Sk * D * 2) +
                        (double)B * Hq * Sq * 4;
    if (need > (double)kCap) return FA_ERR_TOO_LARGE;
    const size_t nq = (size_t)B * Hq * Sq * D * 2, nk = (size_t)B * Hkv * Sk * D * 2, nl = (size_t)B * Hq * Sq * 4;
    const size_t off_q = 0, off_k = off_q + round_up(nq), off_v = off_k + round_up(nk),
                 off_o = off_v + round_up(nk), off_l = off_o + round_up(nq);
    if (off_l + round_up(nl) > kCap) return FA_ERR_TOO_LARGE;

    // The host outputs are written by the copies back: disjoint from each other and the inputs.
    if (!disjoint(o_h, nq, lse_h, nl) || !disjoint(o_h, nq, q_h, nq) || !disjoint(o_h, nq, k_h, nk) ||
        !disjoint(o_h, nq, v_h, nk) || !disjoint(lse_h, nl, q_h, nq) || !disjoint(lse_h, nl, k_h, nk) ||
        !disjoint(lse_h, nl, v_h, nk))
        return FA_ERR_ALIAS;

    // ---- device set-up (once per device), then fa_fwd_host on the staging slices
    if ((st = fa::check_device()) != FA_OK) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
    unsigned char *base = nullptr;
    if ((st = staging_on(dev, &base)) != FA_OK) return st;
    return fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, base + off_q, base + off_k, base + off_v, base + off_o,
                       reinterpret_cast<float *>(base + off_l), B, Hq, Hkv, Sq, Sk, D, causal, scale, dtype, chunks,
                       stream);
}
