// fa_api.cpp -- the C ABI declared in include/fa.h: argument validation (before any
// CUDA call), device checks, TMA descriptor encoding and dispatch to the kernel.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"
#include "schedule.h"

namespace {

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn get_encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Per-device cache of "is this an sm_103 device": 0 unknown, 1 yes, 2 no.
constexpr int kMaxDevices = 64;
std::atomic<int> g_arch_ok[kMaxDevices];

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D view (D, S, B*H) of a dense [B, H, S, D] 16-bit tensor; 64 x rows x 1 boxes, 128B swizzle.
bool encode(EncodeTiledFn enc, CUtensorMap *m, const void *base, bool bf16, int D, int S, long long BH,
            int rows = fa::kBM)
{
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * (cuuint64_t)D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

} // namespace

namespace fa {

// Device checks shared by every entry point (current device must be sm_103).
int check_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
    int st = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (st == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_NO_DEVICE;
        st = (major == 10 && minor == 3) ? 1 : 2;
        g_arch_ok[dev].store(st, std::memory_order_relaxed);
    }
    return st == 1 ? FA_OK : FA_ERR_ARCH;
}

int check_fwd_args(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int D, int causal, float scale, int kernel)
{
    if (B < 0 || Sq < 0 || Sk < 0) return FA_ERR_BAD_DIM;
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return FA_ERR_HEADS;
    if (kernel < 0 || kernel > 3) return FA_ERR_ARG;
    if (kernel == 0) kernel = (D == 256) ? 2 : 1;
    if (kernel == 1 && D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
    if (kernel == 2 && D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED_D;
    if (kernel == 3 && D != 128) return FA_ERR_UNSUPPORTED_D;
    if (!std::isfinite(scale)) return FA_ERR_SCALE;
    if (causal < 0 || causal > 2) return FA_ERR_CAUSAL;
    if (B == 0 || Sq == 0) return FA_OK;
    if (Sk == 0) return FA_ERR_BAD_DIM;
    const long long BHq = (long long)B * Hq, BHkv = (long long)B * Hkv;
    const long long Tq = (Sq + kBM - 1) / kBM;
    if (BHq * Tq > 0x7fffffffLL || BHq > 0x7fffffffLL) return FA_ERR_BAD_DIM;
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_PTR;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA_ERR_ALIGN;
    const size_t nq = (size_t)BHq * Sq * D * 2, nkv = (size_t)BHkv * Sk * D * 2, nl = (size_t)BHq * Sq * 4;
    if (ranges_overlap(o, nq, q, nq) || ranges_overlap(o, nq, k, nkv) || ranges_overlap(o, nq, v, nkv) ||
        ranges_overlap(lse, nl, q, nq) || ranges_overlap(lse, nl, k, nkv) || ranges_overlap(lse, nl, v, nkv) ||
        ranges_overlap(lse, nl, o, nq))
        return FA_ERR_ALIAS;
    return FA_OK;
}

} // namespace fa

namespace {

// kernel: 0 = automatic (two-tile for D <= 128, one-tile for D = 256), 1 = two query tiles per
// CTA with 128-key steps (D 64 / 128), 2 = one query tile per CTA with 64-key steps (D 64 / 128 / 256),
// 3 = one query tile per CTA with 128-key steps (D 128); kernels 2 and 3 double-buffer the scores.
int run(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq, int Sk,
        int D, int causal, float scale, fa_stream_t stream, bool bf16, uint64_t timeout_ns, uint32_t inject,
        int kernel = 0, float tau = fa::kTauDefault)
{
    // ---- argument checks: no CUDA call before these pass
    {
        const int st = fa::check_fwd_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, kernel);
        if (st != FA_OK || B == 0 || Sq == 0) return st;
    }
    if (kernel == 0) kernel = (D == 256) ? 2 : 1;
    const long long BHq = (long long)B * Hq, BHkv = (long long)B * Hkv;
    const int key_tile = kernel == 2 ? 64 : fa::kBN;   // keys per step of the chosen kernel
    const long long Tq = (Sq + fa::kBM - 1) / fa::kBM, Tk = (Sk + key_tile - 1) / key_tile;
    const long long NP = (Tq + 1) / 2;

    // ---- device
    {
        const int st = fa::check_device();
        if (st != FA_OK) return st;
    }

    // ---- TMA descriptors
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return FA_ERR_TENSORMAP;
    fa::Maps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode(enc, &maps.q, q, bf16, D, Sq, BHq) || !encode(enc, &maps.k, k, bf16, D, Sk, BHkv, key_tile) ||
        !encode(enc, &maps.v, v, bf16, D, Sk, BHkv, key_tile) ||
        ((kernel == 1 || D == 256) && !encode(enc, &maps.o, o, bf16, D, Sq, BHq)))
        return FA_ERR_TENSORMAP;

    fa::Params p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.Tq = (int)Tq;
    p.Tk = (int)Tk;
    p.NP = (int)NP;
    p.group = Hq / Hkv;
    p.num_units = (int)(kernel >= 2 ? BHq * Tq : BHq * NP);
    // The kernel masks keys with -inf scores and takes the row maximum before scaling, so it
    // needs a positive multiplier: a negative scale negates the scores instead, and a zero
    // scale replaces every score by 0 (uniform weights), both exactly.
    p.smode = scale > 0.f ? 0u : (scale < 0.f ? 1u : 2u);
    p.sl2 = scale == 0.f ? 1.0f : (float)(std::fabs((double)scale) * 1.4426950408889634);
    p.coff = causal == 2 ? Sk - Sq : 0;
    p.timeout_ns = timeout_ns;
    p.inject = inject;
    p.o_al32 = aligned(o, 32) ? 1u : 0u;   // rows are 2*D bytes, so every row then starts on 32 bytes
    p.tau = tau;
    fa::set_schedule_divisors(p);

    cudaError_t e = kernel >= 2 ? fa::launch_fwd1(D, key_tile, bf16, causal != 0, maps, p, reinterpret_cast<cudaStream_t>(stream))
                                : fa::launch_fwd(D, bf16, causal != 0, maps, p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// 2-D view (inner, outer) of a row-major 16-bit matrix; box inner x outer, 128B swizzle.
bool encode_2d(EncodeTiledFn enc, CUtensorMap *m, const void *base, bool bf16, long long inner, long long outer,
               int box_inner, int box_outer)
{
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


} // namespace

extern "C" {

int fa_gemm(const void *a, const void *b, void *c, const float *bias, int M, int N, int K, int dtype, int out_fp32,
            int epilogue, fa_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return FA_ERR_BAD_DIM;
    if ((dtype != 0 && dtype != 1) || (out_fp32 != 0 && out_fp32 != 1) || epilogue < 0 || epilogue > 2)
        return FA_ERR_ARG;
    if (M == 0 || N == 0) return FA_OK;
    if (K == 0) return FA_ERR_BAD_DIM;
    if (K % 8 != 0 || N % 8 != 0) return FA_ERR_SHAPE;
    const long long Tm = (M + 127) / 128, Tn = (N + 255) / 256, nK = (K + 63) / 64;
    if (Tm * Tn > 0x7fffffffLL) return FA_ERR_BAD_DIM;
    if (!a || !b || !c || (epilogue && !bias)) return FA_ERR_NULL_PTR;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || (bias && !aligned(bias, 4))) return FA_ERR_ALIGN;
    const size_t na = (size_t)M * K * 2, nb = (size_t)K * N * 2, nc = (size_t)M * N * (out_fp32 ? 4 : 2);
    if (ranges_overlap(c, nc, a, na) || ranges_overlap(c, nc, b, nb) ||
        (bias && ranges_overlap(c, nc, bias, (size_t)N * 4)))
        return FA_ERR_ALIAS;
    int st = fa::check_device();
    if (st != FA_OK) return st;
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return FA_ERR_TENSORMAP;
    const bool bf16 = dtype == 0;
    CUtensorMap ma, mb;
    if (!encode_2d(enc, &ma, a, bf16, K, M, 64, 128) || !encode_2d(enc, &mb, b, bf16, N, K, 64, 64))
        return FA_ERR_TENSORMAP;
    fa::GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.c = c;
    p.bias = epilogue ? bias : nullptr;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Tm = (int)Tm;
    p.Tn = (int)Tn;
    p.nK = (int)nK;
    p.num_tiles = (int)(Tm * Tn);
    cudaError_t e = fa::launch_gemm(bf16, out_fp32 != 0, epilogue, ma, mb, p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_softmax_rows(const void *x, void *y, int rows, int cols, int dtype, fa_stream_t stream)
{
    if (rows < 0 || cols < 0) return FA_ERR_BAD_DIM;
    if (dtype != 0 && dtype != 1) return FA_ERR_ARG;
    if (rows == 0) return FA_OK;
    if (cols == 0) return FA_ERR_BAD_DIM;
    if (!x || !y) return FA_ERR_NULL_PTR;
    const uintptr_t al = dtype == 0 ? 4 : 2;
    if (!aligned(x, al) || !aligned(y, al)) return FA_ERR_ALIGN;
    const size_t n = (size_t)rows * cols * (dtype == 0 ? 4 : 2);
    if (x != y && ranges_overlap(x, n, y, n)) return FA_ERR_ALIAS;   // in place is fine, partial overlap is not
    int st = fa::check_device();
    if (st != FA_OK) return st;
    cudaError_t e = fa::launch_softmax_rows(dtype == 1, x, y, rows, cols, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}


int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq, int Sk,
           int D, int causal, float scale, fa_stream_t stream)
{
    return run(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream, true, 0, 0);
}

int fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                int Sk, int D, int causal, float scale, fa_stream_t stream)
{
    return run(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream, false, 0, 0);
}

int fa_fwd_debug(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                 int Sk, int D, int causal, float scale, fa_stream_t stream, int is_fp16, uint64_t timeout_ns,
                 uint32_t inject, int kernel, float tau)
{
    // negative: the default; above 15 an unnormalised P could leave the fp16 range
    if (!(tau >= 0.f && tau <= 15.f)) tau = tau < 0.f ? fa::kTauDefault : NAN;
    if (std::isnan(tau)) return FA_ERR_ARG;
    return run(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream, is_fp16 == 0, timeout_ns, inject,
               kernel, tau);
}

int fa_fwd_select(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, int causal, float scale, fa_stream_t stream, int dtype, int kernel)
{
    if (dtype != 0 && dtype != 1) return FA_ERR_ARG;
    return run(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream, dtype == 0, 0, 0, kernel);
}

const char *fa_strerror(int status)
{
    switch (status) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_NULL_PTR: return "FA_ERR_NULL_PTR: a tensor pointer is NULL";
    case FA_ERR_BAD_DIM: return "FA_ERR_BAD_DIM: negative size, Sk == 0 for a non-empty problem, or problem too large";
    case FA_ERR_HEADS: return "FA_ERR_HEADS: Hq and Hkv must be >= 1 with Hq % Hkv == 0";
    case FA_ERR_UNSUPPORTED_D: return "FA_ERR_UNSUPPORTED_D: D must be 64, 128 or 256 (and supported by the selected kernel)";
    case FA_ERR_ALIGN: return "FA_ERR_ALIGN: q/k/v/o must be 16-byte aligned and lse 4-byte aligned";
    case FA_ERR_ALIAS: return "FA_ERR_ALIAS: o or lse overlaps an input or each other";
    case FA_ERR_SCALE: return "FA_ERR_SCALE: scale is NaN or infinite";
    case FA_ERR_NO_DEVICE: return "FA_ERR_NO_DEVICE: no usable CUDA device";
    case FA_ERR_ARCH: return "FA_ERR_ARCH: the current device is not sm_103 (GB300)";
    case FA_ERR_TENSORMAP: return "FA_ERR_TENSORMAP: TMA descriptor encoding failed";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a bounded device-side wait expired";
    case FA_ERR_CAUSAL: return "FA_ERR_CAUSAL: causal must be 0 (none), 1 (top-left) or 2 (bottom-right)";
    case FA_ERR_SHAPE: return "FA_ERR_SHAPE: matrix rows must be 16-byte multiples (K and N multiples of 8)";
    case FA_ERR_ARG: return "FA_ERR_ARG: dtype, output type or epilogue selector out of range";
    case FA_ERR_TOO_LARGE: return "FA_ERR_TOO_LARGE: the problem needs more staging than FA_HOST_NOALLOC_MAX_BYTES";
    default: return "unknown fa status code";
    }
}

int fa_device_status(fa_stream_t stream, uint32_t *detail)
{
    uint32_t w = 0, wg = 0;
    if (fa::read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &w) != cudaSuccess) return FA_ERR_NO_DEVICE;
    uint32_t w1 = 0;
    if (fa::read_and_clear_gemm_status(&wg) != cudaSuccess) return FA_ERR_NO_DEVICE;
    if (fa::read_and_clear_fa1_status(&w1) != cudaSuccess) return FA_ERR_NO_DEVICE;
    uint32_t ws = 0;
    if (fa::read_and_clear_softmax_status(&ws) != cudaSuccess) return FA_ERR_NO_DEVICE;
    if (!(w & 1u)) w = (w1 & 1u) ? w1 : ((wg & 1u) ? wg : ws);   // attention kernels checked first
    if (detail) *detail = w;
    return (w & 1u) ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

} // extern "C"
