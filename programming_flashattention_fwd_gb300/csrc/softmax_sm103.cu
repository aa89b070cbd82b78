// softmax_sm103.cu -- numerically stable row softmax for GB300 (sm_103a).
//
// "Guia Prático de Programação de GPU com Tiles", section 4 (row softmax, one row per
// program): subtract the row maximum, exponentiate, sum, divide; columns past the row's end
// do not take part.  The kernel is HBM-bound, so each byte is read once and written once:
//  - rows up to 8192 values live in registers, a group of G = 32 .. 256 threads per row with
//    at most 32 values per thread, sized to the row so that short rows keep many rows (and
//    loads) in flight per SM;
//  - longer rows that fit shared memory are copied there whole by the bulk-copy engine, two
//    row buffers per CTA so the next row streams in while this one is normalised;
//  - rows beyond that take two passes (an online max/sum pass, then a normalising pass that
//    re-reads the row), one row per SM at a time so that the re-read comes from L2; rows whose
//    width is not a multiple of the 16-byte vector take a scalar two-pass kernel.
//
// x and y are [rows, cols] row-major, both fp32 or both bf16; arithmetic is fp32, exp via
// exp2 with the input pre-scaled by log2(e).
#include <cstdint>

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "watchdog.cuh"

namespace fa {

__device__ unsigned int g_softmax_status;   // watchdog word of the shared-memory path

namespace sm {

constexpr int THREADS = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <bool BF16>
struct IO;
template <>
struct IO<false> {   // fp32, vectors of 4
    static constexpr int VEC = 4;
    static constexpr int ESZ = 4;
    __device__ static void load(const void *base, size_t i, float (&v)[4])
    {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(base) + i);
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    }
    __device__ static void load_smem(uint32_t addr, float (&v)[4])
    {
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr));
    }
    __device__ static float load1(const void *base, size_t i) { return __ldg(reinterpret_cast<const float *>(base) + i); }
    __device__ static void store(void *base, size_t i, const float (&v)[4])
    {
        st_global_v4(reinterpret_cast<float4 *>(base) + i, __float_as_uint(v[0]), __float_as_uint(v[1]),
                     __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
    __device__ static void store1(void *base, size_t i, float v) { reinterpret_cast<float *>(base)[i] = v; }
};
template <>
struct IO<true> {    // bf16, vectors of 8
    static constexpr int VEC = 8;
    static constexpr int ESZ = 2;
    __device__ static void unpack(const uint32_t (&w)[4], float (&v)[8])
    {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    __device__ static void load(const void *base, size_t i, float (&v)[8])
    {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(base) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        unpack(w, v);
    }
    __device__ static void load_smem(uint32_t addr, float (&v)[8])
    {
        uint32_t w[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
        unpack(w, v);
    }
    __device__ static float load1(const void *base, size_t i)
    {
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(base) + i) << 16);
    }
    __device__ static void store(void *base, size_t i, const float (&v)[8])
    {
        st_global_v4(reinterpret_cast<uint4 *>(base) + i, pack2<true>(v[0], v[1]), pack2<true>(v[2], v[3]),
                     pack2<true>(v[4], v[5]), pack2<true>(v[6], v[7]));
    }
    __device__ static void store1(void *base, size_t i, float v)
    {
        reinterpret_cast<uint16_t *>(base)[i] = (uint16_t)(pack2<true>(v, 0.f) & 0xFFFFu);
    }
};

// Reduction over the G consecutive threads of a group (G = 32: one warp, by shuffles; G = 64 ..
// 256: the group's warps combine through shared memory).  Every thread of the CTA calls it the
// same number of times.
template <int G, bool MAX>
__device__ __forceinline__ float group_reduce(float v, float *scratch)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = MAX ? fmaxf(v, w) : v + w;
    }
    if constexpr (G == 32) {
        return v;
    } else {
        constexpr int NW = G / 32;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        __syncthreads();                    // scratch free from the previous reduction
        if (lane == 0) scratch[warp] = v;
        __syncthreads();
        const int w0 = (warp / NW) * NW;
        float r = scratch[w0];
#pragma unroll
        for (int w = 1; w < NW; ++w) r = MAX ? fmaxf(r, scratch[w0 + w]) : r + scratch[w0 + w];
        return r;
    }
}

// Rows held in registers: a group of G threads per row, at most NV vectors per thread.
// VECTOR: 16-byte vectors (cols a multiple of the vector width); else single elements.
template <bool BF16, int G, int NV, bool VECTOR>
__global__ void __launch_bounds__(THREADS) softmax_regs_kernel(const void *x, void *y, int rows, int cols)
{
    constexpr int W = VECTOR ? IO<BF16>::VEC : 1;
    constexpr int RPC = THREADS / G;     // rows per CTA iteration
    __shared__ float scratch[THREADS / 32];
    const int gi = threadIdx.x / G, t = threadIdx.x % G;
    const int nvec = cols / W;
    for (long long r0 = (long long)blockIdx.x * RPC; r0 < rows; r0 += (long long)gridDim.x * RPC) {
        const long long r = r0 + gi;
        const bool live = r < rows;       // (G == 256: the whole CTA shares one row)
        float v[NV][W];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int vi = t + i * G;
            if (live && vi < nvec) {
                if constexpr (VECTOR) {
                    IO<BF16>::load(x, (size_t)r * nvec + vi, v[i]);
                } else {
                    v[i][0] = IO<BF16>::load1(x, (size_t)r * cols + vi);
                }
#pragma unroll
                for (int e = 0; e < W; ++e) mx = fmaxf(mx, v[i][e]);
            } else {
#pragma unroll
                for (int e = 0; e < W; ++e) v[i][e] = -INFINITY;
            }
        }
        mx = group_reduce<G, true>(mx, scratch);
        const float mb = mx * kLog2e;
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
#pragma unroll
            for (int e = 0; e < W; ++e) {
                v[i][e] = ex2_approx(fmaf(v[i][e], kLog2e, -mb));
                sum += v[i][e];
            }
        sum = group_reduce<G, false>(sum, scratch);
        const float inv = 1.f / sum;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int vi = t + i * G;
            if (live && vi < nvec) {
#pragma unroll
                for (int e = 0; e < W; ++e) v[i][e] *= inv;
                if constexpr (VECTOR) {
                    IO<BF16>::store(y, (size_t)r * nvec + vi, v[i]);
                } else {
                    IO<BF16>::store1(y, (size_t)r * cols + vi, v[i][0]);
                }
            }
        }
    }
}

// Rows copied whole into shared memory by the bulk-copy engine: NBUF row buffers per CTA (the
// next row streams in while this one is normalised).  Three passes over the shared copy (max,
// sum of exponentials, normalised write); x is read from HBM exactly once.  Rows are 16-byte
// aligned (cols a multiple of the vector width, x aligned).
constexpr uint32_t kBulkChunk = 32768;   // bytes per bulk-copy instruction

template <bool BF16, int NBUF>
__global__ void __launch_bounds__(THREADS) softmax_smem_kernel(const void *x, void *y, int rows, int cols,
                                                                uint32_t row_bytes)
{
    constexpr int W = IO<BF16>::VEC;
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float scratch[THREADS / 32];
    __shared__ __align__(8) uint64_t bars[NBUF];
    __shared__ int abort_flag;
    const uint32_t base = smem_u32(dsm);
    const int nvec = cols / W;
    const long long my_rows = rows > (int)blockIdx.x ? (rows - 1 - (long long)blockIdx.x) / gridDim.x + 1 : 0;
    auto bar = [&](int b) { return smem_u32(&bars[b]); };
    if (threadIdx.x == 0) {
        for (int b = 0; b < NBUF; ++b) mbar_init(bar(b), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // thread 0: copy the CTA's i-th row into buffer i % NBUF
    auto issue = [&](long long i) {
        const long long r = blockIdx.x + i * gridDim.x;
        const int b = (int)(i % NBUF);
        const uint32_t dst = base + (uint32_t)b * row_bytes;
        const char *src = static_cast<const char *>(x) + (size_t)r * row_bytes;
        mbar_arrive_expect_tx(bar(b), row_bytes);
        for (uint32_t off = 0; off < row_bytes; off += kBulkChunk)
            bulk_load(dst + off, src + off, min(kBulkChunk, row_bytes - off), bar(b));
    };
    if (threadIdx.x == 0)
        for (long long i = 0; i < NBUF && i < my_rows; ++i) issue(i);
    for (long long i = 0; i < my_rows; ++i) {
        const long long r = blockIdx.x + i * gridDim.x;
        const int b = (int)(i % NBUF);
        if (!bounded_wait(bar(b), (uint32_t)((i / NBUF) & 1), &abort_flag, kTimeoutNs, 1, &g_softmax_status, false))
            return;   // every thread waits on the same copy, so all of them give up together
        const uint32_t rb = base + (uint32_t)b * row_bytes;
        float mx = -INFINITY;
        for (int vi = threadIdx.x; vi < nvec; vi += THREADS) {
            float v[W];
            IO<BF16>::load_smem(rb + (uint32_t)vi * 16u, v);
#pragma unroll
            for (int e = 0; e < W; ++e) mx = fmaxf(mx, v[e]);
        }
        mx = group_reduce<THREADS, true>(mx, scratch);
        const float mb = mx * kLog2e;
        float sum = 0.f;
        for (int vi = threadIdx.x; vi < nvec; vi += THREADS) {
            float v[W];
            IO<BF16>::load_smem(rb + (uint32_t)vi * 16u, v);
#pragma unroll
            for (int e = 0; e < W; ++e) sum += ex2_approx(fmaf(v[e], kLog2e, -mb));
        }
        sum = group_reduce<THREADS, false>(sum, scratch);
        const float inv = 1.f / sum;
        for (int vi = threadIdx.x; vi < nvec; vi += THREADS) {
            float v[W];
            IO<BF16>::load_smem(rb + (uint32_t)vi * 16u, v);
#pragma unroll
            for (int e = 0; e < W; ++e) v[e] = ex2_approx(fmaf(v[e], kLog2e, -mb)) * inv;
            IO<BF16>::store(y, (size_t)r * nvec + vi, v);
        }
        __syncthreads();   // every thread has finished reading buffer b
        if (threadIdx.x == 0 && i + NBUF < my_rows) {
            fence_proxy_async_smem();
            issue(i + NBUF);
        }
    }
}

// Any row length, scalar accesses (widths that are not a multiple of the 16-byte vector): pass 1
// keeps a running (max, sum) per thread and merges them; pass 2 re-reads the row and writes
// the normalised values.
template <bool BF16>
__global__ void __launch_bounds__(THREADS) softmax_twopass_kernel(const void *x, void *y, int rows, int cols)
{
    __shared__ float scratch[THREADS / 32];
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        float m = -INFINITY, s = 0.f;   // running max and sum of exp(x - m)
        for (int c = threadIdx.x; c < cols; c += THREADS) {
            const float xv = IO<BF16>::load1(x, (size_t)r * cols + c);
            if (xv > m) {
                s = (m == -INFINITY) ? 0.f : s * ex2_approx((m - xv) * kLog2e);
                m = xv;
            }
            s += ex2_approx(fmaf(xv, kLog2e, -m * kLog2e));
        }
        const float mr = group_reduce<THREADS, true>(m, scratch);
        const float sr = group_reduce<THREADS, false>(m == -INFINITY ? 0.f : s * ex2_approx((m - mr) * kLog2e), scratch);
        const float inv = 1.f / sr, mb = mr * kLog2e;
        for (int c = threadIdx.x; c < cols; c += THREADS) {
            const float xv = IO<BF16>::load1(x, (size_t)r * cols + c);
            IO<BF16>::store1(y, (size_t)r * cols + c, ex2_approx(fmaf(xv, kLog2e, -mb)) * inv);
        }
    }
}

// Long rows, one CTA of LT threads per SM: pass 1 (online max/sum) and pass 2 (normalise) each
// keep LU independent 16-byte loads in flight per thread, and with one row per SM at a time the
// rows in flight (152 x row bytes) stay in L2 for pass 2's re-read.
constexpr int LT = 1024;

template <bool BF16>
__global__ void __launch_bounds__(LT, 1) softmax_long_kernel(const void *x, void *y, int rows, int cols)
{
    constexpr int W = IO<BF16>::VEC;
    constexpr int LU = BF16 ? 2 : 4;   // 16 values in flight per thread (64 registers at 1024 threads)
    __shared__ float red[2][LT / 32];
    const int n = cols / W, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto reduce = [&](float v, bool is_max, int slot) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float w = __shfl_xor_sync(0xffffffffu, v, o);
            v = is_max ? fmaxf(v, w) : v + w;
        }
        if (lane == 0) red[slot][warp] = v;
        __syncthreads();
        float r = red[slot][0];
        for (int k = 1; k < LT / 32; ++k) r = is_max ? fmaxf(r, red[slot][k]) : r + red[slot][k];
        return r;
    };
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const size_t rb = (size_t)r * n;
        float m = -INFINITY, s = 0.f;
        for (int c0 = threadIdx.x; c0 < n; c0 += LT * LU) {
            float v[LU][W];
#pragma unroll
            for (int u = 0; u < LU; ++u) {
                const int c = c0 + u * LT;
                if (c < n) {
                    IO<BF16>::load(x, rb + c, v[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < W; ++e) v[u][e] = -INFINITY;
                }
            }
            float vm = m;
#pragma unroll
            for (int u = 0; u < LU; ++u)
#pragma unroll
                for (int e = 0; e < W; ++e) vm = fmaxf(vm, v[u][e]);
            if (vm > m) {
                s = (m == -INFINITY) ? 0.f : s * ex2_approx((m - vm) * kLog2e);
                m = vm;
            }
            const float mb = m * kLog2e;
#pragma unroll
            for (int u = 0; u < LU; ++u)
#pragma unroll
                for (int e = 0; e < W; ++e) s += ex2_approx(fmaf(v[u][e], kLog2e, -mb));
        }
        const float mr = reduce(m, true, 0);
        const float sr = reduce(m == -INFINITY ? 0.f : s * ex2_approx((m - mr) * kLog2e), false, 1);
        const float inv = 1.f / sr, mb = mr * kLog2e;
        for (int c0 = threadIdx.x; c0 < n; c0 += LT * LU) {
            float v[LU][W];
#pragma unroll
            for (int u = 0; u < LU; ++u)
                if (c0 + u * LT < n) IO<BF16>::load(x, rb + c0 + u * LT, v[u]);
#pragma unroll
            for (int u = 0; u < LU; ++u) {
                if (c0 + u * LT < n) {
#pragma unroll
                    for (int e = 0; e < W; ++e) v[u][e] = ex2_approx(fmaf(v[u][e], kLog2e, -mb)) * inv;
                    IO<BF16>::store(y, rb + c0 + u * LT, v[u]);
                }
            }
        }
        __syncthreads();   // red[] is reused by the next row
    }
}

static cudaError_t sm_count(int *nsm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(nsm, cudaDevAttrMultiProcessorCount, dev);
}

// Grid-stride launch over `units` (rows or row groups), at most eight CTAs per SM.
template <typename K>
static cudaError_t launch_grid(K kern, long long units, const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    int nsm = 1;
    cudaError_t e = sm_count(&nsm);
    if (e != cudaSuccess) return e;
    const long long grid = units < (long long)nsm * 8 ? units : (long long)nsm * 8;
    kern<<<(int)(grid > 0 ? grid : 1), THREADS, 0, st>>>(x, y, rows, cols);
    return cudaGetLastError();
}

// The register kernel with G threads per row and NV vectors per thread.  A thread holds at most
// 32 values (NV * vector width): more registers per thread cost more in resident warps than
// they gain (bf16 rows of 8192 values: 5051 GB/s with 8 vectors per thread, 6510 with 4).
template <bool BF16, bool VECTOR>
constexpr int kMaxNV = (VECTOR && BF16) ? 4 : 8;

template <bool BF16, bool VECTOR>
static cudaError_t launch_regs(long long n, const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    constexpr int NVM = kMaxNV<BF16, VECTOR>;
#define FA_SM_CASE(GG, NN)                                                                                   \
    if (n <= (long long)(GG) * (NN))                                                                         \
        return launch_grid(softmax_regs_kernel<BF16, GG, NN, VECTOR>, ((long long)rows + THREADS / (GG) - 1) / (THREADS / (GG)), \
                           x, y, rows, cols, st);
    FA_SM_CASE(32, 1) FA_SM_CASE(32, 2) FA_SM_CASE(32, 4)
    if constexpr (NVM == 8) {
        FA_SM_CASE(32, 8)
    }
    if constexpr (NVM == 8) {   // fp32: 4096 values as one 256-thread group (6740 GB/s) rather than two of 128 (6560)
        FA_SM_CASE(64, 8) FA_SM_CASE(256, 8)
    } else {
        FA_SM_CASE(64, NVM) FA_SM_CASE(128, NVM) FA_SM_CASE(256, NVM)
    }
#undef FA_SM_CASE
    return cudaErrorInvalidValue;
}

constexpr uint32_t kSmemLimit = 227 * 1024 - 1024;  // dynamic shared memory for row buffers

template <bool BF16, int NBUF>
static cudaError_t launch_smem(const void *x, void *y, int rows, int cols, uint32_t row_bytes, cudaStream_t st)
{
    auto kern = softmax_smem_kernel<BF16, NBUF>;
    const uint32_t smem = NBUF * row_bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int nsm = 1;
    if ((e = sm_count(&nsm)) != cudaSuccess) return e;
    const int per_sm = (int)(kSmemLimit / smem) > 0 ? (int)(kSmemLimit / smem) : 1;
    const long long cap = (long long)nsm * per_sm;
    const int grid = (int)(rows < cap ? rows : cap);
    kern<<<grid, THREADS, smem, st>>>(x, y, rows, cols, row_bytes);
    return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_typed(const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    constexpr int W = IO<BF16>::VEC;
    const bool vec = (cols % W == 0) && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 == 0);
    const long long n = vec ? cols / W : cols;
    if (vec && n <= (long long)THREADS * kMaxNV<BF16, true>) return launch_regs<BF16, true>(n, x, y, rows, cols, st);
    if (!vec && n <= (long long)THREADS * kMaxNV<BF16, false>) return launch_regs<BF16, false>(n, x, y, rows, cols, st);
    if (vec) {
        const uint64_t row_bytes = (uint64_t)cols * IO<BF16>::ESZ;
        if (2 * row_bytes <= kSmemLimit) return launch_smem<BF16, 2>(x, y, rows, cols, (uint32_t)row_bytes, st);
        if (row_bytes <= kSmemLimit) return launch_smem<BF16, 1>(x, y, rows, cols, (uint32_t)row_bytes, st);
        // one row per SM at a time, so that the second pass re-reads it from L2 (fp32 rows of
        // 65536 values: 5802 GB/s, against 4322 with eight rows per SM re-read from HBM)
        int nsm = 1;
        cudaError_t e = sm_count(&nsm);
        if (e != cudaSuccess) return e;
        softmax_long_kernel<BF16><<<rows < nsm ? rows : nsm, LT, 0, st>>>(x, y, rows, cols);
        return cudaGetLastError();
    }
    return launch_grid(softmax_twopass_kernel<BF16>, rows, x, y, rows, cols, st);
}

} // namespace sm

cudaError_t launch_softmax_rows(bool bf16, const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    return bf16 ? sm::launch_typed<true>(x, y, rows, cols, st) : sm::launch_typed<false>(x, y, rows, cols, st);
}

cudaError_t read_and_clear_softmax_status(uint32_t *word)
{
    unsigned int w = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_softmax_status, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_softmax_status, &zero, sizeof(zero));
    if (word) *word = w;
    return e;
}

} // namespace fa
