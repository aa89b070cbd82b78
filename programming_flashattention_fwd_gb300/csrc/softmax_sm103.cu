// softmax_sm103.cu -- numerically stable row softmax for GB300 (sm_103a).
//
// "Guia Prático de Programação de GPU com Tiles", section 4 (row softmax, one row per
// program): subtract the row maximum, exponentiate, sum, divide; columns past the row's end
// do not take part.  Here a row is handled by one warp (short rows) or one 256-thread CTA
// (rows up to 8192 fp32 / 16384 bf16 values), held in registers between one coalesced read
// and one write -- an HBM-bound kernel touches each byte once.  Longer rows take two passes
// (an online max/sum pass, then a normalising pass over the same row, mostly from L2).
//
// x and y are [rows, cols] row-major, both fp32 or both bf16; arithmetic is fp32, exp via
// exp2 with the input pre-scaled by log2(e).
#include <cstdint>

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace sm {

constexpr int THREADS = 256;
constexpr float kLog2e = 1.4426950408889634f;

template <bool BF16>
struct IO;
template <>
struct IO<false> {   // fp32, vectors of 4
    static constexpr int VEC = 4;
    __device__ static void load(const void *base, size_t i, float (&v)[4])
    {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(base) + i);
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
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
    __device__ static void load(const void *base, size_t i, float (&v)[8])
    {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(base) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
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

// Reduction over a group of G threads (G = 32: one warp; G = 256: the CTA through shared memory).
template <int G, bool MAX>
__device__ __forceinline__ float group_reduce(float v, float *scratch)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = MAX ? fmaxf(v, w) : v + w;
    }
    if (G == 32) return v;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();                    // scratch free from the previous reduction
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
#pragma unroll
    for (int w = 1; w < G / 32; ++w) r = MAX ? fmaxf(r, scratch[w]) : r + scratch[w];
    return r;
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

// Any row length: pass 1 keeps a running (max, sum) per thread and merges them; pass 2
// re-reads the row (from L2 for all but very long rows) and writes the normalised values.
template <bool BF16>
__global__ void __launch_bounds__(THREADS) softmax_twopass_kernel(const void *x, void *y, int rows, int cols)
{
    __shared__ float scratch[THREADS / 32];
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        float m = -INFINITY, s = 0.f;   // running max and sum of exp(x - m)
        for (int c = threadIdx.x; c < cols; c += THREADS) {
            const float xv = IO<BF16>::load1(x, (size_t)r * cols + c);
            if (xv > m) {
                s = s * ex2_approx((m - xv) * kLog2e) + 1.f;
                m = xv;
            } else {
                s += ex2_approx((xv - m) * kLog2e);
            }
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

template <typename K>
static cudaError_t launch_grid(K kern, long long units, const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    int dev = 0, nsm = 1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long grid = units < (long long)nsm * 8 ? units : (long long)nsm * 8;
    kern<<<(int)(grid > 0 ? grid : 1), THREADS, 0, st>>>(x, y, rows, cols);
    return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_typed(const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    constexpr int W = IO<BF16>::VEC;
    const bool vec = (cols % W == 0) && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 == 0);
    constexpr int NV = 8;
    if (vec) {
        if (cols <= 32 * NV * W) return launch_grid(softmax_regs_kernel<BF16, 32, NV, true>, ((long long)rows + 7) / 8, x, y, rows, cols, st);
        if (cols <= THREADS * NV * W) return launch_grid(softmax_regs_kernel<BF16, THREADS, NV, true>, rows, x, y, rows, cols, st);
    } else {
        if (cols <= 32 * NV) return launch_grid(softmax_regs_kernel<BF16, 32, NV, false>, ((long long)rows + 7) / 8, x, y, rows, cols, st);
        if (cols <= THREADS * NV) return launch_grid(softmax_regs_kernel<BF16, THREADS, NV, false>, rows, x, y, rows, cols, st);
    }
    return launch_grid(softmax_twopass_kernel<BF16>, rows, x, y, rows, cols, st);
}

} // namespace sm

cudaError_t launch_softmax_rows(bool bf16, const void *x, void *y, int rows, int cols, cudaStream_t st)
{
    return bf16 ? sm::launch_typed<true>(x, y, rows, cols, st) : sm::launch_typed<false>(x, y, rows, cols, st);
}

} // namespace fa
