// gemm_sm103.cu -- tiled matrix product C = epilogue(A B) for GB300 (sm_103a).
//
// The tiled matrix product of "Guia Prático de Programação de GPU com Tiles", section 5
// (a K loop accumulating products of A and B tiles into an fp32 accumulator), with the
// optional bias + tanh-GELU epilogue of section 3 fused into the store (the course's lesson 9
// fuses a bias add into the matrix product in the same way):
//
//     C[m, n] = sum_k A[m, k] B[k, n]                       (epilogue 0)
//     C[m, n] = sum_k A[m, k] B[k, n] + bias[n]             (epilogue 1)
//     C[m, n] = gelu_tanh(sum_k A[m, k] B[k, n] + bias[n])  (epilogue 2)
//
// A [M, K] and B [K, N] row-major, bf16 or fp16; fp32 accumulation in tensor memory; C in
// the input type or fp32.
//
// Persistent CTAs (one per SM) walk 128 x 256 output tiles in M-grouped order.  Per CTA:
//   warp 0      TMA producer: A tile [128 x 64] (K-major) and B tile [64 x 256] (four
//               64-column MN-major panels) per 64-wide K block, into a 4-stage ring
//   warp 1      TMEM owner and MMA issuer (whole warp, one elected lane issues):
//               tcgen05.mma M=128 N=256 K=16, four per K block, into one of two
//               256-column TMEM accumulators (double-buffered across tiles)
//   warps 4-7   epilogue: one thread per output row reads its accumulator row from TMEM,
//               adds bias / applies tanh-GELU, converts and stores 16-byte chunks
#include <atomic>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"
#include "watchdog.cuh"

namespace fa {

__device__ unsigned int g_gemm_status;

namespace gemm {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;               // 16 KB
constexpr int B_PANEL = BK * 128;                  // 64 K-rows x 64 N-columns x 2 B = 8 KB
constexpr int B_BYTES = 4 * B_PANEL;               // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OFF_BAR = STAGES * STAGE_BYTES;
constexpr int NBAR = 2 * STAGES + 2 + 2 + 1;       // full, empty, acc full, acc empty, done
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int BYTES = OFF_MISC + 16;
constexpr int ALLOC = BYTES + 1024;
constexpr int THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

enum Site : uint32_t { S_EMPTY = 1, S_FULL = 2, S_ACC_EMPTY = 3, S_ACC_FULL = 4, S_DRAIN = 5, S_SMEM = 6 };

struct Tile {
    int tm, tn;
};

// M-grouped order: sixteen M-tiles share each sweep over N, so their B panels are reused in L2
// (the 152 tiles in flight then span about 16 x 10 tiles: 8192^3 bf16 ran 1642 TFLOP/s with
// groups of 8 and 1718 with groups of 16).
__device__ __forceinline__ Tile tile_of(int t, int Tm, int Tn)
{
    constexpr int GM = 16;
    const int per_group = GM * Tn;
    const int group = t / per_group;
    const int first = group * GM;
    const int gsize = min(Tm - first, GM);
    const int in = t - group * per_group;
    return Tile{first + in % gsize, in / gsize};
}

template <bool BF16, bool OUT_F32, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = sb + OFF_BAR;
    auto bar_full = [&](int s) { return bar0 + 8u * s; };
    auto bar_empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t barAccFull = bar0 + 8u * (2 * STAGES);       // + 8 * buffer
    const uint32_t barAccEmpty = barAccFull + 16u;              // + 8 * buffer
    const uint32_t barDone = barAccFull + 32u;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    const uint64_t tmo = p.timeout_ns;

    if (pad + (uint32_t)BYTES > dynamic_smem_size_u32()) {
        if (threadIdx.x == 0) atomicOr(&g_gemm_status, 1u | (S_SMEM << 8));
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(barAccFull, 1);
        mbar_init(barAccFull + 8, 1);
        mbar_init(barAccEmpty, 4);
        mbar_init(barAccEmpty + 8, 4);
        mbar_init(barDone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int G = gridDim.x;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_tiles; t += G) {
                const Tile tl = tile_of(t, p.Tm, p.Tn);
                for (int kb = 0; kb < p.nK; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!bounded_wait(bar_empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, tmo, S_EMPTY, &g_gemm_status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = sb + s * STAGE_BYTES, sB = sA + A_BYTES;
                    mbar_arrive_expect_tx(bar_full(s), STAGE_BYTES);
                    tma_load_2d(sA, &tmA, kb * BK, tl.tm * BM, bar_full(s));
#pragma unroll
                    for (int pn = 0; pn < 4; ++pn)
                        tma_load_2d(sB + pn * B_PANEL, &tmB, tl.tn * BN + pn * 64, kb * BK, bar_full(s));
                }
            }
            for (int x = max(0, it - STAGES); x < it; ++x)
                bounded_wait(bar_full(x % STAGES), (x / STAGES) & 1, abort_flag, tmo, S_DRAIN, &g_gemm_status, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (whole warp)
        constexpr uint32_t idesc = idesc_f16(BF16, BM, BN, true);   // B is MN-major
        constexpr uint32_t HI = sdesc_hi_sw128(1024);
        auto wait_u = [&](uint32_t bar, uint32_t parity, uint32_t site) {
            return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_flag, tmo, site, &g_gemm_status));
        };
        int it = 0, lt = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += G, ++lt) {
            const int ab = lt & 1;
            ok = wait_u(barAccEmpty + 8u * ab, ((lt >> 1) & 1) ^ 1, S_ACC_EMPTY);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(ab * BN);
            for (int kb = 0; kb < p.nK; ++kb, ++it) {
                const int s = it % STAGES;
                ok = wait_u(bar_full(s), (it / STAGES) & 1, S_FULL);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sA = sb + s * STAGE_BYTES, sB = sA + A_BYTES;
                const uint32_t alo = sdesc_lo(sA, 16), blo = sdesc_lo(sB, B_PANEL);
                static_assert(BK == 64, "one four-step group covers the K block");
                mma_ss_kmn4_elect(d, alo, blo, HI, idesc, kb > 0 ? 1u : 0u);
                tc_commit_elect(bar_empty(s));
            }
            if (!ok) break;
            tc_commit_elect(barAccFull + 8u * ab);
        }
        tc_commit_elect(barDone);
        bounded_wait(barDone, 0, abort_flag, tmo, S_DRAIN, &g_gemm_status, false);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int r = threadIdx.x - 128;                      // accumulator row == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        // Full 32-byte sectors when every row of C starts on 32 bytes (c aligned, row pitch a
        // multiple of 32 bytes): half the store instructions of 16-byte stores, no partial sectors.
        const bool al32 = ((reinterpret_cast<uintptr_t>(p.c) & 31u) == 0) && (p.N % (OUT_F32 ? 8 : 16) == 0);
        int lt = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += G, ++lt) {
            const Tile tl = tile_of(t, p.Tm, p.Tn);
            const int ab = lt & 1;
            ok = __all_sync(0xffffffffu, bounded_wait(barAccFull + 8u * ab, (lt >> 1) & 1, abort_flag, tmo,
                                                      S_ACC_FULL, &g_gemm_status));
            if (!ok) break;
            tc_fence_after();
            const int m = tl.tm * BM + r;
            const int n0 = tl.tn * BN;
            const uint32_t tacc = tmem + lane_off + (uint32_t)(ab * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld_x32(tacc + c, v);
                tmem_wait_ld();
                reg_fence_x32(v);
                float h[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) h[e] = __uint_as_float(v[e]);
                if (EPI >= 1) {
                    const int nb = n0 + c;
#pragma unroll
                    for (int e = 0; e < 32; ++e) h[e] += (nb + e < p.N) ? __ldg(p.bias + nb + e) : 0.f;
                }
                if (EPI == 2) {
                    // tanh-GELU: 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)))
                    const float k0 = 0.7978845608028654f, k1 = 0.044715f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float x = h[e];
                        h[e] = 0.5f * x * (1.f + tanh_approx(k0 * fmaf(k1 * x * x, x, x)));
                    }
                }
                if (m < p.M && al32) {
                    if (OUT_F32) {
                        float *crow = static_cast<float *>(p.c) + (size_t)m * p.N + n0 + c;
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8)
                            if (n0 + c + 8 * q8 < p.N) {
                                uint32_t w[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(h[8 * q8 + e]);
                                st_global_v8(crow + 8 * q8, w);
                            }
                    } else {
                        uint16_t *crow = static_cast<uint16_t *>(p.c) + (size_t)m * p.N + n0 + c;
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8)
                            if (n0 + c + 16 * q8 < p.N) {
                                uint32_t pk[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) pk[e] = pack2<BF16>(h[16 * q8 + 2 * e], h[16 * q8 + 2 * e + 1]);
                                st_global_v8(crow + 16 * q8, pk);
                            }
                    }
                } else if (m < p.M) {
                    if (OUT_F32) {
                        float *crow = static_cast<float *>(p.c) + (size_t)m * p.N + n0 + c;
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            if (n0 + c + 4 * q4 < p.N)
                                st_global_v4(crow + 4 * q4, __float_as_uint(h[4 * q4]), __float_as_uint(h[4 * q4 + 1]),
                                             __float_as_uint(h[4 * q4 + 2]), __float_as_uint(h[4 * q4 + 3]));
                    } else {
                        uint16_t *crow = static_cast<uint16_t *>(p.c) + (size_t)m * p.N + n0 + c;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            if (n0 + c + 8 * q4 < p.N)
                                st_global_v4(crow + 8 * q4, pack2<BF16>(h[8 * q4], h[8 * q4 + 1]),
                                             pack2<BF16>(h[8 * q4 + 2], h[8 * q4 + 3]),
                                             pack2<BF16>(h[8 * q4 + 4], h[8 * q4 + 5]),
                                             pack2<BF16>(h[8 * q4 + 6], h[8 * q4 + 7]));
                    }
                }
            }
            // accumulator buffer read: the MMA warp may overwrite it with a later tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barAccEmpty + 8u * ab);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <bool BF16, bool OUT_F32, int EPI>
static cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const GemmParams &p, cudaStream_t st)
{
    auto kern = gemm_kernel<BF16, OUT_F32, EPI>;
    static std::atomic<uint64_t> configured{0};
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ALLOC);
        if (e != cudaSuccess) return e;
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sm_count[dev].store(nsm, std::memory_order_relaxed);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    GemmParams q = p;
    if (q.timeout_ns == 0) q.timeout_ns = kDefaultTimeoutNs;
    const int grid = min(p.num_tiles, max(1, sm_count[dev].load(std::memory_order_relaxed)));
    kern<<<grid, THREADS, ALLOC, st>>>(a, b, q);
    return cudaGetLastError();
}

} // namespace gemm

cudaError_t launch_gemm(bool bf16, bool out_f32, int epilogue, const CUtensorMap &a, const CUtensorMap &b,
                        const GemmParams &p, cudaStream_t st)
{
#define G_CASE(BB, OO, EE) \
    if (bf16 == BB && out_f32 == OO && epilogue == EE) return gemm::launch_one<BB, OO, EE>(a, b, p, st);
    G_CASE(true, false, 0) G_CASE(true, false, 1) G_CASE(true, false, 2)
    G_CASE(true, true, 0) G_CASE(true, true, 1) G_CASE(true, true, 2)
    G_CASE(false, false, 0) G_CASE(false, false, 1) G_CASE(false, false, 2)
    G_CASE(false, true, 0) G_CASE(false, true, 1) G_CASE(false, true, 2)
#undef G_CASE
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_gemm_status(uint32_t *word)
{
    unsigned int w = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_gemm_status, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(zero));
    if (word) *word = w;
    return e;
}

} // namespace fa
