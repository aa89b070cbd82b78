// fa_fwd_sm103.cu -- FlashAttention forward for GB300 (sm_103a): TMA + tcgen05 + TMEM.
//
// Algorithm (the flash-attention section of "Guia Prático de Programação de GPU com
// Tiles", restated): a block of 128 query rows keeps a running row maximum m, a running
// sum l and an fp32 accumulator O; for each 128-key block it forms S = Q K^T, takes
// p = exp(scale*S - m_new), rescales l and O by exp(m_old - m_new), adds sum(p) to l and
// P V (P cast to the input type) to O, and divides O by l once at the end.  The
// FlashAttention-4 features named in "Como Domar o Blackwell Sem Enlouquecer com CUDA"
// -- two MMA stages (S = Q K^T and O += P V), online softmax, grouped-query attention,
// TMA, tensor memory, warp specialisation -- are how it is mapped onto the hardware.
//
// One CTA owns a pair of query tiles (rows [256p, 256p+256) of one (b, hq)) that share
// the key/value stream; while the softmax warps of one tile work, the tensor pipe runs
// the other tile's MMAs.
//
//   warp 0        TMA producer: Q tiles once, then K_j, V_j into a ring of smem slots
//   warp 1        TMEM allocator + MMA issuer (one thread): S_x = Q_x K_j^T, O_x += P_x V_j
//   warps 2-3     idle
//   warps 4-7     softmax + correction + epilogue of query tile a (one thread per row)
//   warps 8-11    the same for query tile b
//
// TMEM (512 columns x 128 lanes, lane = query row):
//   S_a [0,128)  S_b [128,256)  fp32 scores; P (16-bit, two per column) overwrites
//                               the first 64 columns of S in place
//   O_a [256,256+D)  O_b [256+D,256+2D)  fp32 accumulators
//
// Differences from the guide's kernel: exp2 with scale*log2(e) folded into one FMA;
// the rescale of O is lazy (only when the running max grows by more than 2^8, so the
// unnormalised P stays <= 256, well inside bf16/fp16 range; O and l always share the
// same stale max, so the result is unchanged); K/V tails and the causal diagonal are
// masked only on the tiles that need it; fully masked causal tiles are skipped; the
// log-sum-exp is written out.
//
// Every wait is bounded (watchdog): on expiry the kernel records a status word, raises
// a CTA-wide abort flag, lets its own copies and MMAs drain, frees TMEM and returns.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

__device__ unsigned int g_fa_status;  // watchdog word: bit 0 = a wait expired, bits 8-15 = first site

constexpr int kThreads = 384;
constexpr float kTau = 8.0f;          // lazy-rescale threshold in log2 units (factor 256)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

enum WaitSite : uint32_t {
    SITE_PROD_EMPTY = 1, SITE_MMA_Q = 2, SITE_MMA_FULL = 3, SITE_MMA_P = 4,
    SITE_SM_S = 5, SITE_SM_O = 6, SITE_DRAIN = 7
};

template <int D>
struct Cfg {
    static constexpr int TILE = kBM * D * 2;     // bytes of one 128-row, D-column 16-bit tile
    static constexpr int PANELS = D / 64;        // 64-column (128-byte) swizzle panels per tile
    static constexpr int PANEL = kBM * 128;      // bytes of one panel
    static constexpr int NS = (D == 128) ? 5 : 8;// K/V ring slots
    static constexpr int OFF_Q = 0;              // two Q tiles (also the O staging buffers)
    static constexpr int OFF_RING = 2 * TILE;
    static constexpr int OFF_BAR = OFF_RING + NS * TILE;
    static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16 + 1024;   // + slack to align the base to 1024
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    static constexpr uint32_t TMEM_COLS = 512;
};

// Bounded wait on an mbarrier phase.  Returns false (and raises the abort flag, recording
// the site in the status word) when the wait expires, or returns false early when another
// role has already aborted and `check_abort` is set.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         uint64_t timeout_ns, uint32_t site, bool check_abort = true)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (check_abort && *abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) break;
        }
    }
    *abort_flag = 1;
    atomicCAS(&g_fa_status, 0u, 1u | (site << 8));
    atomicOr(&g_fa_status, 1u);
    return false;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Params p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sQ0 = sb + C::OFF_Q, sQ1 = sb + C::OFF_Q + C::TILE;
    const uint32_t sRing = sb + C::OFF_RING;
    const uint32_t barQ = sb + C::OFF_BAR;
    auto bar_full = [&](int s) { return sb + C::OFF_BAR + 8u * (1 + s); };
    auto bar_empty = [&](int s) { return sb + C::OFF_BAR + 8u * (1 + C::NS + s); };
    const uint32_t barS0 = sb + C::OFF_BAR + 8u * (1 + 2 * C::NS);
    const uint32_t barP0 = barS0 + 16u;
    const uint32_t barO0 = barS0 + 32u;
    const uint32_t barDone = barS0 + 48u;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    // ---- work unit: (b, hq, pair of query tiles); causal units are ordered heaviest first
    const int u = blockIdx.x;
    int bh, pr;
    if (CAUSAL) {
        const int nbh = p.B * p.Hq;
        pr = p.NP - 1 - u / nbh;
        bh = u % nbh;
    } else {
        bh = u / p.NP;
        pr = u % p.NP;
    }
    const int b = bh / p.Hq, hq = bh % p.Hq;
    const int kvh = hq / p.group;
    const int zq = b * p.Hq + hq, zkv = b * p.Hkv + kvh;
    const int tA = 2 * pr, tB = 2 * pr + 1;
    const bool hasB = tB < p.Tq;
    const int nA = CAUSAL ? min(p.Tk, tA + 1) : p.Tk;
    const int nB = hasB ? (CAUSAL ? min(p.Tk, tB + 1) : p.Tk) : 0;
    const int n = max(nA, nB);

    if (threadIdx.x == 0) {
        mbar_init(barQ, 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(barS0, 1);
        mbar_init(barS0 + 8, 1);
        mbar_init(barP0, 4);
        mbar_init(barP0 + 8, 4);
        mbar_init(barO0, 1);
        mbar_init(barO0 + 8, 1);
        mbar_init(barDone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(barQ, (hasB ? 2u : 1u) * C::TILE);
            for (int pn = 0; pn < C::PANELS; ++pn) {
                tma_load_3d(sQ0 + pn * C::PANEL, &tmQ, pn * 64, tA * kBM, zq, barQ);
                if (hasB) tma_load_3d(sQ1 + pn * C::PANEL, &tmQ, pn * 64, tB * kBM, zq, barQ);
            }
            const int skip = (p.inject & 1u) ? 1 : -1;   // ring use 1 = V_0
            int armed = 0;                                // ring uses issued so far
            bool ok = true;
            for (int j = 0; j < n && ok; ++j) {
                for (int kv = 0; kv < 2; ++kv) {
                    const int use = 2 * j + kv;
                    const int s = use % C::NS;
                    if (!wait_bar(bar_empty(s), ((use / C::NS) & 1) ^ 1, abort_flag, tmo, SITE_PROD_EMPTY)) {
                        ok = false;
                        break;
                    }
                    armed = use + 1;
                    if (use == skip) continue;
                    mbar_arrive_expect_tx(bar_full(s), C::TILE);
                    const CUtensorMap *m = kv ? &tmV : &tmK;
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_3d(sRing + s * C::TILE + pn * C::PANEL, m, pn * 64, j * kBN, zkv, bar_full(s));
                }
            }
            // Drain: every load this thread armed has landed before the CTA may exit.
            wait_bar(barQ, 0, abort_flag, tmo, SITE_DRAIN, false);
            for (int use = max(0, armed - C::NS); use < armed; ++use)
                if (use != skip)
                    wait_bar(bar_full(use % C::NS), (use / C::NS) & 1, abort_flag, tmo, SITE_DRAIN, false);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(BF16, kBM, kBN, false);
            constexpr uint32_t idPV = idesc_f16(BF16, kBM, D, true);
            const uint32_t tS0 = tmem + C::COL_S0, tS1 = tmem + C::COL_S1;
            const uint32_t tO0 = tmem + C::COL_O0, tO1 = tmem + C::COL_O1;

            // S = Q K^T: A = Q tile, B = K tile, both K-major (rows of D contiguous
            // elements) in 128B-swizzled 64-column panels; 16 columns per instruction.
            auto issue_s = [&](uint32_t dS, uint32_t sQ, uint32_t sK) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::PANEL + (kk & 3) * 32;
                    mma_ss(dS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), idS, kk > 0);
                }
            };
            // O += P V: A = P from TMEM (16-bit pairs per column), B = V tile, MN-major
            // (D contiguous per key row): 8-key groups 1024 bytes apart, 64-column
            // panels C::PANEL bytes apart; 16 keys per instruction.
            auto issue_pv = [&](uint32_t dO, uint32_t tP, uint32_t sV, bool first) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(dO, tP + kk * 8, sdesc_sw128(sV + kk * 2048, C::PANEL, 1024), idPV,
                           (first && kk == 0) ? 0u : 1u);
            };
            auto slot_k = [&](int j) { return (2 * j) % C::NS; };
            auto slot_v = [&](int j) { return (2 * j + 1) % C::NS; };
            auto ph_k = [&](int j) { return (uint32_t)(((2 * j) / C::NS) & 1); };
            auto ph_v = [&](int j) { return (uint32_t)(((2 * j + 1) / C::NS) & 1); };

            bool ok = wait_bar(barQ, 0, abort_flag, tmo, SITE_MMA_Q) &&
                      wait_bar(bar_full(slot_k(0)), ph_k(0), abort_flag, tmo, SITE_MMA_FULL);
            if (ok) {
                tc_fence_after();
                issue_s(tS0, sQ0, sRing + slot_k(0) * C::TILE);
                tc_commit(barS0);
                if (nB > 0) {
                    issue_s(tS1, sQ1, sRing + slot_k(0) * C::TILE);
                    tc_commit(barS0 + 8);
                }
                tc_commit(bar_empty(slot_k(0)));
            }
            for (int j = 0; j < n && ok; ++j) {
                const bool more = j + 1 < n;
                if (!wait_bar(bar_full(slot_v(j)), ph_v(j), abort_flag, tmo, SITE_MMA_FULL)) break;
                if (more && !wait_bar(bar_full(slot_k(j + 1)), ph_k(j + 1), abort_flag, tmo, SITE_MMA_FULL)) break;
                const uint32_t sV = sRing + slot_v(j) * C::TILE;
                const uint32_t sKn = more ? sRing + slot_k(j + 1) * C::TILE : 0u;
                if (j < nA) {
                    if (!wait_bar(barP0, j & 1, abort_flag, tmo, SITE_MMA_P)) break;
                    tc_fence_after();
                    issue_pv(tO0, tS0, sV, j == 0);
                    if (j == nA - 1) tc_commit(barO0);
                }
                if (j + 1 < nA) {
                    issue_s(tS0, sQ0, sKn);
                    tc_commit(barS0);
                }
                if (j < nB) {
                    if (!wait_bar(barP0 + 8, j & 1, abort_flag, tmo, SITE_MMA_P)) break;
                    tc_fence_after();
                    issue_pv(tO1, tS1, sV, j == 0);
                    if (j == nB - 1) tc_commit(barO0 + 8);
                }
                tc_commit(bar_empty(slot_v(j)));
                if (j + 1 < nB) {
                    issue_s(tS1, sQ1, sKn);
                    tc_commit(barS0 + 8);
                }
                if (more) tc_commit(bar_empty(slot_k(j + 1)));
            }
            // Drain: every MMA this thread issued has completed before TMEM is freed.
            tc_commit(barDone);
            wait_bar(barDone, 0, abort_flag, tmo, SITE_DRAIN, false);
        }
    } else if (warp >= 4) {
        // ============================================================ softmax / correction / epilogue
        const int x = (warp - 4) >> 2;             // which query tile of the pair
        const int r = threadIdx.x - 128 * (1 + x); // row within the tile == TMEM lane
        const int t = x ? tB : tA;
        const int nk = x ? nB : nA;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (x ? C::COL_S1 : C::COL_S0);
        const uint32_t tO = tmem + lane_off + (x ? C::COL_O1 : C::COL_O0);
        const uint32_t barS = barS0 + 8u * x, barP = barP0 + 8u * x, barO = barO0 + 8u * x;
        const int row = t * kBM + r;
        const float sl2 = p.sl2;

        float m_used = -INFINITY;  // running max in exp2 units (possibly stale by <= kTau)
        float l = 0.f;             // running sum of p at m_used
        bool ok = nk > 0;
        for (int j = 0; j < nk && ok; ++j) {
            ok = __all_sync(0xffffffffu, wait_bar(barS, j & 1, abort_flag, tmo, SITE_SM_S));
            if (!ok) break;
            tc_fence_after();

            float s[kBN];
            {
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld_x32(tS + 0, v0);
                tmem_ld_x32(tS + 32, v1);
                tmem_ld_x32(tS + 64, v2);
                tmem_ld_x32(tS + 96, v3);
                tmem_wait_ld();
                reg_fence_x32(v0);
                reg_fence_x32(v1);
                reg_fence_x32(v2);
                reg_fence_x32(v3);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = __uint_as_float(v0[c]);
                    s[32 + c] = __uint_as_float(v1[c]);
                    s[64 + c] = __uint_as_float(v2[c]);
                    s[96 + c] = __uint_as_float(v3[c]);
                }
            }

            if (p.smode == 1) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) s[c] = -s[c];
            } else if (p.smode == 2) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) s[c] = 0.f;
            }

            // Mask keys past Sk (last key tile) and keys after the query row (causal diagonal).
            const int kbase = j * kBN;
            const bool tail = kbase + kBN > p.Sk;
            const bool diag = CAUSAL && (kbase + kBN - 1 > t * kBM);
            if (tail || diag) {
                int lim = p.Sk - 1 - kbase;
                if (CAUSAL) lim = min(lim, row - kbase);
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c > lim) s[c] = -INFINITY;
            }

            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < kBN; c += 4) {
                mx0 = fmaxf(mx0, s[c]);
                mx1 = fmaxf(mx1, s[c + 1]);
                mx2 = fmaxf(mx2, s[c + 2]);
                mx3 = fmaxf(mx3, s[c + 3]);
            }
            const float m_new = fmaxf(m_used, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);

            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_used = m_new;
            } else if (m_new - m_used > kTau) {
                alpha = ex2_approx(m_used - m_new);
                l *= alpha;
                m_used = m_new;
                rescale = true;
            }
            // Lazy correction of O (this row's previous P V products are complete: the
            // S MMA that produced this tile was issued after them).
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t ov[32];
                    tmem_ld_x32(tO + c, ov);
                    tmem_wait_ld();
                    reg_fence_x32(ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st_x32(tO + c, ov);
                }
            }

            const float msub = (m_used == -INFINITY) ? 0.f : m_used;
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2_approx(fmaf(s[32 * c + 2 * e], sl2, -msub));
                    const float p1 = ex2_approx(fmaf(s[32 * c + 2 * e + 1], sl2, -msub));
                    ls0 += p0;
                    ls1 += p1;
                    pk[e] = pack2<BF16>(p0, p1);
                }
                tmem_st_x16(tS + 16 * c, pk);
            }
            l += ls0 + ls1;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barP);
        }

        // ---- epilogue: O / l -> 16-bit -> swizzled smem (the tile's Q buffer) -> TMA store
        const uint32_t stage = x ? sQ1 : sQ0;
        uint8_t *stage_ptr = smem + C::OFF_Q + x * C::TILE;
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(barO, 0, abort_flag, tmo, SITE_SM_O));
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t ov[32];
                tmem_ld_x32(tO + c, ov);
                tmem_wait_ld();
                reg_fence_x32(ov);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2<BF16>(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
                const int panel = c >> 6;
                const int chunk0 = (c & 63) >> 3;   // first 16-byte chunk of these 32 columns
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int chunk = (chunk0 + q4) ^ (r & 7);
                    uint4 val = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    *reinterpret_cast<uint4 *>(stage_ptr + panel * C::PANEL + r * 128 + chunk * 16) = val;
                }
            }
            if (row < p.Sq) {
                const float lse = l > 0.f ? (m_used + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
                p.lse[(size_t)zq * p.Sq + row] = lse;
            }
            fence_proxy_async_smem();
        }
        named_bar_sync(1 + x, 128);
        if (r == 0 && nk > 0 && !*abort_flag) {
            for (int pn = 0; pn < C::PANELS; ++pn)
                tma_store_3d(&tmO, pn * 64, t * kBM, zq, stage + pn * C::PANEL);
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------- host side
template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_one(const Maps &m, const Params &p, cudaStream_t stream)
{
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL>;
    const int smem = Cfg<D>::BYTES;
    static std::atomic<uint64_t> configured{0};   // bit d: attribute set on device d
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    Params q = p;
    if (q.timeout_ns == 0) q.timeout_ns = kDefaultTimeoutNs;
    kern<<<p.num_units, kThreads, smem, stream>>>(m.q, m.k, m.v, m.o, q);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int D, bool bf16, bool causal, const Maps &m, const Params &p, cudaStream_t st)
{
#define FA_CASE(DD, BB, CC) \
    if (D == DD && bf16 == BB && causal == CC) return launch_one<DD, BB, CC>(m, p, st);
    FA_CASE(64, true, false) FA_CASE(64, true, true) FA_CASE(64, false, false) FA_CASE(64, false, true)
    FA_CASE(128, true, false) FA_CASE(128, true, true) FA_CASE(128, false, false) FA_CASE(128, false, true)
#undef FA_CASE
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *word)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int w = 0;
    e = cudaMemcpyFromSymbol(&w, g_fa_status, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero));
    if (word) *word = w;
    return e;
}

} // namespace fa
