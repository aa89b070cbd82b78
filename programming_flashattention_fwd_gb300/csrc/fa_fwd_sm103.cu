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
// Persistent CTAs (one per SM) walk a static list of work units; a unit is a pair of
// 128-row query tiles ("a" = rows [256p, 256p+128), "b" = the next 128) of one (b, hq)
// that share the key/value stream.  While the softmax warps of one tile work, the tensor
// pipe runs the other tile's MMAs.
//
//   warp 0        TMA producer of K_j, V_j into a ring of shared-memory slots
//   warp 1        TMEM allocator + MMA issuer: S_x = Q_x K_j^T, O_x += P_x V_j (the whole warp in
//                 uniform control flow; one elected lane issues each group of four K-steps)
//   warp 2        TMA producer of query tiles into three rotating Q buffers
//   warp 3        idle
//   warps 4-7     softmax + correction + epilogue of tile a of every unit (one thread per row)
//   warps 8-11    the same for tile b
//
// TMEM (512 columns x 128 lanes, lane = query row):
//   S_a [0,128)  S_b [128,256)  fp32 scores; P (16-bit, two per column) overwrites
//                               the first 64 columns of S in place
//   O_a [256,256+D)  O_b [256+D,256+2D)  fp32 accumulators
//
// Differences from the guide's kernel: exp2 with |scale|*log2(e) folded into one FMA; the
// rescale of O is lazy (only when the running max grows by more than a factor 2^tau,
// tau = 12 unless a test sets it, so the unnormalised P stays <= 4096, well inside bf16/fp16
// range; O and l always share the same stale max, so the result is unchanged); a negative
// scale negates S inside the MMA and a zero scale zeroes Q at load time; K/V tails and the causal diagonal are masked only
// on the tiles that need it; fully masked causal tiles are skipped; the log-sum-exp is
// written out; output rows go out in full 32-byte sectors when o is 32-byte aligned, except
// that without the mask tile b's rows are staged in its finished query buffer and written by
// bulk tensor stores; K/V loads carry an L2 evict_last hint and query loads evict_first.
//
// Every wait is bounded (watchdog): on expiry the kernel records a status word, raises a
// CTA-wide abort flag, lets its own copies and MMAs drain, frees TMEM, writes NaN into o and lse
// of every query row the CTA was responsible for (so that no row of an abandoned call keeps a
// value that looks valid) and returns.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"
#include "schedule.h"

namespace fa {

__device__ unsigned int g_fa_status;  // watchdog word: bit 0 = a wait expired, bits 8-15 = first site

constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168;      // 65536 / 384, rounded down to the allocation granule
constexpr uint32_t kRegsLoad = 88;    // warps 0-3 after setmaxnreg.dec
constexpr uint32_t kRegsSoftmax = 208;// warps 4-11 after setmaxnreg.inc: 88*128 + 208*256 == 168*384
static_assert(kRegsLoad * 128 + kRegsSoftmax * 256 == kRegsLaunch * kThreads, "register split");
constexpr uint32_t kNegateA = 1u << 13;  // instruction-descriptor bit: negate A (scale < 0 -> S = -Q K^T)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

enum WaitSite : uint32_t {
    SITE_PROD_EMPTY = 1, SITE_MMA_Q = 2, SITE_MMA_FULL = 3, SITE_MMA_P = 4,
    SITE_SM_S = 5, SITE_SM_O = 6, SITE_DRAIN = 7, SITE_QFREE = 8, SITE_STAGED = 9
};

template <int D>
struct Cfg {
    static constexpr int TILE = kBM * D * 2;     // bytes of one 128-row, D-column 16-bit tile
    static constexpr int PANELS = D / 64;        // 64-column (128-byte) swizzle panels per tile
    static constexpr int PANEL = kBM * 128;      // bytes of one panel
    static constexpr int NQ = 3;                 // rotating query-tile buffers
    static constexpr int NS = (D == 128) ? 4 : 8;// K/V ring slots
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = NQ * TILE;
    static constexpr int OFF_BAR = OFF_RING + NS * TILE;
    static constexpr int NBAR = 2 * NQ + 2 * NS + 2 + 4 + 2 + 1 + 1;   // ..., O[2], done, tile b staged
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

// One probe of a phase by the whole (converged) warp, combined by a warp vote: true when the
// phase has completed for every lane.  The fast path of a warp-uniform wait, without a per-lane
// branch before the vote.
__device__ __forceinline__ bool mbar_try_wait_all(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "vote.sync.all.pred q, p, 0xffffffff;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// One arrival on `bar` by one elected lane of the (converged) warp, without a branch.
__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

// NaN (all-ones: NaN in bf16, fp16 and fp32) into query row `row` of head plane zq of o and lse.
template <int D>
__device__ __forceinline__ void poison_row(const Params &p, int zq, int row)
{
    if (row >= p.Sq) return;
    uint8_t *orow = static_cast<uint8_t *>(p.o) + ((size_t)zq * p.Sq + row) * (size_t)(D * 2);
#pragma unroll 1
    for (int c = 0; c < D * 2; c += 16) st_global_v4(orow + c, ~0u, ~0u, ~0u, ~0u);
    p.lse[(size_t)zq * p.Sq + row] = __uint_as_float(~0u);
}

// S = Q K^T at D = 128 in one block: both 64-column panels (eight 16-column K-steps; the second
// panel's operands start PANEL_OFF 16-byte units further) behind a single elect.sync, followed
// by the commit that tells the softmax warps S is ready -- fewer instructions for the MMA warp,
// which shares its SM sub-partition with two softmax warps.
template <uint32_t PANEL_OFF, bool TWO = false>
__device__ __forceinline__ void mma_s_d128_commit_elect(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                        uint32_t idesc, uint32_t bar, uint32_t bar2 = 0)
{
    if constexpr (TWO) {   // ... and a second commit (the K slot the MMAs read), same elected lane
        asm volatile("{\n\t.reg .b32 al, bl;\n\t.reg .b64 a, b;\n\t.reg .pred e, f, t;\n\t"
                     "setp.eq.b32 t, 0, 0;\n\tsetp.ne.b32 f, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                     "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, f;\n\t"
                     "add.u32 al, %1, 2;\n\tadd.u32 bl, %2, 2;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, 4;\n\tadd.u32 bl, %2, 4;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, 6;\n\tadd.u32 bl, %2, 6;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, %7;\n\tadd.u32 bl, %2, %7;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, %8;\n\tadd.u32 bl, %2, %8;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, %9;\n\tadd.u32 bl, %2, %9;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "add.u32 al, %1, %10;\n\tadd.u32 bl, %2, %10;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                     "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
                     "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
                     ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(bar), "r"(bar2), "n"(PANEL_OFF),
                       "n"(PANEL_OFF + 2), "n"(PANEL_OFF + 4), "n"(PANEL_OFF + 6)
                     : "memory");
        return;
    }
    asm volatile("{\n\t.reg .b32 al, bl;\n\t.reg .b64 a, b;\n\t.reg .pred e, f, t;\n\t"
                 "setp.eq.b32 t, 0, 0;\n\tsetp.ne.b32 f, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, f;\n\t"
                 "add.u32 al, %1, 2;\n\tadd.u32 bl, %2, 2;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, 4;\n\tadd.u32 bl, %2, 4;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, 6;\n\tadd.u32 bl, %2, 6;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, %6;\n\tadd.u32 bl, %2, %6;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, %7;\n\tadd.u32 bl, %2, %7;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, %8;\n\tadd.u32 bl, %2, %8;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "add.u32 al, %1, %9;\n\tadd.u32 bl, %2, %9;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}"
                 ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(bar), "n"(PANEL_OFF), "n"(PANEL_OFF + 2),
                   "n"(PANEL_OFF + 4), "n"(PANEL_OFF + 6)
                 : "memory");
}

// O += P V for one 64-key half (four 16-key steps, as mma_ts_mn4_elect) followed by a commit to
// `bar` from the same elected lane.
__device__ __forceinline__ void mma_pv_commit_elect(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                                    uint32_t idesc, uint32_t accumulate, uint32_t bar)
{
    asm volatile("{\n\t.reg .b32 ta, bl;\n\t.reg .b64 b;\n\t.reg .pred p, e, t;\n\t"
                 "setp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 t, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 b, {%2, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t"
                 "add.u32 ta, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, t;\n\t"
                 "add.u32 ta, %1, 16;\n\tadd.u32 bl, %2, 256;\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, t;\n\t"
                 "add.u32 ta, %1, 24;\n\tadd.u32 bl, %2, 384;\n\tmov.b64 b, {bl, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, t;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate), "r"(bar)
                 : "memory");
}

// One work unit, decoded identically by every role (the schedule is in schedule.h).
using Unit = PairUnit;

template <bool CAUSAL>
__device__ __forceinline__ bool unit_at(const Params &p, int round, Unit &u)
{
    return pair_unit<CAUSAL>(p, gridDim.x, blockIdx.x, round, u);
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p)
{
    using C = Cfg<D>;
    // Without the mask both tiles of a unit end on the same key step and their epilogues' row
    // stores compete: tile b's rows then go out as bulk tensor stores staged in its finished
    // query buffer (+2 % on the fp16 non-causal workload).  With the mask tile a ends a step
    // earlier and that staging measured 0.4 % slower, so there both tiles store rows directly.
    constexpr bool kStageB = !CAUSAL;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sQ = sb + C::OFF_Q;
    const uint32_t sRing = sb + C::OFF_RING;
    const uint32_t bar0 = sb + C::OFF_BAR;
    auto bar_q = [&](int i) { return bar0 + 8u * i; };                       // Q buffer i loaded
    auto bar_qfree = [&](int i) { return bar0 + 8u * (C::NQ + i); };         // Q buffer i no longer read
    auto bar_full = [&](int s) { return bar0 + 8u * (2 * C::NQ + s); };
    auto bar_empty = [&](int s) { return bar0 + 8u * (2 * C::NQ + C::NS + s); };
    const uint32_t barS0 = bar0 + 8u * (2 * C::NQ + 2 * C::NS);   // S_x ready (x = 0, 1)
    const uint32_t barP0 = barS0 + 16u;                            // P_x keys [64h, 64h+64) written: + 16x + 8h
    const uint32_t barO0 = barS0 + 48u;                            // O_x final for the unit
    const uint32_t barDone = barS0 + 64u;
    const uint32_t barStaged = barS0 + 72u;   // tile b's output rows staged in shared memory (4 warps)
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(bar_q(i), 1);
            mbar_init(bar_qfree(i), 1);
        }
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(barS0, 1);
        mbar_init(barS0 + 8, 1);
        for (int i = 0; i < 4; ++i) mbar_init(barP0 + 8 * i, 4);
        mbar_init(barO0, 1);
        mbar_init(barO0 + 8, 1);
        mbar_init(barDone, 1);
        mbar_init(barStaged, 4);
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

    if (warp < 4) {
        regs_dec<kRegsLoad>();
        if (warp == 0 && lane == 0) {
            // ======================================================== K/V producer
            // fault injection: bit 0 -- every CTA skips its first V tile (ring use 1); bit 1 -- only CTA 0 does
            const bool inj = (p.inject & 1u) || ((p.inject & 2u) && blockIdx.x == 0);
            const int skip = inj ? 1 : -1;
            const uint64_t keep = l2_policy_evict_last(); // K/V tiles are read again by other tiles
            int use = 0;                                  // ring uses armed so far
            bool ok = true;
            Unit u;
            for (int round = 0; ok && unit_at<CAUSAL>(p, round, u); ++round) {
                for (int j = 0; j < u.n && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv, ++use) {
                        const int s = use % C::NS;
                        if (!wait_bar(bar_empty(s), ((use / C::NS) & 1) ^ 1, abort_flag, tmo, SITE_PROD_EMPTY)) {
                            ok = false;
                            break;
                        }
                        if (use == skip) continue;
                        mbar_arrive_expect_tx(bar_full(s), C::TILE);
                        const CUtensorMap *m = kv ? &tmV : &tmK;
#pragma unroll
                        for (int pn = 0; pn < C::PANELS; ++pn)
                            tma_load_3d_hint(sRing + s * C::TILE + pn * C::PANEL, m, pn * 64, j * kBN, u.zkv,
                                             bar_full(s), keep);
                    }
                }
            }
            // Drain: every load this thread armed has landed before the CTA may exit.
            for (int x = max(0, use - C::NS); x < use; ++x)
                if (x != skip) wait_bar(bar_full(x % C::NS), (x / C::NS) & 1, abort_flag, tmo, SITE_DRAIN, false);
        } else if (warp == 2 && lane == 0) {
            // ======================================================== Q producer
            int tau = 0;   // query tiles loaded so far (buffer tau % 3)
            const uint64_t once = l2_policy_evict_first();   // each query tile is read once
            bool ok = true;
            Unit u;
            for (int round = 0; ok && unit_at<CAUSAL>(p, round, u); ++round) {
                for (int x = 0; x < 2; ++x) {
                    if ((x ? u.nB : u.nA) == 0) continue;   // absent, or no allowed key at all
                    const int buf = tau % C::NQ;
                    if (tau >= C::NQ &&
                        !wait_bar(bar_qfree(buf), ((tau / C::NQ) - 1) & 1, abort_flag, tmo, SITE_QFREE)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_q(buf), C::TILE);
                    const int t = x ? u.tB : u.tA;
                    // scale == 0: every score is 0, so load Q from a plane past the end of the
                    // tensor, which the copy engine fills with zeros
                    const int zq = p.smode == 2 ? p.B * p.Hq : u.zq;
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_3d_hint(sQ + buf * C::TILE + pn * C::PANEL, &tmQ, pn * 64, t * kBM, zq, bar_q(buf),
                                         once);
                    ++tau;
                }
            }
            for (int x = max(0, tau - C::NQ); x < tau; ++x)
                wait_bar(bar_q(x % C::NQ), (x / C::NQ) & 1, abort_flag, tmo, SITE_DRAIN, false);
        } else if (warp == 1) {
            // ======================================================== MMA issuer
            // The whole warp runs this loop in uniform control flow (so descriptors live in
            // uniform registers); one elected lane issues each tcgen05 instruction.
            const uint32_t idS = idesc_f16(BF16, kBM, kBN, false) | (p.smode == 1 ? kNegateA : 0u);
            constexpr uint32_t idPV = idesc_f16(BF16, kBM, D, true);
            constexpr uint32_t HI = sdesc_hi_sw128(1024);   // 8-row groups 1024 bytes apart
            const uint32_t tS[2] = {tmem + C::COL_S0, tmem + C::COL_S1};
            const uint32_t tO[2] = {tmem + C::COL_O0, tmem + C::COL_O1};
            auto wait_u = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
                if (mbar_try_wait_all(bar, parity)) return true;   // the usual case: already complete
                return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, tmo, site)) != 0;
            };

            // S = Q K^T: A = Q tile, B = K tile, both K-major (rows of D contiguous
            // elements) in 128B-swizzled 64-column panels; 16 columns per instruction.
            auto issue_s = [&](uint32_t dS, uint32_t sQt, uint32_t sK) {
                const uint32_t qlo = sdesc_lo(sQt, 16), klo = sdesc_lo(sK, 16);
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn) {   // 4 K-steps per 64-column panel
                    const uint32_t off = (uint32_t)(pn * C::PANEL) >> 4;
                    mma_ss_kk4_elect(dS, qlo + off, klo + off, HI, idS, pn > 0);
                }
            };
            // the same followed by commits to `bar` and `bar2` (at D = 128 in one block, one elect.sync)
            auto issue_s_commit2 = [&](uint32_t dS, uint32_t sQt, uint32_t sK, uint32_t bar, uint32_t bar2) {
                if constexpr (D == 128) {
                    constexpr uint32_t kPanelOff = (uint32_t)C::PANEL / 16;
                    mma_s_d128_commit_elect<kPanelOff, true>(dS, sdesc_lo(sQt, 16), sdesc_lo(sK, 16), HI, idS, bar, bar2);
                } else {
                    issue_s(dS, sQt, sK);
                    tc_commit_elect(bar);
                    tc_commit_elect(bar2);
                }
            };
            // the same followed by the commit to `bar` (at D = 128 in one block, one elect.sync)
            auto issue_s_commit = [&](uint32_t dS, uint32_t sQt, uint32_t sK, uint32_t bar) {
                if constexpr (D == 128) {
                    constexpr uint32_t kPanelOff = (uint32_t)C::PANEL / 16;
                    mma_s_d128_commit_elect<kPanelOff>(dS, sdesc_lo(sQt, 16), sdesc_lo(sK, 16), HI, idS, bar);
                } else {
                    issue_s(dS, sQt, sK);
                    tc_commit_elect(bar);
                }
            };
            // O += P V for keys [64h, 64h+64): A = P from TMEM (16-bit pairs per column),
            // B = V tile, MN-major (D contiguous per key row): 8-key groups 1024 bytes apart,
            // 64-column panels C::PANEL bytes apart; 16 keys per K-step.
            auto issue_pv_half = [&](uint32_t dO, uint32_t tP, uint32_t sV, int h, bool first) {
                const uint32_t vlo = sdesc_lo(sV, C::PANEL);
                mma_ts_mn4_elect(dO, tP + 32 * h, vlo + (uint32_t)((4 * h * 2048) >> 4), HI, idPV,
                                 (first && h == 0) ? 0u : 1u);
            };
            // tile b's second half releases the V slot in the same block (its P V are the last readers)
            auto issue_pv_half_commit = [&](uint32_t dO, uint32_t tP, uint32_t sV, uint32_t bar) {
                const uint32_t vlo = sdesc_lo(sV, C::PANEL);
                mma_pv_commit_elect(dO, tP + 32, vlo + (uint32_t)((4 * 2048) >> 4), HI, idPV, 1u, bar);
            };

            int use = 0;               // ring uses consumed (K_j = use, V_j = use + 1 within a step)
            int tau = 0;               // query tiles consumed
            uint32_t ks[2] = {0, 0};   // key steps done per tile slot (barS / barP phase)
            bool ok = true;
            Unit u;
            for (int round = 0; ok && unit_at<CAUSAL>(p, round, u); ++round) {
                const int nt = 2;                      // tile slots; a slot with nk == 0 has no work
                const int nk[2] = {u.nA, u.nB};
                int buf[2] = {0, 0}, qi[2] = {0, 0}, na = 0;
                for (int x = 0; x < 2; ++x) {
                    if (nk[x] == 0) continue;
                    qi[x] = tau + na;
                    buf[x] = qi[x] % C::NQ;
                    ++na;
                }
                tau += na;
                if (na == 0) continue;                 // no query row of this unit has a key
                const int uK0 = use;
                if (!wait_u(bar_full(uK0 % C::NS), (uK0 / C::NS) & 1, SITE_MMA_FULL)) {
                    ok = false;
                    break;
                }
                for (int x = 0; x < nt; ++x) {
                    if (nk[x] == 0) continue;
                    // each tile's first S goes out as soon as its own Q tile is in (tile b's Q is
                    // the one loaded last, into the buffer tile a of the previous unit released)
                    if (!wait_u(bar_q(buf[x]), (qi[x] / C::NQ) & 1, SITE_MMA_Q)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s_commit(tS[x], sQ + buf[x] * C::TILE, sRing + (uK0 % C::NS) * C::TILE, barS0 + 8u * x);
                    // without the mask tile b's buffer is released by its softmax warps once the
                    // output rows staged in it have been stored (its last S has completed by then)
                    if (nk[x] == 1 && (x == 0 || !kStageB)) tc_commit_elect(bar_qfree(buf[x]));
                }
                if (!ok) break;
                tc_commit_elect(bar_empty(uK0 % C::NS));
                for (int j = 0; j < u.n; ++j) {
                    const bool more = j + 1 < u.n;
                    const int uV = use + 1, uKn = use + 2;
                    if (!wait_u(bar_full(uV % C::NS), (uV / C::NS) & 1, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sV = sRing + (uV % C::NS) * C::TILE;
                    const uint32_t sKn = sRing + (uKn % C::NS) * C::TILE;
                    // At D = 128, K_{j+1} is waited for only before its first S MMA, so a late K
                    // tile does not hold back P_a V_j (+2 % at 4096 tokens, +4.5 % at 16384); at
                    // D = 64 the wait stays here (the later one measured 3.5 % slower there).
                    bool kn_ready = !more;
                    if (D != 128 && more) {
                        if (!wait_u(bar_full(uKn % C::NS), (uKn / C::NS) & 1, SITE_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        kn_ready = true;
                    }
                    for (int x = 0; x < nt; ++x) {
                        if (j < nk[x]) {
                            for (int h = 0; h < 2 && ok; ++h) {
                                ok = wait_u(barP0 + 16u * x + 8u * h, ks[x] & 1, SITE_MMA_P);
                                if (!ok) break;
                                tc_fence_after();
                                if (x == nt - 1 && h == 1)
                                    issue_pv_half_commit(tO[x], tS[x], sV, bar_empty(uV % C::NS));
                                else
                                    issue_pv_half(tO[x], tS[x], sV, h, j == 0);
                            }
                            if (!ok) break;
                            ++ks[x];
                            if (j == nk[x] - 1) tc_commit_elect(barO0 + 8u * x);
                        } else if (x == nt - 1) {
                            tc_commit_elect(bar_empty(uV % C::NS));   // tile b has no step j
                        }
                        if (j + 1 < nk[x]) {
                            if (!kn_ready) {
                                ok = wait_u(bar_full(uKn % C::NS), (uKn / C::NS) & 1, SITE_MMA_FULL);
                                if (!ok) break;
                                tc_fence_after();
                                kn_ready = true;
                            }
                            // tile b's S is the last reader of K_{j+1}: release its slot in the same block
                            if (x == nt - 1)
                                issue_s_commit2(tS[x], sQ + buf[x] * C::TILE, sKn, barS0 + 8u * x, bar_empty(uKn % C::NS));
                            else
                                issue_s_commit(tS[x], sQ + buf[x] * C::TILE, sKn, barS0 + 8u * x);
                            if (j + 2 == nk[x] && (x == 0 || !kStageB)) tc_commit_elect(bar_qfree(buf[x]));
                        }
                    }
                    if (!ok) break;
                    if (more && !(j + 1 < nk[nt - 1])) tc_commit_elect(bar_empty(uKn % C::NS));   // tile b had no S(j+1)
                    use += 2;
                }
            }
            // Drain: every MMA this warp issued has completed before TMEM is freed.
            tc_commit_elect(barDone);
            wait_bar(barDone, 0, abort_flag, tmo, SITE_DRAIN, false);
            __syncwarp();
        }
    } else {
        regs_inc<kRegsSoftmax>();
        // ============================================================ softmax / correction / epilogue
        const int x = (warp - 4) >> 2;             // tile slot: a (0) or b (1)
        const int r = threadIdx.x - 128 * (1 + x); // row within the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (x ? C::COL_S1 : C::COL_S0);
        const uint32_t tO = tmem + lane_off + (x ? C::COL_O1 : C::COL_O0);
        const uint32_t barS = barS0 + 8u * x, barP = barP0 + 16u * x, barO = barO0 + 8u * x;
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t ks = 0, uo = 0;
        int qt = 0;   // query tiles loaded so far (the Q producer's count: buffer of tile b = its index % NQ)
        uint32_t ub = 0;   // tile b epilogues staged (barStaged phase)
        bool ok = true;
        Unit u;
        for (int round = 0; ok && unit_at<CAUSAL>(p, round, u); ++round) {
            const int qb = qt + (u.nA > 0 ? 1 : 0);   // tile b's query-tile index (if it has keys)
            qt = qb + (u.nB > 0 ? 1 : 0);
            if (x == 1 && !u.hasB) continue;
            const int t = x ? u.tB : u.tA;
            const int nk = x ? u.nB : u.nA;
            const int row = t * kBM + r;
            if (nk == 0) {
                // no allowed key for any row of this tile: the empty softmax, o = 0, lse = -inf
                if (row < p.Sq) {
                    uint8_t *orow = static_cast<uint8_t *>(p.o) + ((size_t)u.zq * p.Sq + row) * (size_t)(D * 2);
#pragma unroll
                    for (int c = 0; c < D * 2; c += 16) st_global_v4(orow + c, 0u, 0u, 0u, 0u);
                    p.lse[(size_t)u.zq * p.Sq + row] = -INFINITY;
                }
                continue;
            }

            float m_used = -INFINITY;  // running max in exp2 units (possibly stale by <= p.tau)
            float l = 0.f;             // running sum of p at m_used
            for (int j = 0; j < nk; ++j) {
                ok = mbar_try_wait_all(barS, ks & 1) ||
                     __all_sync(0xffffffffu, wait_bar(barS, ks & 1, abort_flag, tmo, SITE_SM_S)) != 0;
                if (!ok) break;
                ++ks;
                tc_fence_after();

                // S in four 32-column loads; each load also returns the maximum of the 32 scores it
                // read (the reducing TMEM load), so an unmasked step needs no row-max arithmetic.
                uint32_t sv[kBN];
                float pm0, pm1, pm2, pm3;
                {
                    uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 0);
                    uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 32);
                    uint32_t(&v2)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 64);
                    uint32_t(&v3)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 96);
                    tmem_ld_red_max_x32(tS + 0, v0, pm0);
                    tmem_ld_red_max_x32(tS + 32, v1, pm1);
                    tmem_ld_red_max_x32(tS + 64, v2, pm2);
                    tmem_ld_red_max_x32(tS + 96, v3, pm3);
                    tmem_wait_ld();
                    reg_fence_x32(v0);
                    reg_fence_x32(v1);
                    reg_fence_x32(v2);
                    reg_fence_x32(v3);
                    reg_fence_f4(pm0, pm1, pm2, pm3);
                }
                float *s = reinterpret_cast<float *>(sv);

                // Mask keys past Sk (last key tile) and keys after the query row (causal diagonal);
                // those steps take the row maximum over the masked scores instead.
                const int kbase = j * kBN;
                const bool tail = kbase + kBN > p.Sk;
                const bool diag = CAUSAL && (kbase + kBN - 1 > t * kBM + p.coff);
                float mrow = fmaxf(fmax3(pm0, pm1, pm2), pm3);
                if (tail || diag) {
                    int lim = p.Sk - 1 - kbase;
                    if (CAUSAL) lim = min(lim, row + p.coff - kbase);
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c > lim) s[c] = -INFINITY;
                    // eight independent chains; 16 scores seed them, then each round of
                    // three-input max consumes 16 more (16 + 7 * 16 == 128 == kBN)
                    static_assert(kBN % 16 == 0 && kBN >= 16, "row-max chains cover the tile exactly");
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
                    for (int c = 16; c + 16 <= kBN; c += 16) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
                    }
                    mrow = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
                }
                const float m_new = fmaxf(m_used, mrow * sl2);

                // (branch-free: the warp's softmax step is bound by issue, and branches cost it)
                const bool rescale = j > 0 && m_new - m_used > p.tau;
                const float a_new = ex2_approx(m_used - m_new);
                const float alpha = rescale ? a_new : 1.f;
                l *= alpha;
                m_used = (j == 0 || rescale) ? m_new : m_used;
                const float msub = (m_used == -INFINITY) ? 0.f : m_used;
                const uint64_t negm2 = f2_pack(-msub, -msub);
                // p = exp2(s*sl2 - m) for 32 keys -> 16 packed 16-bit pairs; l accumulates fp32 p
                // in eight independent packed partial sums (no long dependent add chain).
                uint64_t lsum2[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) lsum2[i] = f2_pack(0.f, 0.f);
                auto exp_chunk = [&](int c, uint32_t(&pk)[16]) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = 32 * c + 2 * e;
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(s[i], s[i + 1]), sl2x2, negm2), t0, t1);
                        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                        lsum2[e & 7] = f2_add(lsum2[e & 7], f2_pack(p0, p1));
                        pk[e] = pack2<BF16>(p0, p1);
                    }
                };
                // P goes out in two halves (keys 0-63, 64-127) so the MMA warp can start the
                // first half of O += P V while the second half is still being exponentiated.
                auto publish = [&](uint32_t bar) {
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_elect(bar);
                };
                {
                    uint32_t pk0[16], pk1[16], pk2[16], pk3[16];
                    exp_chunk(0, pk0);
                    tmem_st_x16(tS + 0, pk0);
                    exp_chunk(1, pk1);
                    tmem_st_x16(tS + 16, pk1);
                    // Lazy correction of O (this row's previous P V products are complete: the
                    // S MMA that produced this tile was issued after them); it only has to land
                    // before the first half of P is published, so the vote waits until here.
                    if (__any_sync(0xffffffffu, rescale)) {
                        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                        for (int c = 0; c < D; c += 32) {
                            uint32_t ov[32];
                            tmem_ld_x32(tO + c, ov);
                            tmem_wait_ld();
                            reg_fence_x32(ov);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                float lo, hi;
                                f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), a2), lo, hi);
                                ov[e] = __float_as_uint(lo);
                                ov[e + 1] = __float_as_uint(hi);
                            }
                            tmem_st_x32(tO + c, ov);
                        }
                    }
                    exp_chunk(2, pk2);
                    publish(barP);
                    tmem_st_x16(tS + 32, pk2);
                    exp_chunk(3, pk3);
                    tmem_st_x16(tS + 48, pk3);
                    publish(barP + 8);
                }
                const uint64_t q0 = f2_add(f2_add(lsum2[0], lsum2[1]), f2_add(lsum2[2], lsum2[3]));
                const uint64_t q1 = f2_add(f2_add(lsum2[4], lsum2[5]), f2_add(lsum2[6], lsum2[7]));
                float la, lb;
                f2_unpack(f2_add(q0, q1), la, lb);
                l += la + lb;
            }
            if (!ok) break;

            // ---- epilogue: O / l -> 16-bit -> global (one 2*D-byte row per thread), and lse
            ok = mbar_try_wait_all(barO, uo & 1) ||
                 __all_sync(0xffffffffu, wait_bar(barO, uo & 1, abort_flag, tmo, SITE_SM_O)) != 0;
            if (!ok) break;
            ++uo;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const uint64_t il2 = f2_pack(inv_l, inv_l);
            uint8_t *orow = static_cast<uint8_t *>(p.o) + ((size_t)u.zq * p.Sq + row) * (size_t)(D * 2);
            // Without a causal mask both tiles of a unit end on the same key step, so their
            // epilogues run together with no other tile's work beside them: there O is read in
            // one round trip (all D columns, one wait).  With the mask, tile b's extra diagonal
            // step runs beside tile a's epilogue, and four shorter round trips measured faster.
            constexpr int kChunk = CAUSAL ? 32 : D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += kChunk) {
                uint32_t ovc[kChunk];
#pragma unroll
                for (int c = 0; c < kChunk; c += 32)
                    tmem_ld_x32(tO + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(ovc + c));
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kChunk; c += 32) reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(ovc + c));
#pragma unroll
                for (int c = c0; c < c0 + kChunk; c += 32) {
                    const uint32_t *ov = ovc + (c - c0);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float lo, hi;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1])), il2),
                                  lo, hi);
                        pk[e] = pack2<BF16>(lo, hi);
                    }
                    if (kStageB && x == 1) {
                        // tile b: rows staged in its finished query buffer (128B-swizzled, as the
                        // tensor map expects), written out below by bulk tensor stores
                        const uint32_t line = sQ + (uint32_t)(qb % C::NQ) * C::TILE + (uint32_t)(c / 64) * C::PANEL +
                                              (uint32_t)r * 128u;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t chunk = (uint32_t)(((c & 63) >> 3) + i) ^ (uint32_t)(r & 7);
                            st_shared_v4(line + (chunk << 4), pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    } else if (row < p.Sq) {
                        if (p.o_al32) {   // full 32-byte sectors: half the store instructions, no partial sectors
                            st_global_v8(orow + c * 2, pk);
                            st_global_v8(orow + c * 2 + 32, pk + 8);
                        } else {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                st_global_v4(orow + c * 2 + q4 * 16, pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2],
                                             pk[4 * q4 + 3]);
                        }
                    }
                }
            }
            if (row < p.Sq) {
                const float lse = l > 0.f ? (m_used + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
                p.lse[(size_t)u.zq * p.Sq + row] = lse;
            }
            if (kStageB && x == 1) {
                // Tile b's rows leave the SM as bulk tensor stores (rows >= Sq are clipped by the
                // map), so its softmax warps do not stall on 2*D-byte row stores while tile a's
                // epilogue stores its own rows.  Every writer makes its rows visible to the copy
                // engine and each warp arrives; the storing thread's wait is bounded like every
                // other (a warp that gave up on an earlier wait never arrives, and then no store
                // is issued).  The query buffer goes back to the Q producer once the stores have
                // read it; it holds the query tile of the unit after next.
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_elect(barStaged);
                if (r == 0 && wait_bar(barStaged, ub & 1, abort_flag, tmo, SITE_STAGED)) {
                    const uint32_t sb_b = sQ + (uint32_t)(qb % C::NQ) * C::TILE;
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn) tma_store_3d(&tmO, pn * 64, t * kBM, u.zq, sb_b + pn * C::PANEL);
                    tma_store_commit();
                    tma_store_wait_read();
                    mbar_arrive(bar_qfree(qb % C::NQ));
                }
                ++ub;
            }
        }
        if (kStageB && x == 1 && r == 0) tma_store_wait_all();   // every output store has landed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    } else if (warp >= 4 && *abort_flag) {
        // This CTA gave up on a wait: every row of every unit it was given gets NaN in o and lse
        // (all roles have stopped), so that none of them keeps a value that looks valid.  Each
        // softmax warpgroup covers the rows of its own tile slot.
        const int x = (warp - 4) >> 2;
        const int r = threadIdx.x - 128 * (1 + x);
        Unit u;
        for (int round = 0; unit_at<CAUSAL>(p, round, u); ++round)
            if (x == 0 || u.hasB) poison_row<D>(p, u.zq, (x ? u.tB : u.tA) * kBM + r);
    }
}

// ------------------------------------------------------------------------- host side
template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_one(const Maps &m, const Params &p, cudaStream_t stream)
{
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL>;
    const int smem = Cfg<D>::BYTES;
    // Per device: shared-memory opt-in, SM count, and a check that the compiled kernel
    // really uses kRegsLaunch registers per thread -- the setmaxnreg split above adds up
    // to exactly that launch allocation and could never be satisfied with less.
    static std::atomic<uint64_t> configured{0};
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        if (attr.numRegs != kRegsLaunch) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sm_count[dev].store(nsm, std::memory_order_relaxed);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    Params q = p;
    if (q.timeout_ns == 0) q.timeout_ns = kDefaultTimeoutNs;
    const int grid = min(p.num_units, max(1, sm_count[dev].load(std::memory_order_relaxed)));
    kern<<<grid, kThreads, smem, stream>>>(m.q, m.k, m.v, m.o, q);
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
