// fa_fwd1_sm103.cu -- FlashAttention forward, one query tile per CTA, with double-buffered
// scores in tensor memory: the variant for head dimension 256 (64-key steps) and two
// alternatives for D = 128 (64- or 128-key steps).  Same computation as fa_fwd_sm103.cu (the flash-attention
// section of "Guia Prático de Programação de GPU com Tiles"; the FlashAttention-4 features of
// "Como Domar o Blackwell Sem Enlouquecer com CUDA"); the guide's troubleshooting item trades
// the 128-row block for 64 to save memory, which is what the key tile does here.
//
// With D = 256 the two-tile layout of the main kernel no longer fits in TMEM (2 x 128 score
// columns + 2 x 256 accumulator columns > 512).  Instead one 128-row query tile owns
//   S_0 [0,BN)  S_1 [BN,2BN)   fp32 scores of two consecutive key tiles of BN keys; P (16-bit
//                              pairs) overwrites the first BN/2 columns of its S
//   O   [2BN, 2BN+D)           fp32 accumulator
//   Q   [2BN+D, 2BN+3D/2)      the query tile (16-bit pairs; D >= 128), copied in from shared
//                              memory by tcgen05.cp at the start of the tile
// and the MMA warp computes S(j+1) = Q K_{j+1}^T while the softmax works on S(j); then
// O += P(j) V_j.  Per 64-key step the tensor pipe has 2 x 128*64*D multiply-adds (1024 cycles
// at D = 256), which the softmax of 64 keys per row fits under.  With Q read from tensor memory
// the score MMAs take only K from shared memory: 64 KB of operand reads per step at D = 256
// instead of 128 KB, which had held the tensor pipe to about 80 % of its rate.
//
//   warp 0       TMA producer of K / V tiles in the order the MMAs consume them (K_0, K_1,
//                V_0, K_2, V_1, ...), into a ring of BN-row slots
//   warp 1       TMEM owner and MMA issuer (whole warp; one elected lane issues)
//   warp 2       TMA producer of query tiles (two rotating buffers at D = 128, one at D = 256);
//                at D = 256 also the bulk tensor stores of each tile's output rows, which the
//                epilogue stages in the query buffer once the next query tile is in TMEM
//   warps 4-7    softmax / lazy correction / epilogue, one thread per query row
//
// The softmax publishes P(j) as soon as it is written; only a step that rescales O first waits
// for P V(j-1), and the epilogue waits for the last P V of its tile.  Every wait is bounded, as
// in the main kernel; a CTA that gives up writes NaN into o and lse of every query row it was
// given.
#include <atomic>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"
#include "schedule.h"
#include "watchdog.cuh"

namespace fa {

__device__ unsigned int g_fa1_status;

namespace one {

constexpr int BM = 128;
constexpr int THREADS = 256;
constexpr uint32_t kNegateA = 1u << 13;  // instruction-descriptor bit: negate A (scale < 0 -> S = -Q K^T)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

enum Site : uint32_t {
    S_EMPTY = 1, S_Q = 2, S_FULL = 3, S_P = 4, S_S = 5, S_PV = 6, S_DRAIN = 7, S_QFREE = 8, S_SMEM = 9, S_STAGED = 10
};

// BN keys per step: 64 (the only width at D = 256 whose two score buffers and O fit TMEM; at
// D = 128 the smaller-tile variant) or 128 (D = 128: the same step as the two-tile kernel).
constexpr int KVTILE_BYTES(int D, int BN) { return BN * D * 2; }

template <int D, int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int QTILE = BM * D * 2;       // 128 rows
    static constexpr int KVTILE = BN * D * 2;      // BN rows
    static constexpr int PANELS = D / 64;
    static constexpr int QPANEL = BM * 128;        // 16 KB
    static constexpr int KVPANEL = BN * 128;       // BN rows of one 64-column panel
    // D = 256: one query buffer and a five-slot K/V ring.  With two query buffers only three
    // 32 KB slots fit, one tile of lookahead, and the MMAs wait for K/V loads (+6 % causal,
    // +12 % non-causal measured for the deeper ring).  D = 128: two query buffers and as many
    // K/V slots as fit (eight of 16 KB for 64-key steps, five of 32 KB for 128-key steps).  From
    // D = 128 up a query buffer is free again once its tile has been copied into tensor memory.
    static constexpr int NQ = (D == 256) ? 1 : 2;
    static constexpr int NS = (KVTILE_BYTES(D, BN_) == 16384) ? 8 : 5;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = NQ * QTILE;
    static constexpr int OFF_BAR = OFF_RING + NS * KVTILE;
    // D = 256: the finished tile's output rows are staged in the query buffer (free once the next
    // tile's query tile has been copied into tensor memory) and leave by bulk tensor stores
    static constexpr bool STAGE_O = (D == 256);
    static constexpr int NBAR = 2 * NQ + 2 * NS + 2 + 2 + 2 + 1 + 4;   // q, qfree, full, empty, S[2], P[2], PV[2], done, qcp, staged[2], oread
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    // at D = 64 at least 80 KB, so that no third CTA is co-resident on an SM (two allocations of
    // 256 tensor-memory columns fill it)
    static constexpr int ALLOC_MIN = (D == 64) ? 80 * 1024 : 0;
    static constexpr int ALLOC_RAW = (BYTES + 1024 <= 232448) ? BYTES + 1024 : 232448;
    static constexpr int ALLOC = ALLOC_RAW > ALLOC_MIN ? ALLOC_RAW : ALLOC_MIN;
    // D >= 128: the query tile also lives in tensor memory (16-bit pairs, D/2 columns), copied
    // in once per tile, so that the score MMAs read only K from shared memory (at D = 256 the
    // operand reads of Q K^T from shared memory otherwise bound the tensor pipe)
    static constexpr bool QT = (D >= 128);
    static constexpr uint32_t COL_S0 = 0, COL_S1 = BN, COL_O = 2 * BN, COL_Q = 2 * BN + D;
    static_assert(!STAGE_O || (QT && NQ == 1 && QTILE == BM * D * 2), "O staged in the one query buffer");
    static constexpr uint32_t TMEM_COLS = (2 * BN + D + (QT ? D / 2 : 0) <= 256) ? 256 : 512;
    static_assert(2 * BN + D + (QT ? D / 2 : 0) <= 512, "tensor-memory columns");
};

// One arrival on `bar` by one elected lane of the (converged) warp.
__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

// One non-blocking probe of a phase by the whole (converged) warp, combined by a warp vote (the
// fast path of a warp-uniform wait, without a per-lane branch before the vote).
__device__ __forceinline__ bool mbar_try_wait_all(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "vote.sync.all.pred q, p, 0xffffffff;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// S = Q K^T over all NP 64-column panels of D (four 16-column K-steps each; the panels of Q and K
// start QOFF and KOFF 16-byte units apart) behind one elect.sync, followed by two commits from the
// same elected lane (S ready; the K slot released): fewer instructions for the MMA warp, which
// shares its SM sub-partition with a softmax warp.
#define F1_S_STEP(OFF) "add.u32 al, qa, " #OFF ";\n\tadd.u32 bl, ka, " #OFF ";\n\t"                        \
                       "mov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"                                   \
                       "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
#define F1_S_PANEL(ACC) "mov.b64 a, {qa, %3};\n\tmov.b64 b, {ka, %3};\n\t"                                  \
                        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, " #ACC ";\n\t"                 \
                        F1_S_STEP(2) F1_S_STEP(4) F1_S_STEP(6)
#define F1_S_NEXT "add.u32 qa, qa, %7;\n\tadd.u32 ka, ka, %8;\n\t" F1_S_PANEL(t)
#define F1_S_HEAD "{\n\t.reg .b32 qa, ka, al, bl;\n\t.reg .b64 a, b;\n\t.reg .pred e, f, t;\n\t"          \
                  "setp.eq.b32 t, 0, 0;\n\tsetp.ne.b32 f, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"          \
                  "mov.b32 qa, %1;\n\tmov.b32 ka, %2;\n\t" F1_S_PANEL(f)
#define F1_S_TAIL "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"        \
                  "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
template <int NP, uint32_t QOFF, uint32_t KOFF>
__device__ __forceinline__ void mma_s_commit2_elect(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                                    uint32_t idesc, uint32_t bar1, uint32_t bar2)
{
    static_assert(NP == 1 || NP == 2 || NP == 4, "64-column panels of D");
    if constexpr (NP == 1)
        asm volatile(F1_S_HEAD F1_S_TAIL ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(bar1),
                     "r"(bar2), "n"(QOFF), "n"(KOFF) : "memory");
    else if constexpr (NP == 2)
        asm volatile(F1_S_HEAD F1_S_NEXT F1_S_TAIL ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc),
                     "r"(bar1), "r"(bar2), "n"(QOFF), "n"(KOFF) : "memory");
    else
        asm volatile(F1_S_HEAD F1_S_NEXT F1_S_NEXT F1_S_NEXT F1_S_TAIL ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi),
                     "r"(idesc), "r"(bar1), "r"(bar2), "n"(QOFF), "n"(KOFF) : "memory");
}
#undef F1_S_STEP
#undef F1_S_PANEL
#undef F1_S_NEXT
#undef F1_S_HEAD
#undef F1_S_TAIL

// The query tile into tensor memory: one 128-row x 32-byte copy per 16 columns of D (lane = row,
// 8 columns of 16-bit pairs each), read from the 128-byte-swizzled, K-major tile that TMA wrote
// (the same addressing as an MMA A operand), all NP panels behind one elect.sync, then a commit
// that releases the shared-memory buffer once the copies are done.
#define F1_CP_STEP(TOFF, SOFF) "add.u32 ta, tq, " #TOFF ";\n\tadd.u32 al, qa, " #SOFF ";\n\t"                   \
                               "mov.b64 a, {al, %2};\n\t@e tcgen05.cp.cta_group::1.128x256b [ta], a;\n\t"
#define F1_CP_PANEL "mov.b64 a, {qa, %2};\n\t@e tcgen05.cp.cta_group::1.128x256b [tq], a;\n\t"                  \
                    F1_CP_STEP(8, 2) F1_CP_STEP(16, 4) F1_CP_STEP(24, 6)
#define F1_CP_NEXT "add.u32 tq, tq, 32;\n\tadd.u32 qa, qa, %4;\n\t" F1_CP_PANEL
#define F1_CP_HEAD "{\n\t.reg .b32 tq, qa, ta, al;\n\t.reg .b64 a;\n\t.reg .pred e;\n\t"                      \
                   "elect.sync _|e, 0xffffffff;\n\tmov.b32 tq, %0;\n\tmov.b32 qa, %1;\n\t" F1_CP_PANEL
#define F1_CP_TAIL "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%3];\n\t}"
template <int NP, uint32_t QOFF>
__device__ __forceinline__ void copy_q_commit_elect(uint32_t t_q, uint32_t q_lo, uint32_t hi, uint32_t bar)
{
    static_assert(NP == 2 || NP == 4, "64-column panels of D");
    if constexpr (NP == 2)
        asm volatile(F1_CP_HEAD F1_CP_NEXT F1_CP_TAIL ::"r"(t_q), "r"(q_lo), "r"(hi), "r"(bar), "n"(QOFF) : "memory");
    else
        asm volatile(F1_CP_HEAD F1_CP_NEXT F1_CP_NEXT F1_CP_NEXT F1_CP_TAIL ::"r"(t_q), "r"(q_lo), "r"(hi), "r"(bar),
                     "n"(QOFF) : "memory");
}
#undef F1_CP_STEP
#undef F1_CP_PANEL
#undef F1_CP_NEXT
#undef F1_CP_HEAD
#undef F1_CP_TAIL

// S = Q K^T with A = Q from tensor memory (8 columns per 16-column K-step, 32 per panel) and B = K
// from shared memory, then the two commits (S ready; the K slot released), behind one elect.sync.
#define F1_T_STEP(TOFF, BOFF) "add.u32 ta, qa, " #TOFF ";\n\tadd.u32 bl, ka, " #BOFF ";\n\t"                  \
                              "mov.b64 b, {bl, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, t;\n\t"
#define F1_T_PANEL(ACC) "mov.b64 b, {ka, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [qa], b, %4, " #ACC ";\n\t" \
                        F1_T_STEP(8, 2) F1_T_STEP(16, 4) F1_T_STEP(24, 6)
#define F1_T_NEXT "add.u32 qa, qa, 32;\n\tadd.u32 ka, ka, %7;\n\t" F1_T_PANEL(t)
#define F1_T_HEAD "{\n\t.reg .b32 qa, ka, ta, bl;\n\t.reg .b64 b;\n\t.reg .pred e, f, t;\n\t"                  \
                  "setp.eq.b32 t, 0, 0;\n\tsetp.ne.b32 f, 0, 0;\n\telect.sync _|e, 0xffffffff;\n\t"              \
                  "mov.b32 qa, %1;\n\tmov.b32 ka, %2;\n\t" F1_T_PANEL(f)
#define F1_T_TAIL "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"            \
                  "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
template <int NP, uint32_t KOFF>
__device__ __forceinline__ void mma_s_tq_commit2_elect(uint32_t d_tmem, uint32_t t_q, uint32_t b_lo, uint32_t hi,
                                                       uint32_t idesc, uint32_t bar1, uint32_t bar2)
{
    static_assert(NP == 2 || NP == 4, "64-column panels of D");
    if constexpr (NP == 2)
        asm volatile(F1_T_HEAD F1_T_NEXT F1_T_TAIL ::"r"(d_tmem), "r"(t_q), "r"(b_lo), "r"(hi), "r"(idesc),
                     "r"(bar1), "r"(bar2), "n"(KOFF) : "memory");
    else
        asm volatile(F1_T_HEAD F1_T_NEXT F1_T_NEXT F1_T_NEXT F1_T_TAIL ::"r"(d_tmem), "r"(t_q), "r"(b_lo), "r"(hi),
                     "r"(idesc), "r"(bar1), "r"(bar2), "n"(KOFF) : "memory");
}
#undef F1_T_STEP
#undef F1_T_PANEL
#undef F1_T_NEXT
#undef F1_T_HEAD
#undef F1_T_TAIL

// O += P V over 64 keys (four 16-key steps, as mma_ts_mn4_elect) followed by two commits from
// the same elected lane (P V done; the V slot released).
__device__ __forceinline__ void mma_pv_commit2_elect(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                                     uint32_t idesc, uint32_t accumulate, uint32_t bar1, uint32_t bar2)
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
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate), "r"(bar1), "r"(bar2)
                 : "memory");
}

// One work unit, decoded identically by every role (the schedule is in schedule.h).
using Unit = TileUnit;

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

template <bool CAUSAL, int BN>
__device__ __forceinline__ bool unit_at(const Params &p, int round, Unit &u)
{
    return tile_unit<CAUSAL, BN>(p, gridDim.x, blockIdx.x, round, u);
}

// At D = 64 a CTA needs 192 tensor-memory columns (a 256-column allocation) and ~74 KB of shared
// memory, so two CTAs share an SM; the launch then gives every query tile its own CTA.
template <int D>
constexpr int kMinBlocks = (D == 64) ? 2 : 1;

template <int D, int KEYS, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, kMinBlocks<D>)
    fa_fwd1_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p)
{
    using C = Cfg<D, KEYS>;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t sQ = sb + C::OFF_Q, sRing = sb + C::OFF_RING, bar0 = sb + C::OFF_BAR;
    auto bar_q = [&](int i) { return bar0 + 8u * i; };
    auto bar_qfree = [&](int i) { return bar0 + 8u * (C::NQ + i); };
    auto bar_full = [&](int s) { return bar0 + 8u * (2 * C::NQ + s); };
    auto bar_empty = [&](int s) { return bar0 + 8u * (2 * C::NQ + C::NS + s); };
    const uint32_t barS = bar0 + 8u * (2 * C::NQ + 2 * C::NS);   // + 8 * buffer
    // Key step g signals S ready, P written and P V done on barS / barP / barPV + 8 * (g & 1),
    // phase (g / 2) & 1.  The softmax publishes P(g + 1) without waiting for P V(g), so it may
    // run one step ahead of the MMA warp's wait for P(g), and a waiter for P V(g) may have
    // skipped steps; with two barriers per event neither ever meets a barrier two phases past
    // the one it waits for (S(g + 2), P(g + 2) and P V(g + 2) all follow the MMA warp's wait
    // for P(g), which follows the softmax's wait for S(g)).
    const uint32_t barP = barS + 16u, barPV = barS + 32u, barDone = barS + 48u;
    // With staged output (C::STAGE_O) the one query buffer holds in turn the query tile of tile t
    // (until its copy into tensor memory completes: barQcp phase t) and the output rows of tile
    // t - 1 (staged by the softmax warps once Q(t) has been copied: barStaged + 8 * ((t - 1) & 1),
    // phase ((t - 1) / 2) & 1).  The Q producer writes those rows out with bulk tensor stores and,
    // once the stores have read them (barOread phase t - 1), loads Q(t + 1) into the buffer.  The
    // CTA's last tile has no next query copy to wait for: its epilogue waits for barOread of the
    // tile before it instead.  t counts the CTA's tiles that have keys.
    const uint32_t barQcp = barS + 56u, barStaged = barS + 64u, barOread = barS + 80u;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    unsigned int *status = &g_fa1_status;
    const uint64_t tmo = p.timeout_ns;

    if (pad + (uint32_t)C::BYTES > dynamic_smem_size_u32()) {
        if (threadIdx.x == 0) atomicOr(status, 1u | (S_SMEM << 8));
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(bar_q(i), 1);
            mbar_init(bar_qfree(i), 1);
        }
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(barS, 1);
        mbar_init(barS + 8, 1);
        mbar_init(barP, 4);
        mbar_init(barP + 8, 4);
        mbar_init(barPV, 1);
        mbar_init(barPV + 8, 1);
        mbar_init(barDone, 1);
        mbar_init(barQcp, 1);
        mbar_init(barStaged, 4);
        mbar_init(barStaged + 8, 4);
        mbar_init(barOread, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ K/V producer (consumption order)
        if (lane == 0) {
            int use = 0;
            int skip = -1;   // fault injection: the first V tile is never loaded (bit 0: every CTA; bit 1: CTA 0)
            const bool inj = (p.inject & 1u) || ((p.inject & 2u) && blockIdx.x == 0);
            const uint64_t keep = l2_policy_evict_last();   // K/V tiles are read again by other tiles
            bool ok = true;
            auto load = [&](const CUtensorMap *m, int j, int zkv) {
                const int s = use % C::NS;
                if (!bounded_wait(bar_empty(s), ((use / C::NS) & 1) ^ 1, abort_flag, tmo, S_EMPTY, status))
                    return false;
                if (inj && m == &tmV && skip < 0) {
                    skip = use++;
                    return true;
                }
                mbar_arrive_expect_tx(bar_full(s), C::KVTILE);
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_3d_hint(sRing + s * C::KVTILE + pn * C::KVPANEL, m, pn * 64, j * BN, zkv, bar_full(s),
                                     keep);
                ++use;
                return true;
            };
            Unit u;
            for (int round = 0; ok && unit_at<CAUSAL, C::BN>(p, round, u); ++round) {
                if (u.nk == 0) continue;
                ok = load(&tmK, 0, u.zkv);
                for (int j = 0; j < u.nk && ok; ++j) {
                    if (j + 1 < u.nk) ok = load(&tmK, j + 1, u.zkv);
                    if (ok) ok = load(&tmV, j, u.zkv);
                }
            }
            for (int x = max(0, use - C::NS); x < use; ++x)
                if (x != skip)
                    bounded_wait(bar_full(x % C::NS), (x / C::NS) & 1, abort_flag, tmo, S_DRAIN, status, false);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ Q producer
        if (lane == 0) {
            int tau = 0;
            const uint64_t once = l2_policy_evict_first();   // each query tile is read once
            bool ok = true;
            // staged output (C::STAGE_O): tile index and head plane of the last two tiles, whose
            // rows this thread writes out once their epilogues have staged them
            int pend_t0 = 0, pend_z0 = 0, pend_t1 = 0, pend_z1 = 0;
            auto store_o = [&](int k) {
                if (!bounded_wait(barStaged + 8u * (k & 1), (k >> 1) & 1, abort_flag, tmo, S_STAGED, status))
                    return false;
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_store_3d(&tmO, pn * 64, ((k & 1) ? pend_t1 : pend_t0) * BM, (k & 1) ? pend_z1 : pend_z0,
                                 sQ + pn * C::QPANEL);
                tma_store_commit();
                tma_store_wait_read();   // the buffer may take the next query tile, or the last tile's rows
                mbar_arrive(barOread);
                return true;
            };
            Unit u;
            for (int round = 0; ok && unit_at<CAUSAL, C::BN>(p, round, u); ++round) {
                if (u.nk == 0) continue;
                const int buf = tau % C::NQ;
                if constexpr (C::STAGE_O) {
                    // Q(1) once Q(0) is in tensor memory; Q(t) for t >= 2 once the rows of tile
                    // t - 2, staged in the buffer, have been read by their bulk stores
                    if (tau == 1 && !bounded_wait(barQcp, 0, abort_flag, tmo, S_QFREE, status)) break;
                    if (tau >= 2 && !store_o(tau - 2)) break;
                } else if (tau >= C::NQ &&
                           !bounded_wait(bar_qfree(buf), ((tau / C::NQ) - 1) & 1, abort_flag, tmo, S_QFREE, status)) {
                    break;
                }
                mbar_arrive_expect_tx(bar_q(buf), C::QTILE);
                // scale == 0: every score is 0, so load Q from a plane past the end of the
                // tensor, which the copy engine fills with zeros
                const int zq = p.smode == 2 ? p.B * p.Hq : u.zq;
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_3d_hint(sQ + buf * C::QTILE + pn * C::QPANEL, &tmQ, pn * 64, u.t * BM, zq, bar_q(buf),
                                     once);
                if (tau & 1) {
                    pend_t1 = u.t;
                    pend_z1 = u.zq;
                } else {
                    pend_t0 = u.t;
                    pend_z0 = u.zq;
                }
                ++tau;
            }
            if constexpr (C::STAGE_O) {
                // the last two tiles' rows
                for (int k = max(0, tau - 2); ok && k < tau; ++k) ok = store_o(k);
                tma_store_wait_all();   // every output store has landed before the CTA exits
            }
            for (int x = max(0, tau - C::NQ); x < tau; ++x)
                bounded_wait(bar_q(x % C::NQ), (x / C::NQ) & 1, abort_flag, tmo, S_DRAIN, status, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (whole warp)
        const uint32_t idS = idesc_f16(BF16, BM, BN, false) | (p.smode == 1 ? kNegateA : 0u);
        constexpr uint32_t idPV = idesc_f16(BF16, BM, D, true);
        constexpr uint32_t HI = sdesc_hi_sw128(1024);
        auto wait_u = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
            if (mbar_try_wait_all(bar, parity)) return true;   // the usual case: already complete
            return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_flag, tmo, site, status)) != 0;
        };
        // S = Q K^T over D (both K-major, 16 columns of D per instruction), then the commits for
        // S ready and the K slot released, all in one block
        auto issue_s_commit2 = [&](uint32_t dS, uint32_t sQt, uint32_t sK, uint32_t bar1, uint32_t bar2) {
            if constexpr (C::QT)
                mma_s_tq_commit2_elect<D / 64, (uint32_t)C::KVPANEL / 16>(dS, tmem + C::COL_Q, sdesc_lo(sK, 16), HI,
                                                                         idS, bar1, bar2);
            else
                mma_s_commit2_elect<D / 64, (uint32_t)C::QPANEL / 16, (uint32_t)C::KVPANEL / 16>(
                    dS, sdesc_lo(sQt, 16), sdesc_lo(sK, 16), HI, idS, bar1, bar2);
        };
        // O += P V over BN keys: A = P from TMEM, B = V (MN-major, 64-column panels C::KVPANEL
        // apart); one group of four 16-key steps per 64 keys, the last group followed by the
        // commits for P V done and the V slot released
        auto issue_pv_commit2 = [&](uint32_t tP, uint32_t sV, bool first, uint32_t bar1, uint32_t bar2) {
            const uint32_t vlo = sdesc_lo(sV, C::KVPANEL);
#pragma unroll
            for (int h = 0; h + 1 < BN / 64; ++h)
                mma_ts_mn4_elect(tmem + C::COL_O, tP + 32 * h, vlo + (uint32_t)((4 * h * 2048) >> 4), HI, idPV,
                                 (first && h == 0) ? 0u : 1u);
            constexpr int hl = BN / 64 - 1;
            mma_pv_commit2_elect(tmem + C::COL_O, tP + 32 * hl, vlo + (uint32_t)((4 * hl * 2048) >> 4), HI, idPV,
                                 (first && hl == 0) ? 0u : 1u, bar1, bar2);
        };
        auto tS = [&](uint32_t gs) { return tmem + ((gs & 1) ? C::COL_S1 : C::COL_S0); };
        int use = 0, tau = 0;
        uint32_t g = 0;   // global key step: S buffer and barS / barP / barPV barrier g % 2, phase (g / 2) & 1
        bool ok = true;
        Unit u;
        for (int round = 0; ok && unit_at<CAUSAL, C::BN>(p, round, u); ++round) {
            if (u.nk == 0) continue;
            const int buf = tau % C::NQ;
            ok = wait_u(bar_q(buf), (tau / C::NQ) & 1, S_Q);
            ++tau;
            const uint32_t sQt = sQ + buf * C::QTILE;
            if constexpr (C::QT) {
                // The previous tile's score MMAs, the only readers of the query columns, are done:
                // the softmax read their results before it published the last P waited for above.
                if (!ok) break;
                tc_fence_after();
                copy_q_commit_elect<D / 64, (uint32_t)C::QPANEL / 16>(tmem + C::COL_Q, sdesc_lo(sQt, 16), HI,
                                                                      C::STAGE_O ? barQcp : bar_qfree(buf));
            }
            if (ok) ok = wait_u(bar_full(use % C::NS), (use / C::NS) & 1, S_FULL);
            if (!ok) break;
            tc_fence_after();
            issue_s_commit2(tS(g), sQt, sRing + (use % C::NS) * C::KVTILE, barS + 8u * (g & 1), bar_empty(use % C::NS));
            if (!C::QT && u.nk == 1) tc_commit_elect(bar_qfree(buf));
            ++use;
            for (int j = 0; j < u.nk && ok; ++j) {
                const uint32_t gs = g + j;
                // K(j+1) and V(j) (the next two ring slots) are checked before S(j+1) is issued:
                // its issue blocks while the tensor pipe works through earlier MMAs, and only the
                // wait for P(j) then stands between it and P V(j)
                if (j + 1 < u.nk) {
                    ok = wait_u(bar_full(use % C::NS), (use / C::NS) & 1, S_FULL) &&
                         wait_u(bar_full((use + 1) % C::NS), ((use + 1) / C::NS) & 1, S_FULL);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s_commit2(tS(gs + 1), sQt, sRing + (use % C::NS) * C::KVTILE, barS + 8u * ((gs + 1) & 1),
                                    bar_empty(use % C::NS));
                    if (!C::QT && j + 2 == u.nk) tc_commit_elect(bar_qfree(buf));
                    ++use;
                } else {
                    ok = wait_u(bar_full(use % C::NS), (use / C::NS) & 1, S_FULL);
                }
                ok = ok && wait_u(barP + 8u * (gs & 1), (gs >> 1) & 1, S_P);
                if (!ok) break;
                tc_fence_after();
                issue_pv_commit2(tS(gs), sRing + (use % C::NS) * C::KVTILE, j == 0, barPV + 8u * (gs & 1),
                                 bar_empty(use % C::NS));
                ++use;
            }
            g += u.nk;
        }
        tc_commit_elect(barDone);
        bounded_wait(barDone, 0, abort_flag, tmo, S_DRAIN, status, false);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int r = threadIdx.x - 128;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tO = tmem + lane_off + C::COL_O;
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t g = 0;
        uint32_t tt = 0;   // tiles with keys finished by this CTA (barQcp, barStaged, bar_qfree phases)
        bool ok = true;
        Unit u;
        for (int round = 0; ok && unit_at<CAUSAL, C::BN>(p, round, u); ++round) {
            const int row = u.t * BM + r;
            uint8_t *orow = static_cast<uint8_t *>(p.o) + ((size_t)u.zq * p.Sq + row) * (size_t)(D * 2);
            if (u.nk == 0) {   // no allowed key for any row of this tile: o = 0, lse = -inf
                if (row < p.Sq) {
#pragma unroll 4
                    for (int c = 0; c < D * 2; c += 16) st_global_v4(orow + c, 0u, 0u, 0u, 0u);
                    p.lse[(size_t)u.zq * p.Sq + row] = -INFINITY;
                }
                continue;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < u.nk; ++j) {
                const uint32_t gs = g + j;
                const uint32_t tSb = tmem + lane_off + ((gs & 1) ? C::COL_S1 : C::COL_S0);
                ok = mbar_try_wait_all(barS + 8u * (gs & 1), (gs >> 1) & 1) ||
                     __all_sync(0xffffffffu, bounded_wait(barS + 8u * (gs & 1), (gs >> 1) & 1, abort_flag, tmo, S_S, status));
                if (!ok) break;
                tc_fence_after();
                // S in 32-column reducing loads: each also returns the maximum of its 32 scores
                uint32_t sv[BN];
                float pm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < BN; c += 32)
                    tmem_ld_red_max_x32(tSb + c, *reinterpret_cast<uint32_t(*)[32]>(sv + c), pm[c / 32]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BN; c += 32) reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(sv + c));
                reg_fence_f4(pm[0], pm[1], pm[2], pm[3]);
                float *s = reinterpret_cast<float *>(sv);
                const int kbase = j * BN;
                const bool tail = kbase + BN > p.Sk;
                const bool diag = CAUSAL && (kbase + BN - 1 > u.t * BM + p.coff);
                float mrow = fmaxf(fmax3(pm[0], pm[1], pm[2]), pm[3]);
                if (tail || diag) {   // masked steps: the row maximum over the masked scores
                    int lim = p.Sk - 1 - kbase;
                    if (CAUSAL) lim = min(lim, row + p.coff - kbase);
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c > lim) s[c] = -INFINITY;
                    // eight chains seeded with 16 scores, then rounds of 16 more
                    static_assert(BN % 16 == 0 && BN >= 32, "row-max chains cover the step exactly");
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
                    for (int c = 16; c + 16 <= BN; c += 16) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
                    }
                    mrow = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
                }
                const float m_new = fmaxf(m_used, mrow * sl2);
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_used = m_new;
                } else if (m_new - m_used > p.tau) {
                    alpha = ex2_approx(m_used - m_new);
                    l *= alpha;
                    m_used = m_new;
                    rescale = true;
                }
                const float msub = (m_used == -INFINITY) ? 0.f : m_used;
                const uint64_t negm2 = f2_pack(-msub, -msub);
                uint64_t lsum2[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) lsum2[i] = f2_pack(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = 32 * c + 2 * e;
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(s[i], s[i + 1]), sl2x2, negm2), t0, t1);
                        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                        lsum2[e & 7] = f2_add(lsum2[e & 7], f2_pack(p0, p1));
                        pk[e] = pack2<BF16>(p0, p1);
                    }
                    tmem_st_x16(tSb + 16 * c, pk);
                }
                // O may be rescaled only once P V(j-1) is complete; P(j) is published without
                // that wait otherwise, so that P V(j) can follow P V(j-1) directly.  (S(j) was
                // issued after P V(j-2), so the barrier of P V(j-1) is at most one phase behind.)
                if (__any_sync(0xffffffffu, rescale)) {   // only for j > 0
                    const uint32_t bpv = barPV + 8u * ((gs - 1) & 1), ppv = ((gs - 1) >> 1) & 1;
                    ok = mbar_try_wait_all(bpv, ppv) ||
                         __all_sync(0xffffffffu, bounded_wait(bpv, ppv, abort_flag, tmo, S_PV, status));
                    if (!ok) break;
                    {
                        tc_fence_after();
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
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(barP + 8u * (gs & 1));
                const uint64_t q0 = f2_add(f2_add(lsum2[0], lsum2[1]), f2_add(lsum2[2], lsum2[3]));
                const uint64_t q1 = f2_add(f2_add(lsum2[4], lsum2[5]), f2_add(lsum2[6], lsum2[7]));
                float la, lb;
                f2_unpack(f2_add(q0, q1), la, lb);
                l += la + lb;
            }
            if (!ok) break;
            // epilogue: the last P V of this tile, then O / l -> 16-bit rows, and the lse
            const uint32_t gl = g + u.nk - 1;
            ok = __all_sync(0xffffffffu, bounded_wait(barPV + 8u * (gl & 1), (gl >> 1) & 1, abort_flag, tmo, S_PV, status));
            if (!ok) break;
            g += u.nk;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const uint64_t il2 = f2_pack(inv_l, inv_l);
            if constexpr (C::STAGE_O) {
                // The query buffer takes this tile's rows once the next tile's query tile (when
                // this CTA has one) has been copied out of it into tensor memory.
                bool next = false;
                {
                    Unit v;
                    for (int rr = round + 1; !next && unit_at<CAUSAL, C::BN>(p, rr, v); ++rr) next = v.nk > 0;
                }
                if (next) {
                    ok = mbar_try_wait_all(barQcp, (tt + 1) & 1) ||
                         __all_sync(0xffffffffu, bounded_wait(barQcp, (tt + 1) & 1, abort_flag, tmo, S_QFREE, status));
                    if (!ok) break;
                } else if (tt >= 1) {
                    // the last tile: the previous tile's rows must have been read out of the buffer
                    ok = mbar_try_wait_all(barOread, (tt - 1) & 1) ||
                         __all_sync(0xffffffffu, bounded_wait(barOread, (tt - 1) & 1, abort_flag, tmo, S_QFREE, status));
                    if (!ok) break;
                }
            }
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t ov[32];
                tmem_ld_x32(tO + c, ov);
                tmem_wait_ld();
                reg_fence_x32(ov);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float lo, hi;
                    f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1])), il2), lo, hi);
                    pk[e] = pack2<BF16>(lo, hi);
                }
                if constexpr (C::STAGE_O) {
                    // row r of the 64-column panel c / 64, 128B-swizzled as the o tensor map expects
                    const uint32_t line = sQ + (uint32_t)(c / 64) * C::QPANEL + (uint32_t)r * 128u;
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
            if (row < p.Sq) {
                const float lse = l > 0.f ? (m_used + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
                p.lse[(size_t)u.zq * p.Sq + row] = lse;
            }
            if constexpr (C::STAGE_O) {
                // The rows leave by bulk tensor stores that the Q producer issues (rows >= Sq
                // clipped by the map), instead of 2*D-byte stores from every thread.  Each writer
                // makes its rows visible to the copy engine, then each warp arrives.
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_elect(barStaged + 8u * (tt & 1));
            }
            ++tt;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    } else if (warp >= 4 && *abort_flag) {
        // This CTA gave up on a wait: every row of every tile it was given gets NaN in o and lse
        // (all roles have stopped), so that none of them keeps a value that looks valid.
        const int r = threadIdx.x - 128;
        Unit u;
        for (int round = 0; unit_at<CAUSAL, C::BN>(p, round, u); ++round) poison_row<D>(p, u.zq, u.t * BM + r);
    }
}

template <int D, int KEYS, bool BF16, bool CAUSAL>
static cudaError_t launch_one(const Maps &m, const Params &p, cudaStream_t stream)
{
    auto kern = fa_fwd1_kernel<D, KEYS, BF16, CAUSAL>;
    static std::atomic<uint64_t> configured{0};
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, KEYS>::ALLOC);
        if (e != cudaSuccess) return e;
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sm_count[dev].store(nsm, std::memory_order_relaxed);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    Params q = p;
    if (q.timeout_ns == 0) q.timeout_ns = kDefaultTimeoutNs;
    // D = 64: one CTA per query tile (two resident per SM), issued heaviest first, so the block
    // scheduler balances the causal tiles of unequal length; otherwise one persistent CTA per SM.
    const int grid = (D == 64) ? p.num_units : min(p.num_units, max(1, sm_count[dev].load(std::memory_order_relaxed)));
    kern<<<grid, THREADS, Cfg<D, KEYS>::ALLOC, stream>>>(m.q, m.k, m.v, m.o, q);
    return cudaGetLastError();
}

} // namespace one

cudaError_t launch_fwd1(int D, int keys, bool bf16, bool causal, const Maps &m, const Params &p, cudaStream_t st)
{
#define F1_CASE(DD, KK, BB, CC) \
    if (D == DD && keys == KK && bf16 == BB && causal == CC) return one::launch_one<DD, KK, BB, CC>(m, p, st);
    F1_CASE(64, 64, true, false) F1_CASE(64, 64, true, true) F1_CASE(64, 64, false, false) F1_CASE(64, 64, false, true)
    F1_CASE(128, 64, true, false) F1_CASE(128, 64, true, true) F1_CASE(128, 64, false, false) F1_CASE(128, 64, false, true)
    F1_CASE(128, 128, true, false) F1_CASE(128, 128, true, true) F1_CASE(128, 128, false, false) F1_CASE(128, 128, false, true)
    F1_CASE(256, 64, true, false) F1_CASE(256, 64, true, true) F1_CASE(256, 64, false, false) F1_CASE(256, 64, false, true)
#undef F1_CASE
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_fa1_status(uint32_t *word)
{
    unsigned int w = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_fa1_status, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_fa1_status, &zero, sizeof(zero));
    if (word) *word = w;
    return e;
}

} // namespace fa
