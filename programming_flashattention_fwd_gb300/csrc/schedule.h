// schedule.h -- the static work schedule of the persistent attention kernels, shared by the
// device code (fa_fwd_sm103.cu, fa_fwd1_sm103.cu) and host-side checks of it.
//
// A launch has G persistent CTAs.  CTA c takes work unit g = round * G + c in even rounds and
// g = round * G + (G - 1 - c) in odd rounds (a snake order, so that a CTA that took a heavy unit
// in one round takes a light one in the next).  With the causal mask the units are ordered
// heaviest first (the query tiles nearest the end of the sequence need the most key tiles);
// without it consecutive units share a head, so that its K/V stays in L2 while they run.
// Query head hq reads KV head hq / (Hq / Hkv): consecutive query heads share a KV head.
#pragma once

#include "fa_internal.h"

namespace fa {

// The multiplier and shift of FastDiv for divisor d >= 1 (host side).
inline FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while (l < 31 && (1u << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return FastDiv{d, (uint32_t)m, l};
}

// n / d for 0 <= n < 2^31 (the sum below then stays under 2^32).
__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f)
{
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi(n, f.mul);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)n * f.mul) >> 32);
#endif
    return (hi + n) >> f.shr;
}

// Fills the schedule's divisors from B, Hq, group, Tq and NP (host side, before a launch).
inline void set_schedule_divisors(Params &p)
{
    p.f_nbh = make_fastdiv((uint32_t)(p.B * p.Hq));
    p.f_np = make_fastdiv((uint32_t)p.NP);
    p.f_tq = make_fastdiv((uint32_t)p.Tq);
    p.f_hq = make_fastdiv((uint32_t)p.Hq);
    p.f_group = make_fastdiv((uint32_t)p.group);
}

// Index of the work unit that CTA c takes in round `round` (past the last unit when the
// CTA has no more work).
__host__ __device__ __forceinline__ long long unit_index(int G, int c, int round)
{
    return (long long)round * G + ((round & 1) ? (G - 1 - c) : c);
}

// Key tiles of `bn` keys that the 128-row query tile t reads: every key tile without the
// mask; with it, up to the tile holding key (last row of the tile + coff), where a key j is
// allowed for query row i iff j <= i + coff; 0 when even the tile's last row has no key.
__host__ __device__ __forceinline__ int key_tiles(const Params &p, bool causal, int t, int bn)
{
    if (!causal) return p.Tk;
    const long long hi = (long long)t * kBM + (kBM - 1) + p.coff;
    if (hi < 0) return 0;
    const long long n = hi / bn + 1;
    return n < p.Tk ? (int)n : p.Tk;
}

// The two-tile kernel's unit: two 128-row query tiles of one (b, hq) sharing one K/V stream.
struct PairUnit {
    int zq, zkv;      // q/o head plane (b*Hq + hq) and k/v head plane (b*Hkv + kvh)
    int tA, tB;       // query tile indices
    bool hasB;
    int nA, nB, n;    // key tiles for tile a, tile b, and their maximum
};

// Units of the two-tile kernel: p.num_units = B * Hq * p.NP pairs (p.NP = ceil(Tq / 2)).
template <bool CAUSAL>
__host__ __device__ __forceinline__ bool pair_unit(const Params &p, int G, int c, int round, PairUnit &u)
{
    const long long g64 = unit_index(G, c, round);
    if (g64 >= p.num_units) return false;
    const uint32_t g = (uint32_t)g64;   // below num_units < 2^31
    int bh, pr;
    if (CAUSAL) {   // heaviest query-tile pairs first
        const uint32_t q = fdiv(g, p.f_nbh);
        pr = p.NP - 1 - (int)q;
        bh = (int)(g - q * p.f_nbh.d);
    } else {        // consecutive units share a head (and its K/V in L2)
        const uint32_t q = fdiv(g, p.f_np);
        bh = (int)q;
        pr = (int)(g - q * p.f_np.d);
    }
    const int b = (int)fdiv((uint32_t)bh, p.f_hq), hq = bh - b * p.Hq;
    u.zq = bh;
    u.zkv = b * p.Hkv + (int)fdiv((uint32_t)hq, p.f_group);
    u.tA = 2 * pr;
    u.tB = 2 * pr + 1;
    u.hasB = u.tB < p.Tq;
    u.nA = key_tiles(p, CAUSAL, u.tA, kBN);
    u.nB = u.hasB ? key_tiles(p, CAUSAL, u.tB, kBN) : 0;
    u.n = u.nA > u.nB ? u.nA : u.nB;
    return true;
}

// The one-tile kernel's unit: one 128-row query tile read against key tiles of BN keys.
struct TileUnit {
    int zq, zkv, t, nk;
};

// Units of the one-tile kernel: p.num_units = B * Hq * Tq.
template <bool CAUSAL, int BN>
__host__ __device__ __forceinline__ bool tile_unit(const Params &p, int G, int c, int round, TileUnit &u)
{
    const long long g64 = unit_index(G, c, round);
    if (g64 >= p.num_units) return false;
    const uint32_t g = (uint32_t)g64;   // below num_units < 2^31
    int bh, t;
    if (CAUSAL) {   // heaviest query tiles first
        const uint32_t q = fdiv(g, p.f_nbh);
        t = p.Tq - 1 - (int)q;
        bh = (int)(g - q * p.f_nbh.d);
    } else {
        const uint32_t q = fdiv(g, p.f_tq);
        bh = (int)q;
        t = (int)(g - q * p.f_tq.d);
    }
    const int b = (int)fdiv((uint32_t)bh, p.f_hq), hq = bh - b * p.Hq;
    u.zq = bh;
    u.zkv = b * p.Hkv + (int)fdiv((uint32_t)hq, p.f_group);
    u.t = t;
    u.nk = key_tiles(p, CAUSAL, t, BN);
    return true;
}

} // namespace fa
