// schedule_check.cpp -- host-side check of the persistent attention kernels' work schedule
// (schedule.h), built and run by tests/test_schedule_cpu.py.
//
// For each shape, mask and grid size it walks every CTA's rounds exactly as the kernels do
// and checks that every (batch, query head, 128-row query tile) is visited exactly once, that
// each unit reads the KV head its query head maps to, that the key tiles a query tile reads
// cover every key any of its rows may attend to and at most one key tile more (only a ragged
// last query tile can over-reach, by its padding rows), and that every TMA coordinate the
// kernels derive from a unit lies inside the tensors.  Prints "ok" or the first failure.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "schedule.h"

using fa::Params;

namespace {

int fails = 0;

void fail(const char *what, int B, int Hq, int Hkv, int Sq, int Sk, int causal, int G)
{
    if (fails++ < 20)
        std::printf("FAIL %s: B=%d Hq=%d Hkv=%d Sq=%d Sk=%d causal=%d G=%d\n", what, B, Hq, Hkv, Sq, Sk, causal, G);
}

// Key tiles of `bn` keys that the real rows of query tile t need, by brute force over rows.
int needed_key_tiles(int t, int Sq, int Sk, int causal, int bn)
{
    long long last = -1;
    for (int i = t * 128; i < Sq && i < t * 128 + 128; ++i) {
        long long hi = Sk - 1;
        if (causal == 1 && i < hi) hi = i;
        if (causal == 2 && i + (long long)Sk - Sq < hi) hi = i + (long long)Sk - Sq;
        if (hi > last) last = hi;
    }
    return last < 0 ? 0 : (int)(last / bn + 1);
}

Params make_params(int B, int Hq, int Hkv, int Sq, int Sk, int causal, int key_tile, bool pairs)
{
    Params p{};
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk;
    p.Tq = (Sq + 127) / 128;
    p.Tk = (Sk + key_tile - 1) / key_tile;
    p.NP = (p.Tq + 1) / 2;
    p.group = Hq / Hkv;
    p.num_units = pairs ? B * Hq * p.NP : B * Hq * p.Tq;
    p.coff = causal == 2 ? Sk - Sq : 0;
    fa::set_schedule_divisors(p);
    return p;
}

void check_tile(const Params &p, int zq, int zkv, int t, int nk, int bn, int causal, std::vector<int> &seen,
                int G)
{
    const int B = p.B, Hq = p.Hq, Hkv = p.Hkv, Sq = p.Sq, Sk = p.Sk;
    if (zq < 0 || zq >= B * Hq || t < 0 || t >= p.Tq) return fail("query tile out of range", B, Hq, Hkv, Sq, Sk, causal, G);
    ++seen[(size_t)zq * p.Tq + t];
    if (zkv != (zq / Hq) * Hkv + (zq % Hq) / (Hq / Hkv)) fail("wrong KV head", B, Hq, Hkv, Sq, Sk, causal, G);
    if (zkv < 0 || zkv >= B * Hkv) fail("KV plane out of range", B, Hq, Hkv, Sq, Sk, causal, G);
    const int need = needed_key_tiles(t, Sq, Sk, causal, bn);
    const bool last_tile = t == p.Tq - 1;
    if (nk < need) fail("a needed key tile is not read", B, Hq, Hkv, Sq, Sk, causal, G);
    if (nk > need + (last_tile ? 1 : 0)) fail("key tiles read past the mask", B, Hq, Hkv, Sq, Sk, causal, G);
    if (nk > p.Tk) fail("key tile past the end of k/v", B, Hq, Hkv, Sq, Sk, causal, G);
    // TMA boxes: key tile j covers keys [j*bn, j*bn + bn), its first key must exist
    if (nk > 0 && (long long)(nk - 1) * bn >= Sk) fail("key box starts past Sk", B, Hq, Hkv, Sq, Sk, causal, G);
}

template <bool CAUSAL>
void check_shape(int B, int Hq, int Hkv, int Sq, int Sk, int causal, int G)
{
    // two-tile kernel: pairs of query tiles, 128-key steps
    {
        const Params p = make_params(B, Hq, Hkv, Sq, Sk, causal, 128, true);
        std::vector<int> seen((size_t)B * Hq * p.Tq, 0);
        long long units = 0;
        for (int c = 0; c < G; ++c) {
            fa::PairUnit u;
            for (int r = 0; fa::pair_unit<CAUSAL>(p, G, c, r, u); ++r) {
                ++units;
                check_tile(p, u.zq, u.zkv, u.tA, u.nA, 128, causal, seen, G);
                if (u.hasB) check_tile(p, u.zq, u.zkv, u.tB, u.nB, 128, causal, seen, G);
                else if (u.tB < p.Tq) fail("tile b dropped", B, Hq, Hkv, Sq, Sk, causal, G);
                if (u.n != (u.nA > u.nB ? u.nA : u.nB)) fail("unit length", B, Hq, Hkv, Sq, Sk, causal, G);
            }
        }
        if (units != p.num_units) fail("pair units visited != num_units", B, Hq, Hkv, Sq, Sk, causal, G);
        for (int s : seen)
            if (s != 1) { fail("pair schedule: a query tile not visited exactly once", B, Hq, Hkv, Sq, Sk, causal, G); break; }
    }
    // one-tile kernel: 64- and 128-key steps
    for (int bn : {64, 128}) {
        const Params p = make_params(B, Hq, Hkv, Sq, Sk, causal, bn, false);
        std::vector<int> seen((size_t)B * Hq * p.Tq, 0);
        long long units = 0;
        for (int c = 0; c < G; ++c) {
            fa::TileUnit u;
            if (bn == 64) {
                for (int r = 0; fa::tile_unit<CAUSAL, 64>(p, G, c, r, u); ++r, ++units)
                    check_tile(p, u.zq, u.zkv, u.t, u.nk, 64, causal, seen, G);
            } else {
                for (int r = 0; fa::tile_unit<CAUSAL, 128>(p, G, c, r, u); ++r, ++units)
                    check_tile(p, u.zq, u.zkv, u.t, u.nk, 128, causal, seen, G);
            }
        }
        if (units != p.num_units) fail("tile units visited != num_units", B, Hq, Hkv, Sq, Sk, causal, G);
        for (int s : seen)
            if (s != 1) { fail("tile schedule: a query tile not visited exactly once", B, Hq, Hkv, Sq, Sk, causal, G); break; }
    }
}

// The launch's divisors (B*Hq, NP, Tq, Hq, Hq/Hkv) are applied as a multiply-high and a shift;
// check that against exact division: every divisor up to 4096 on a spread of numerators, and
// powers of two, their neighbours and large divisors near the 2^31 edge.
void check_fastdiv()
{
    std::vector<uint32_t> divs;
    for (uint32_t d = 1; d <= 4096; ++d) divs.push_back(d);
    for (int k = 12; k <= 30; ++k)
        for (int64_t e : {-1, 0, 1}) divs.push_back((uint32_t)((1ll << k) + e));
    for (uint32_t d : {100000u, 999983u, 65537u, 1u << 30, 0x7fffffffu}) divs.push_back(d);
    uint64_t x = 88172645463325252ull;   // xorshift64 for the random numerators
    for (uint32_t d : divs) {
        const fa::FastDiv f = fa::make_fastdiv(d);
        auto check = [&](uint32_t n) {
            if (n > 0x7fffffffu) return;
            if (fa::fdiv(n, f) != n / d && fails++ < 20) std::printf("FAIL fastdiv: %u / %u\n", n, d);
        };
        for (uint32_t n = 0; n < 2048; ++n) check(n);
        for (uint32_t k = 1; k < 64; ++k) {
            const uint64_t m = (uint64_t)d * k;
            if (m <= 0x80000000ull) { check((uint32_t)(m - 1)); check((uint32_t)m); check((uint32_t)(m + 1)); }
        }
        for (uint64_t k : {0x7fffffffull / d, 0x7fffffffull / d - 1}) {
            const uint64_t m = k * d;
            check((uint32_t)m); check((uint32_t)(m - 1 < m ? m - 1 : 0)); check((uint32_t)(m + d - 1));
        }
        check(0x7fffffffu);
        for (int i = 0; i < 256; ++i) {
            x ^= x << 13; x ^= x >> 7; x ^= x << 17;
            check((uint32_t)(x & 0x7fffffffu));
        }
    }
}

} // namespace

int main()
{
    check_fastdiv();
    const int seqs[] = {1, 17, 127, 128, 129, 255, 256, 257, 300, 513, 1000, 2000, 4096};
    const int heads[][2] = {{1, 1}, {2, 1}, {4, 2}, {8, 8}, {32, 8}, {6, 3}};
    const int grids[] = {1, 3, 152, 1000};
    long long cases = 0;
    for (int B : {1, 3})
        for (auto &h : heads)
            for (int Sq : seqs)
                for (int Sk : seqs)
                    for (int causal = 0; causal <= 2; ++causal)
                        for (int G : grids) {
                            if (causal == 0) check_shape<false>(B, h[0], h[1], Sq, Sk, causal, G);
                            else check_shape<true>(B, h[0], h[1], Sq, Sk, causal, G);
                            ++cases;
                        }
    if (fails) {
        std::printf("%d failures in %lld cases\n", fails, cases);
        return 1;
    }
    std::printf("ok %lld cases\n", cases);
    return 0;
}
