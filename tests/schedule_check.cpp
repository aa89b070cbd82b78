// schedule_check.cpp -- host-side check of the persistent attention kernels' work schedule
// (schedule.h), built and run by tests/test_schedule_cpu.py.
//
// For each shape, mask and grid size it walks every CTA's rounds exactly as the kernels do
// and checks that every (batch, query head, 128-row query tile) is visited exactly once, that
// each unit reads the KV head its query head maps to, that the key tiles a query tile reads
// cover every key any of its rows may attend to and at most one key tile more (only a ragged
// last query tile can over-reach, by its padding rows), and that every TMA coordinate the
// kernels derive from a unit lies inside the tensors.  Prints "ok" or the first failure.
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

} // namespace

int main()
{
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
