// Host checks of the FP4 decode kernel's scheduling arithmetic, built from
// the kernel's own header (moe_expert_cache_gb300/csrc/fp4_steps.cuh):
//   * steps: every phase-A item of every entry is taken by exactly one CTA
//     (item a by CTA a mod G); each CTA seals each group once, after its
//     phase-A items of the group and before the group's phase-B items, in
//     group order; every (entry, token group) phase-B item is taken by every
//     CTA with output rows; and a simulation of the waits (a phase-B item
//     waits until every CTA has sealed its group) runs to completion;
//   * fill shares: the chunks of all CTAs' shares of both parts tile the
//     record exactly once, each 16-byte aligned, non-empty, at most the
//     chunk size and inside one range of its part;
//   * shared-memory plans, over every shape the FP4 formats accept (H, F up
//     to 8192), k up to 16 and T up to 256: each plan fits the dynamic
//     shared-memory limit with two ring slots and two fill chunks at least,
//     a slot holds a phase-A item and a phase-B item with its converted tail,
//     the head holds x (when in shared memory), the per-route outputs and the
//     worklist, and every T below a T that has a plan has one too (contexts
//     are accepted by their T_max).
// Exits 0 and prints "ok", or prints the first failure and exits 1.
#include "fp4_steps.cuh"

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <utility>
#include <vector>

using namespace fp4sched;

namespace {

[[noreturn]] void fail(const char* what, long long a, long long b) {
    std::printf("FAIL %s %lld %lld\n", what, a, b);
    std::exit(1);
}

struct Step { int kind, ent, item, g; };

unsigned rnd(unsigned& s) {
    s = s * 1664525u + 1013904223u;
    return s >> 8;
}

void check_steps(int H, int F, int G, int TG, int ugpu, int q, const std::vector<int>& ntok) {
    const int cpe = F / 16, nA = ugpu - q;
    std::vector<int> off(ugpu + 1, 0);
    for (int e = 0; e < ugpu; ++e) off[e + 1] = off[e] + ntok[e];
    std::vector<std::vector<Step>> seq(G);
    std::vector<int> owner((size_t)ugpu * cpe, -1);
    for (int c = 0; c < G; ++c) {
        const int R = (int)((long long)H * (c + 1) / G - (long long)H * c / G);
        Steps sq;
        sq.c = c; sq.G = G; sq.cpe = cpe; sq.nA = nA; sq.nfill = q; sq.R = R; sq.TG = TG;
        sq.m_off = off.data();
        sq.open(0);
        Step s;
        int guard = 0;
        while (sq.next(s.kind, s.ent, s.item, s.g)) {
            seq[c].push_back(s);
            if (++guard > 10000000) fail("runaway sequence", c, guard);
        }
        // group order, seal placement, item ownership
        int grp = 0;
        bool sealed = false;
        std::vector<std::vector<int>> bseen(ugpu);
        for (const Step& t : seq[c]) {
            const int tg = t.kind == STEP_SEAL ? t.ent : (t.ent < nA ? 0 : t.ent - nA + 1);
            if (tg < grp) fail("group order", c, tg);
            if (tg > grp) {
                if (!sealed) fail("group left unsealed", c, grp);
                grp = tg;
                sealed = false;
            }
            if (t.kind == STEP_SEAL) {
                if (sealed) fail("second seal", c, grp);
                sealed = true;
            } else if (t.kind == STEP_A) {
                if (sealed) fail("phase-A item after the seal", c, t.item);
                if (t.item / cpe != t.ent || t.item % G != c) fail("phase-A item", c, t.item);
                if (owner[t.item] >= 0) fail("phase-A item taken twice", c, t.item);
                owner[t.item] = c;
            } else {
                if (!sealed) fail("phase-B item before the seal", c, t.ent);
                if (R == 0) fail("phase-B item without rows", c, t.ent);
                bseen[t.ent].push_back(t.g);
            }
        }
        if (!sealed || grp != q) fail("groups not all sealed", c, grp);
        for (int e = 0; e < ugpu; ++e) {
            std::vector<int> want;
            if (R > 0)
                for (int g = 0; g < ntok[e]; g += TG) want.push_back(g);
            if (bseen[e] != want) fail("phase-B token groups", c, e);
        }
    }
    for (size_t i = 0; i < owner.size(); ++i)
        if (owner[i] < 0) fail("phase-A item not taken", (long long)i, 0);
    // the waits: a phase-B item of group g waits until every CTA has sealed g
    std::vector<size_t> pos(G, 0);
    std::vector<int> sealed_count(q + 1, 0);
    for (bool moved = true; moved;) {
        moved = false;
        for (int c = 0; c < G; ++c) {
            while (pos[c] < seq[c].size()) {
                const Step& t = seq[c][pos[c]];
                if (t.kind == STEP_B) {
                    const int g = t.ent < nA ? 0 : t.ent - nA + 1;
                    if (sealed_count[g] < G) break;
                }
                if (t.kind == STEP_SEAL) ++sealed_count[t.ent];
                ++pos[c];
                moved = true;
            }
        }
    }
    for (int c = 0; c < G; ++c)
        if (pos[c] != seq[c].size()) fail("waits do not complete", c, (long long)pos[c]);
}

void check_fill(int H, int F, int SB, int G, unsigned fch) {
    const FillParts fp = fp4_fill_parts(H, F, SB);
    const unsigned long long n = 3ull * H * F;
    const unsigned long long rb = n / 2 + n / SB;  // the record size of the format
    std::vector<std::pair<unsigned long long, unsigned>> got;
    for (int c = 0; c < G; ++c) {
        for (int pt = 0; pt < 2; ++pt) {
            const unsigned long long L = fp.len[pt][0] + fp.len[pt][1];
            unsigned long long b0, b1;
            fill_share(L, G, c, b0, b1);
            if (b0 % 16 || (b1 % 16 && b1 != L)) fail("share bounds", c, (long long)b0);
            for (unsigned long long o = b0; o < b1;) {
                unsigned long long at;
                const unsigned k = fill_chunk(fp, pt, o, b1, fch, at);
                if (k == 0 || k > fch || k % 16 || at % 16) fail("chunk", (long long)at, k);
                const bool first = o < fp.len[pt][0];
                if (first != (o + k <= fp.len[pt][0]) && first) fail("chunk straddles the ranges", (long long)at, k);
                got.emplace_back(at, k);
                o += k;
            }
        }
    }
    std::sort(got.begin(), got.end());
    unsigned long long p = 0;
    for (const auto& g : got) {
        if (g.first != p) fail("record not tiled", (long long)g.first, (long long)p);
        p += g.second;
    }
    if (p != rb) fail("record size", (long long)p, (long long)rb);
}

void check_plans(int SB, int G) {
    for (int H = 256; H <= 8192; H += 256)
        for (int F = SB == 16 ? 256 : 512; F <= 8192; F += SB == 16 ? 256 : 512)
            for (int k : {1, 2, 4, 8, 16}) {
                bool gap = false;  // some T has had no plan
                for (int T = 1; T <= 256 && T * k <= 4096; ++T) {
                    Fp4Plan pl;
                    if (!fp4_plan(H, F, T, k, SB, G, pl)) {
                        gap = true;
                        continue;
                    }
                    if (gap) fail("plan after a T without one", H * 100000 + F, T);
                    const size_t RMAX = (size_t)(H + G - 1) / G, TK = (size_t)T * k;
                    auto r128 = [](size_t v) { return (v + 127) & ~(size_t)127; };
                    const size_t need_head = HEAD + (pl.xm == X_SMEM ? r128((size_t)T * H * 2) : 0) +
                                             r128(TK * RMAX * 4) + r128((6 * TK + 1 + T) * 4);
                    const size_t wpart = r128(RMAX * (F / 2 + F / SB));
                    const size_t need_b = wpart + (size_t)pl.tg * F * 4 + (size_t)pl.tg * F * 2 +
                                          (size_t)pl.tg * (F / 16) * 4;
                    const size_t need_a = (size_t)2 * FPC * (H / 2 + H / SB);
                    if (pl.head + (size_t)pl.nst * pl.slot + (size_t)pl.nf * pl.fch > kSmemLimit4)
                        fail("plan exceeds shared memory", H * 100000 + F, T);
                    if (pl.nst < 2 || pl.nf < 2) fail("ring depth", pl.nst, pl.nf);
                    if (pl.slot < need_a || pl.slot < need_b) fail("slot too small", (long long)pl.slot, T);
                    if (pl.head < need_head) fail("head too small", (long long)pl.head, T);
                    if (pl.head % 128 || pl.slot % 128) fail("alignment", (long long)pl.head, (long long)pl.slot);
                    if (pl.tg < 1 || pl.tg > (T < 16 ? T : 16)) fail("token group", pl.tg, T);
                    if (pl.xm == X_SMEM && (size_t)T * H * 2 > 32768) fail("x in shared memory", H, T);
                }
            }
}

}  // namespace

int main() {
    for (int SB : {16, 32})
        for (int G : {152, 148}) check_plans(SB, G);
    // fill shares: NVFP4 (SB 16) and MXFP4 (SB 32) shapes the kernel accepts
    const int shapes[][3] = {{4096, 2048, 16}, {4096, 2048, 32}, {256, 256, 16}, {256, 512, 32},
                             {1024, 512, 16}, {2048, 768 + 256, 16}};
    for (const auto& s : shapes)
        for (int G : {152, 148, 132, 7, 1}) check_fill(s[0], s[1], s[2], G, 4096u);
    // steps: random worklists (resident entries first, then the fills)
    unsigned seed = 12345u;
    for (int trial = 0; trial < 400; ++trial) {
        const int H = 256 << (rnd(seed) % 5);          // 256 .. 4096
        const int F = 256 << (rnd(seed) % 4);          // 256 .. 2048
        const int Gs[] = {152, 148, 16, 3, 1};
        const int G = Gs[rnd(seed) % 5];
        const int TG = 1 + (int)(rnd(seed) % 16);
        const int ugpu = (int)(rnd(seed) % 13);
        const int q = ugpu ? (int)(rnd(seed) % (ugpu + 1)) : 0;
        std::vector<int> ntok(ugpu);
        for (int& t : ntok) t = 1 + (int)(rnd(seed) % 40);
        check_steps(H, F, G, TG, ugpu, q, ntok);
    }
    std::printf("ok\n");
    return 0;
}
