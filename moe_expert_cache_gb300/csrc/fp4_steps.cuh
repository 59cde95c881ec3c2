// Host-and-device scheduling arithmetic of the FP4 decode kernel
// (decode_fp4.cu): the order in which a CTA takes its ring items, and the
// split of each fill record into the CTAs' copy shares.  Kept free of device
// intrinsics so that a host compiler can build it for the schedule tests.
#pragma once

#include <cstddef>

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace fp4sched {

// Launch layout of the kernel.
constexpr int CW = 16;                // consumer warps
constexpr int CONS = CW * 32;
constexpr int FILL_WARPS = 1;         // fused cache fill (one TMA thread)
constexpr int THREADS = CONS + 32 + FILL_WARPS * 32;  // + producer warp + fill warps
constexpr int FPC = CW;               // features per phase-A chunk: one per consumer warp
constexpr int RW = 2;                 // W_d rows per warp pass in phase B
constexpr size_t HEAD = 256;          // ring barriers (and the fill ring's) at the start of shared memory
// Phase-A activations: f16 pairs in shared memory (X_SMEM) or in a global
// scratch row block written at the start of the launch (X_GLOBAL).
enum { X_SMEM = 0, X_GLOBAL = 1 };
constexpr size_t kSmemLimit4 = 227 * 1024 - 256;  // dynamic shared memory; the rest is static

// Shared-memory plan of one launch of T tokens: where x lives, the phase-B
// token group, ring slots and their bytes, fill ring chunks and their bytes,
// and the bytes ahead of the ring.
struct Fp4Plan {
    int xm, tg, nst, nf;
    size_t head, slot, fch;
};

// The plan with x placed as xm, or false when two ring slots do not fit.
inline bool fp4_plan_x(int H, int F, int T, int k, int SB, int G, int xm, Fp4Plan& pl) {
    const int RMAX = (H + G - 1) / G;
    const size_t TK = (size_t)T * k;
    pl.xm = xm;
    const size_t xbytes = pl.xm == X_SMEM ? (size_t)T * H * 2 : 0;
    const size_t head0 = HEAD + ((xbytes + 127) & ~(size_t)127) + ((TK * RMAX * 4 + 127) & ~(size_t)127);
    const size_t chunk = (size_t)2 * FPC * (H / 2 + H / SB);
    const size_t wpart = ((size_t)RMAX * (F / 2 + F / SB) + 127) & ~(size_t)127;
    // The fill ring is kept small (3 x 4 KiB per SM): host reads queued beyond
    // the link's bandwidth-delay product delay every SM's HBM reads.
    pl.fch = 4096;
    // token group of phase B: the most h rows (at most 16) whose staging in a
    // slot (fp32 as copied, then f16 pairs and their block factors) leaves room
    // for two slots
    int tg = T < 16 ? T : 16;
    for (; tg >= 1; --tg) {
        pl.head = head0 + (((6 * TK + 1 + (size_t)T) * 4 + 127) & ~(size_t)127);
        pl.slot = wpart + (size_t)tg * F * 6 + (size_t)tg * (F / 16) * 4;
        if (pl.slot < chunk) pl.slot = chunk;
        pl.slot = (pl.slot + 127) & ~(size_t)127;
        if (pl.head + 2 * pl.fch + 2 * pl.slot <= kSmemLimit4) break;
    }
    if (tg < 1) return false;
    pl.tg = tg;
    pl.nst = (int)((kSmemLimit4 - pl.head - 2 * pl.fch) / pl.slot);
    if (pl.nst > 4) pl.nst = 4;
    pl.nf = (int)((kSmemLimit4 - pl.head - pl.slot * pl.nst) / pl.fch);
    if (pl.nf > 3) pl.nf = 3;
    return true;
}

// x in shared memory when T*H*2 bytes fit there (at most 32 KiB) and still
// leave room for two slots; else x in the global block (always allocated for
// FP4 contexts), whose plan only shrinks as T falls, so a context whose T_max
// has a plan has one for every T up to it.
inline bool fp4_plan(int H, int F, int T, int k, int SB, int G, Fp4Plan& pl) {
    if ((size_t)T * H * 2 <= 32768 && fp4_plan_x(H, F, T, k, SB, G, X_SMEM, pl)) return true;
    return fp4_plan_x(H, F, T, k, SB, G, X_GLOBAL, pl);
}

// The steps of CTA c, in the order its producer issues them and its
// consumers take them: the phase-A items of the resident entries (a = c,
// c + G, ...), a seal, their phase-B items (entry, group of <= TG tokens),
// then for each fill in turn its phase-A items, a seal and its phase-B items.
// At a seal the consumers count the CTA in the group's counter (every CTA's
// h of the group is written once it holds G); a seal takes no ring slot.  A
// phase-B item waits for its group's count, each group's phase-A items come
// before its seal on every CTA, and the groups are taken in the same order
// everywhere: no wait can close a cycle.
enum { STEP_A = 0, STEP_SEAL = 1, STEP_B = 2 };
struct Steps {
    int c, G, cpe, nA, nfill, R, TG;
    const int* m_off;
    int grp, eb, ee, a, e, g0;
    bool inB;
    __host__ __device__ void open(int g) {  // group 0: the resident entries; group 1 + r: fill r
        grp = g;
        eb = g == 0 ? 0 : nA + g - 1;
        ee = g == 0 ? nA : eb + 1;
        int m = (int)(((long long)c - (long long)eb * cpe) % G);
        if (m < 0) m += G;
        a = eb * cpe + m;
        inB = false;
    }
    // The next step (false past the last): its kind, its entry (for a seal:
    // the group), and the phase-A item index or the first token of the
    // phase-B group.
    __host__ __device__ bool next(int& kind, int& ent, int& item, int& g) {
        for (;;) {
            if (grp > nfill) return false;
            if (!inB) {
                if (a < ee * cpe) {
                    kind = STEP_A;
                    ent = a / cpe;
                    item = a;
                    a += G;
                    return true;
                }
                inB = true;
                e = eb;
                g0 = 0;
                kind = STEP_SEAL;
                ent = grp;
                return true;
            }
            if (R > 0 && e < ee) {
                kind = STEP_B;
                ent = e;
                g = g0;
                g0 += TG;
                if (g0 >= m_off[e + 1] - m_off[e]) {
                    g0 = 0;
                    ++e;
                }
                return true;
            }
            open(grp + 1);
        }
    }
};

// A fill record copied in two parts (part 0: the W_gu values and scales,
// part 1: the W_d values and scales), each part two byte ranges of the
// record taken as one run.
struct FillParts {
    unsigned long long off[2][2];  // [part][range] record offsets
    unsigned long long len[2][2];  // [part][range] bytes (multiples of 16)
};

// The parts of an FP4 record of H x F experts with SB values per scale
// (record layout [W_gu values][W_d values][W_gu scales][W_d scales]).
__host__ __device__ inline FillParts fp4_fill_parts(int H, int F, int SB) {
    const unsigned long long VGU = (unsigned long long)F * H, VD = (unsigned long long)H * F / 2;
    const unsigned long long SGU = 2ull * F * H / SB, SD = (unsigned long long)H * F / SB;
    FillParts fp;
    fp.off[0][0] = 0;
    fp.len[0][0] = VGU;        // W_gu values
    fp.off[0][1] = VGU + VD;
    fp.len[0][1] = SGU;        // W_gu scales
    fp.off[1][0] = VGU;
    fp.len[1][0] = VD;         // W_d values
    fp.off[1][1] = VGU + VD + SGU;
    fp.len[1][1] = SD;         // W_d scales
    return fp;
}

// CTA c's share [b0, b1) of a run of L bytes split into G equal shares of a
// multiple of 16 bytes (the last ones shorter or empty).
__host__ __device__ inline void fill_share(unsigned long long L, int G, int c, unsigned long long& b0,
                                           unsigned long long& b1) {
    const unsigned long long per = ((L / 16 + G - 1) / G) * 16;
    const unsigned long long s = per * (unsigned long long)c;
    b0 = s < L ? s : L;
    b1 = s + per < L ? s + per : L;
}

// The chunk at offset o of a share of part pt ending at b1: its bytes (at
// most fch, not crossing the boundary between the part's two ranges) and its
// offset in the record (*at).
__host__ __device__ inline unsigned fill_chunk(const FillParts& fp, int pt, unsigned long long o,
                                               unsigned long long b1, unsigned fch, unsigned long long& at) {
    const unsigned long long la = fp.len[pt][0];
    unsigned long long end = b1;
    if (o < la && la < end) end = la;
    at = o < la ? fp.off[pt][0] + o : fp.off[pt][1] + (o - la);
    return (unsigned)(end - o < fch ? end - o : fch);
}

}  // namespace fp4sched
