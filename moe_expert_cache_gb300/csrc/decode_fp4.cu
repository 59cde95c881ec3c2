// Decode expert FFN over FP4 records (W4A16): the same persistent,
// cooperatively launched streaming design as the BF16 kernel, reading packed
// e2m1 values and their block scales.  Two record formats share the code,
// selected by the scale block SB:
//   * NVFP4 (SB = 16): one e4m3 scale per 16 values, and a per-expert fp32
//     global.  deepmox "One logical expert, two physical levels of memory":
//     an NVFP4 bank stores packed four-bit values plus scale information;
//     small per-expert globals stay GPU-resident.
//   * MXFP4 (SB = 32, OCP Microscaling v1.0): one E8M0 scale, 2^(code-127),
//     per 32 values; no global (the kernel reads 1.0).  The same section
//     lists MXFP4 among the bank layouts.
// Weight w = e2m1 * scale(block along K) * global(expert).  Activations are
// not quantised to FP4 (W4A16); the arithmetic is packed f16:
//   * e2m1 codes are decoded two at a time, adjacent values, into f16 pairs
//     by the hardware pair conversion (exact);
//   * activation rows (x for phase A, h for phase B) are held as f16 pairs in
//     the same order, each token row multiplied by a power of two chosen from
//     its largest magnitude (exact for x; one f16 rounding for h), so that a
//     product is below 6 * 2^10 and eight of them below 2^16;
//   * each 16-value block is summed with packed f16 FMAs (two chains of four
//     products per half), widened to fp32, multiplied by its block scale and
//     added in fp32; the row total is rescaled once by the row's power of two
//     and the expert's global.
// x rows are scaled per token; h per 16-value block, when phase B converts
// the staged rows, so no maximum is shared between CTAs (the block's factor
// multiplies its sum together with the weight block's scale).
//
// Record (per layer-expert): [W_gu values 2F x H/2 bytes, low nibble first,
// gate/up rows interleaved in groups of 16][W_d values H x F/2]
// [W_gu scales 2F x H/SB][W_d scales H x F/SB].
//
// Layout of the work: 16 consumer warps, one producer warp (TMA ring) and one
// fill warp (one thread) per CTA, one CTA per SM.  A phase-A item is 16
// features (16 gate rows, the 16 up rows and their scale rows, one warp per
// feature); CTA c takes the items c, c + G, ... of each group of entries.  A
// phase-B item is (entry, group of at most TG tokens): the CTA's W_d rows
// [r0, r1), the staged fp32 h rows and, in the slot's tail, those rows
// converted to f16 pairs, two W_d rows per warp pass; phase-B items
// alternate between the two halves of the consumer warps.  The CTA takes the
// resident entries' phase-A and phase-B items, then each fill's phase-A and
// phase-B items; when a group's phase-A items are done the CTA counts itself
// in the group's counter, and a phase-B item's h rows are copied once all G
// CTAs have.  The producer and the fill thread start at the launch's entry,
// while the consumers stage the worklist and x: x goes into shared memory
// when T*H*2 bytes fit, else into a global block behind a grid barrier.
// Fills the control pass left pending are copied by this launch: the fill
// thread of every CTA copies its equal share of each fill record in turn,
// the W_gu values and scales first, then W_d (host pool -> shared ring ->
// victim slot by bulk copies), counting itself after each part; a fill's
// phase-A items wait for every CTA's W_gu share, its phase-B items for the
// whole record and every CTA's count of the fill's group, so the resident
// entries' two phases run while the fills stream and a fill's phase A runs
// while its W_d streams.
#include "ft_common.cuh"
#include "fp4_steps.cuh"
#include "../../include/ft.h"

using namespace fp4sched;

namespace {

constexpr int kXTarget = 9;  // token rows are scaled so their largest magnitude is in [2^9, 2^10)

// Scale bytes: two e4m3 codes (low byte first) to a float pair, by the
// hardware conversion (one per 16 values).
__device__ __forceinline__ float2 e4m3x2_f32(const uint8_t* p2) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(*reinterpret_cast<const unsigned short*>(p2)));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Scales of the 32 values of 16-byte group v of a row whose scale bytes
// start at `srow`: two e4m3 codes (NVFP4) or one E8M0 code used for both
// halves (MXFP4).  E8M0 is placed as an IEEE single bit pattern: code c is
// the exponent field; codes 0 and 255 also set the top mantissa bit, which
// makes code 0 the subnormal 2^-127 and code 255 a NaN.  (t - 1) >> 9 has
// that bit set exactly when t = (c + 1) & 0xFE is 0, i.e. c is 0 or 255.
__device__ __forceinline__ float e8m0_f32(uint32_t c) {
    const uint32_t t = (c + 1u) & 0xFEu;
    return __uint_as_float((c << 23) | (((t - 1u) >> 9) & 0x00400000u));
}

template <int SB>
__device__ __forceinline__ float2 scales32(const uint8_t* srow, int v) {
    if (SB == 16) return e4m3x2_f32(srow + 2 * v);
    const float s = e8m0_f32(srow[v]);
    return make_float2(s, s);
}

// The h rows phase B stages (fp32, shared memory) are swizzled so that a
// warp's loads of its lanes' 32-value groups spread over all banks: within
// group v (128 bytes), 16-byte chunk i is stored at chunk (i + v) mod 8.
__device__ __forceinline__ int swz_f32(int e) {  // element e of a row -> its stored position
    const int v = e >> 5, i = (e >> 2) & 7;
    return (v << 5) | (((i + v) & 7) << 2) | (e & 3);
}

// Phase-A activations as f16 pairs, in the order the weight decode produces:
// for word q of a row (values 8q..8q+7) one 16-byte chunk holds the pairs
// (x[8q+2J], x[8q+2J+1]), J = 0..3.  The four chunks of the 32-value group v
// are stored rotated by v/2 (chunk c at (c + v/2) mod 4), so that the eight
// lanes of a quarter warp (groups v = lane + 32i) read eight different bank
// quads.  Token row t is held multiplied by 2^a_t, with a_t chosen from the
// row's largest magnitude (kXTarget): every scaled value is an exact f16
// (a bf16 value below 2^10), a product with an e2m1 value (at most 6) is
// below 6 * 2^10, the eight products one f16 half of a 16-value block sums
// stay below 2^16, and values down to 2^-23 of the row's largest stay normal
// f16.  The row's factor 2^-a_t turns its sums back into dot products.
__device__ __forceinline__ int xpos(int q) {  // word q of a row -> its stored chunk
    const int v = q >> 2;
    return (v << 2) | (((q & 3) + (v >> 1)) & 3);
}

// The scale exponent a_t of a token row from its largest magnitude:
// kXTarget - floor(log2 amax), within [-100, 100] (2^a finite); 0 for a
// zero row, 100 for a row whose largest magnitude is subnormal.
__device__ __forceinline__ int x_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    if (amax < 1.17549435e-38f) return 100;
    const int a = kXTarget - ((int)((__float_as_uint(amax) >> 23) & 255u) - 127);
    return a < -100 ? -100 : (a > 100 ? 100 : a);
}

// 2^b for an exponent from x_exponent (|b| <= 100: a normal float).
__device__ __forceinline__ float pow2i(int b) { return __int_as_float((b + 127) << 23); }

// n arrivals on an mbarrier by one thread.
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(ft::smem_addr(bar)), "r"(n) : "memory");
}

// Eight bf16 values (one word's activations) times `up` as the chunk of
// four f16 pairs (x[2J], x[2J+1]).
__device__ __forceinline__ uint4 x_pairs(const uint4& raw, float up) {
    float f[8];
    ft::bf16x8_to_f32(raw, f);
    uint4 c;
    uint32_t* cw = reinterpret_cast<uint32_t*>(&c);
#pragma unroll
    for (int J = 0; J < 4; ++J) {
        const __half2 h = __floats2half2_rn(f[2 * J] * up, f[2 * J + 1] * up);
        cw[J] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return c;
}

// One warp converts token row `xr` (H bf16 values) into the paired layout
// at `dst` (H/8 chunks); returns the row factor 2^-a_t (all lanes).
__device__ __forceinline__ float stage_x_row(const uint4* xr, int H, uint4* dst, int lane) {
    float amax = 0.f;
    for (int q = lane; q < H / 8; q += 32) {
        float f[8];
        ft::bf16x8_to_f32(xr[q], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int a = x_exponent(amax);
    const float up = ldexpf(1.f, a);
    for (int q = lane; q < H / 8; q += 32) dst[xpos(q)] = x_pairs(xr[q], up);
    return ldexpf(1.f, -a);
}

// e2m1 decode, two adjacent values at a time: byte J of word w (values 2J
// in the low nibble, 2J+1 in the high nibble) becomes an f16 pair (low half
// = low nibble) by the hardware conversion, exact for every code.  The four
// pairs of one word, in J order:
__device__ __forceinline__ void e2m1_word_h2(uint32_t w, uint32_t* d) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(w));
}

__device__ __forceinline__ __half2 hfma2_u(uint32_t a, uint32_t b, __half2 c) {
    return __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b), c);
}

// 16 values (two words, decoded pairs d[0..7]) against their activation
// chunks x0, x1: the f16 sum of the 16 products, widened to fp32.  Two
// partial chains of four products per half.
__device__ __forceinline__ float dot16_h(const uint32_t* d, const uint4& x0, const uint4& x1) {
    const __half2 z = __float2half2_rn(0.f);
    __half2 p = hfma2_u(d[0], x0.x, z), q = hfma2_u(d[4], x1.x, z);
    p = hfma2_u(d[1], x0.y, p);
    q = hfma2_u(d[5], x1.y, q);
    p = hfma2_u(d[2], x0.z, p);
    q = hfma2_u(d[6], x1.z, q);
    p = hfma2_u(d[3], x0.w, p);
    q = hfma2_u(d[7], x1.w, q);
    const float2 f = __half22float2(__hadd2(p, q));
    return f.x + f.y;
}

// Phase A: gate and up rows of one feature against NT tokens; returns the
// row sums, in units of each token row's 2^a_t and without the
// expert's global, in ag / au.  `xs` is the paired activation block (H/8
// chunks per token row).
template <int NT, int XM, int SB>
__device__ __forceinline__ void gu_dots4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                         const uint4* xs, const int* tk, int H, int lane, float* ag, float* au) {
#pragma unroll
    for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
    const int nv = H >> 5;  // uint4 (32 values) per row
    const int rq = H >> 3;  // activation chunks per token row
    for (int v = lane; v < nv; v += 32) {
        const uint4 wg = gv[v], wu = uv[v];
        const float2 gsc = scales32<SB>(gs, v), usc = scales32<SB>(us, v);
        uint32_t dg[16], du[16];
        e2m1_word_h2(wg.x, dg);
        e2m1_word_h2(wg.y, dg + 4);
        e2m1_word_h2(wg.z, dg + 8);
        e2m1_word_h2(wg.w, dg + 12);
        e2m1_word_h2(wu.x, du);
        e2m1_word_h2(wu.y, du + 4);
        e2m1_word_h2(wu.z, du + 8);
        e2m1_word_h2(wu.w, du + 12);
        const int rot = (v >> 1) & 3;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint4* xr = xs + (size_t)tk[n] * rq + (size_t)v * 4;
            uint4 xc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) xc[c] = xr[(c + rot) & 3];
            ag[n] = fmaf(gsc.x, dot16_h(dg, xc[0], xc[1]), fmaf(gsc.y, dot16_h(dg + 8, xc[2], xc[3]), ag[n]));
            au[n] = fmaf(usc.x, dot16_h(du, xc[0], xc[1]), fmaf(usc.y, dot16_h(du + 8, xc[2], xc[3]), au[n]));
        }
    }
}

template <int NT, int XM, int SB>
__device__ __forceinline__ void gu_group4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                          const uint4* xs, const float* xf, int H, const int* m_tok, int off, int g0,
                                          int F, int f, int lane, float gsc, float* hbuf) {
    int tk[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) tk[n] = m_tok[off + g0 + n];
    float ag[NT], au[NT];
    gu_dots4<NT, XM, SB>(gv, uv, gs, us, xs, tk, H, lane, ag, au);
    float mine = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float rs = xf[tk[n]] * gsc;
        const float sg = ft::warp_sum(ag[n]) * rs;
        const float su = ft::warp_sum(au[n]) * rs;
        if (lane == n) mine = ft::silu_mul(sg, su);
    }
    // read only by phase B, as staged rows: swizzled for its fp32 loads
    if (lane < NT) hbuf[(size_t)(off + g0 + lane) * F + swz_f32(f)] = mine;
}

template <int XM, int SB>
__device__ __forceinline__ void gu_feature4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                            const uint4* xs, const float* xf, int H, const int* m_tok, int off,
                                            int ntok, int F, int f, int lane, float gsc, float* hbuf) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 2) {
            gu_group4<2, XM, SB>(gv, uv, gs, us, xs, xf, H, m_tok, off, g0, F, f, lane, gsc, hbuf);
            g0 += 2;
        } else {
            gu_group4<1, XM, SB>(gv, uv, gs, us, xs, xf, H, m_tok, off, g0, F, f, lane, gsc, hbuf);
            g0 += 1;
        }
    }
}

// Phase B: the W_d rows rb + WS*r (r < RW, row < R) of a slot (values +
// scales) against NT h rows held as scaled f16 pairs (the layout of the
// phase-A activations, F/8 chunks per row), each 16-value block of a row
// with its factor in hfb (F/16 per row).  Each h chunk is loaded once and
// applied to every row of the warp.
template <int NT, int SB, int WS>
__device__ __forceinline__ void down_group4(const uint8_t* wrows, const uint8_t* srows, unsigned dvrow,
                                            unsigned dsrow, const uint4* hp, const float* hfb, int g, int F,
                                            int lane, float gsc, float* o_s, int obase, int RMAX, int rb, int R) {
    float acc[RW][NT];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[r][n] = 0.f;
    const int nv = F >> 5;
    const int rq = F >> 3;
    for (int v = lane; v < nv; v += 32) {
        uint32_t d[RW][16];
        float2 sc[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int rl = rb + WS * r < R ? rb + WS * r : rb;  // rows past R repeat row rb (not stored)
            const uint4 w = reinterpret_cast<const uint4*>(wrows + (size_t)rl * dvrow)[v];
            sc[r] = scales32<SB>(srows + (size_t)rl * dsrow, v);
            e2m1_word_h2(w.x, d[r]);
            e2m1_word_h2(w.y, d[r] + 4);
            e2m1_word_h2(w.z, d[r] + 8);
            e2m1_word_h2(w.w, d[r] + 12);
        }
        const int rot = (v >> 1) & 3;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint4* hr = hp + (size_t)(g + n) * rq + (size_t)v * 4;
            uint4 hc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) hc[c] = hr[(c + rot) & 3];
            const float2 hb = *reinterpret_cast<const float2*>(hfb + (size_t)(g + n) * (F / 16) + 2 * v);
#pragma unroll
            for (int r = 0; r < RW; ++r)
                acc[r][n] = fmaf(sc[r].x * hb.x, dot16_h(d[r], hc[0], hc[1]),
                                 fmaf(sc[r].y * hb.y, dot16_h(d[r] + 8, hc[2], hc[3]), acc[r][n]));
        }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int rl = rb + WS * r;
        if (rl < R) {  // warp-uniform
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float sv = ft::warp_sum(acc[r][n]) * gsc;
                if (lane == 0) o_s[(size_t)(obase + g + n) * RMAX + rl] = sv;
            }
        }
    }
}

// The rows rb + WS*r (r < RW) of a slot against its ng h rows, two tokens
// at a time (WS: the warps sharing the item).
template <int SB, int WS>
__device__ __forceinline__ void down_rows4(const uint8_t* wrows, const uint8_t* srows, unsigned dvrow,
                                        unsigned dsrow, const uint4* hp, const float* hfb, int ng, int F, int lane,
                                        float gsc, float* o_s, int obase, int RMAX, int rb, int R) {
    int g = 0;
    while (g < ng) {
        if (ng - g >= 2) {
            down_group4<2, SB, WS>(wrows, srows, dvrow, dsrow, hp, hfb, g, F, lane, gsc, o_s, obase, RMAX, rb, R);
            g += 2;
        } else {
            down_group4<1, SB, WS>(wrows, srows, dvrow, dsrow, hp, hfb, g, F, lane, gsc, o_s, obase, RMAX, rb, R);
            g += 1;
        }
    }
}

// Eight fp32 values (h elements 8q..8q+7 of a staged row, swizzled as
// swz_f32) as the chunk of four f16 pairs (h[2J], h[2J+1]), scaled by the
// power of two that puts the largest magnitude of their 16-value block (this
// chunk and the one of lane ^ 1, which converts chunk q ^ 1 in the same
// step) in [2^9, 2^10); returns the block's factor 2^-b in *fb.
__device__ __forceinline__ uint4 h_pairs_block(const float* hr, int q, float* fb) {
    const float4 lo = *reinterpret_cast<const float4*>(hr + swz_f32(8 * q));
    const float4 hi = *reinterpret_cast<const float4*>(hr + swz_f32(8 * q + 4));
    float m = fmaxf(fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))),
                    fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const int b = x_exponent(m);
    const float up = pow2i(b);
    *fb = pow2i(-b);
    uint4 c;
    __half2 t;
    t = __floats2half2_rn(lo.x * up, lo.y * up); c.x = *reinterpret_cast<const uint32_t*>(&t);
    t = __floats2half2_rn(lo.z * up, lo.w * up); c.y = *reinterpret_cast<const uint32_t*>(&t);
    t = __floats2half2_rn(hi.x * up, hi.y * up); c.z = *reinterpret_cast<const uint32_t*>(&t);
    t = __floats2half2_rn(hi.z * up, hi.w * up); c.w = *reinterpret_cast<const uint32_t*>(&t);
    return c;
}

}  // namespace

namespace {


// Fused fill, run by ONE thread of CTA c (of G): each fill record is copied
// in two parts, each split into G equal 16-byte-aligned shares (CTA c takes
// share c) and sent host pool -> shared ring (bulk loads on mbarriers, up to
// nf in flight) -> victim slot (bulk stores): part 0 = the W_gu values and
// scales (the bytes the fill's phase-A items read), part 1 = the W_d values
// and scales.  A part is two byte ranges of the record taken as one run; a
// chunk never straddles them.  Once a part's share is stored (the stores
// complete, then the async-proxy writes are ordered before a GPU-scope
// release) the CTA counts itself: part 0 in the high half-word of cnt0[r],
// part 1 in ready[r].  Every wait is bounded.

__device__ __noinline__ void fill_parts_tma(const uint8_t* host, uint8_t* pool, unsigned long long rb, int q,
                                            const int* fslot, const int* ffid, unsigned* ready, unsigned* cnt0,
                                            int c, int G, const FillParts& fp, uint8_t* fring, uint64_t* fbar,
                                            unsigned fch, int nf, unsigned* err) {
    for (int s = 0; s < nf; ++s) ft::mbar_init(&fbar[s], 1);
    ft::mbar_fence_init();
    // CTA c's share [b0, b1) of part pt (offsets within the part's run)
    unsigned long long sb0[2], sb1[2];
    for (int pt = 0; pt < 2; ++pt) fill_share(fp.len[pt][0] + fp.len[pt][1], G, c, sb0[pt], sb1[pt]);
    struct Cur { int r, pt; unsigned long long o; };
    auto settle = [&](Cur& u) {  // onto a chunk, or r == q past the last
        while (u.r < q && u.o >= sb1[u.pt]) {
            if (++u.pt == 2) {
                u.pt = 0;
                ++u.r;
            }
            u.o = sb0[u.pt];
        }
    };
    // the chunk at u: record offset and bytes (not crossing the part's range boundary)
    auto chunk = [&](const Cur& u, unsigned long long& at, unsigned& n) {
        n = fill_chunk(fp, u.pt, u.o, sb1[u.pt], fch, at);
    };
    auto advance = [&](Cur& u) {
        unsigned long long at;
        unsigned n;
        chunk(u, at, n);
        u.o += n;
        settle(u);
    };
    // everything before cursor u is stored: count the parts it completes
    int done_parts = 0;  // parts (2 per fill, in order) counted so far
    auto publish = [&](const Cur& u) {
        const int upto = u.r * 2 + u.pt;
        if (done_parts >= upto) return;
        ft::bulk_wait_all();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        for (; done_parts < upto; ++done_parts) {
            const int r = done_parts >> 1;
            if ((done_parts & 1) == 0)
                atomicAdd(&cnt0[r], 1u << 16);
            else
                atomicAdd(&ready[r], 1u);
        }
    };
    Cur ui{0, 0, sb0[0]}, us{0, 0, sb0[0]};
    settle(ui);
    settle(us);
    publish(us);
    int issued = 0, done = 0;
    for (; ui.r < q && issued < nf; ++issued) {
        unsigned long long at;
        unsigned n;
        chunk(ui, at, n);
        ft::mbar_arrive_expect_tx(&fbar[issued], n);
        ft::bulk_g2s(fring + (size_t)issued * fch, host + (unsigned long long)ffid[ui.r] * rb + at, n, &fbar[issued]);
        advance(ui);
    }
    bool ok = true;
    while (us.r < q) {
        const int s = done % nf;
        if (!ft::mbar_wait(&fbar[s], (uint32_t)(done / nf) & 1u, err)) {
            ok = false;
            break;
        }
        unsigned long long at;
        unsigned n;
        chunk(us, at, n);
        ft::bulk_s2g(pool + (unsigned long long)fslot[us.r] * rb + at, fring + (size_t)s * fch, n);
        ft::bulk_commit();
        ft::bulk_wait_read_all();
        ++done;
        advance(us);
        if (ui.r < q) {
            chunk(ui, at, n);
            ft::mbar_arrive_expect_tx(&fbar[s], n);
            ft::bulk_g2s(fring + (size_t)s * fch, host + (unsigned long long)ffid[ui.r] * rb + at, n, &fbar[s]);
            ++issued;
            advance(ui);
        }
        publish(us);
    }
    ft::bulk_wait_all();
    // after a failed wait, loads still in flight land before the CTA may exit (bounded)
    for (int g = done + (ok ? 0 : 1); g < issued; ++g) ft::mbar_wait(&fbar[g % nf], (uint32_t)(g / nf) & 1u, err);
}

// Bounded wait until the field (*c >> shift) & 0xFFFF (shift 0 or 16), or the
// whole word for shift 32, reaches target (acquire at GPU scope), then order
// the async proxy (bulk copies) after the acquired writes.
__device__ __forceinline__ bool wait_field(const unsigned* c, unsigned shift, unsigned target, unsigned* err) {
    const uint64_t t0 = ft::globaltimer();
    for (unsigned it = 0;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        if (shift < 32) v = (v >> shift) & 0xFFFFu;
        if (v >= target) break;
        __nanosleep(64);
        if ((it & 15u) == 15u && ft::globaltimer() - t0 > FT_WAIT_LIMIT_NS) {
            atomicOr(err, FT_DEVERR_TIMEOUT);
            return false;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

template <int XM, int SB>
__global__ void __launch_bounds__(THREADS, 1) expert_ffn_fp4_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int H = p.H, F = p.F, T = p.T, k = p.k, TG = p.tgroup;
    const int nst = p.nstage;
    const unsigned slot_bytes = p.stage_bytes;
    const int ugpu = p.info[INFO_UGPU];
    const int nasg = p.info[INFO_NASSIGN];
    const int q = p.do_fill ? p.info[INFO_Q] : 0;  // fills performed by this launch: the last q entries
    const int nA = ugpu - q;                        // entries resident before the launch
    const int G = gridDim.x, c = blockIdx.x;
    const int cpe = F / FPC;
    const int r0 = (int)((long long)H * c / G), r1 = (int)((long long)H * (c + 1) / G);
    const int R = r1 - r0;
    const int RMAX = (H + G - 1) / G;
    const int TK = T * k;
    const size_t VGU = (size_t)F * H;                 // W_gu value bytes (2F x H/2)
    const size_t VD = (size_t)H * F / 2;              // W_d value bytes
    const size_t SGU = (size_t)2 * F * H / SB;        // W_gu scale bytes
    const unsigned vrow = (unsigned)H / 2, srow = (unsigned)H / SB;      // W_gu row bytes
    const unsigned dvrow = (unsigned)F / 2, dsrow = (unsigned)F / SB;    // W_d row bytes

    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + nst;
    size_t o = HEAD;
    uint4* x_s = reinterpret_cast<uint4*>(smem + o);  // paired activations (X_SMEM)
    if (XM == X_SMEM) o += ((size_t)T * H * 2 + 127) & ~(size_t)127;
    float* o_s = reinterpret_cast<float*>(smem + o);
    o += ((size_t)TK * RMAX * 4 + 127) & ~(size_t)127;
    int* m_off = reinterpret_cast<int*>(smem + o);
    int* m_slot = m_off + TK + 1;
    int* m_tok = m_slot + TK;
    float* m_gate = reinterpret_cast<float*>(m_tok + TK);
    int* m_pos = reinterpret_cast<int*>(m_gate + TK);
    float* m_gs = reinterpret_cast<float*>(m_pos + TK);   // global scale of each entry
    float* xf = m_gs + TK;                                // row factor 2^-a_t of each token
    o += ((size_t)(6 * TK + 1 + T) * 4 + 127) & ~(size_t)127;
    unsigned char* ring = smem + o;
    const unsigned wpart = ((unsigned)RMAX * (dvrow + dsrow) + 127u) & ~127u;
    const uint4* xsrc = XM == X_GLOBAL ? p.x16 : x_s;

    // --------------------------------------------------------- fused fill
    // The fill thread owns its ring and barriers and starts at once; the
    // consumers stage the worklist and x meanwhile (named barrier 4).
    if (wid > CW) {
        if (lane == 0 && q > 0) {
            const FillParts fp = fp4_fill_parts(H, F, SB);
            fill_parts_tma(reinterpret_cast<const uint8_t*>(p.host_pool), const_cast<uint8_t*>(p.slot_pool), p.rb,
                           q, p.fill_slot, p.fill_fid, p.ready, p.wdc, c, G, fp, ring + (size_t)nst * slot_bytes,
                           reinterpret_cast<uint64_t*>(smem + 128), p.fill_chunk, p.fill_slots, p.err);
        }
        return;
    }
    // Group counters: CTAs whose phase-A items of the group are done (the
    // resident entries in gbar[3], fill r in the low half-word of wdc[r];
    // its high half-word counts the CTAs whose share of the fill's W_gu is in
    // the slot).  Exit count: the consumers and the producer of every CTA
    // count out once they are done with the counters; whoever completes the
    // count returns them to zero for the next launch.  (ready[r], the CTAs
    // whose shares of both parts of fill r are stored, is zeroed by the
    // control pass that schedules the fill.)
    auto group_count = [&](int grp) { return grp == 0 ? p.gbar + 3 : p.wdc + grp - 1; };
    auto count_out = [&]() {
        unsigned n;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(n) : "l"(p.gbar + 2) : "memory");
        if (n == 2u * (unsigned)G - 1u) {
            for (int r = 0; r < q; ++r) p.wdc[r] = 0u;
            p.gbar[3] = 0u;
            p.gbar[2] = 0u;
        }
    };
    // ------------------------------------------------------------ producer
    // The producer starts at once as well: it initialises the ring barriers,
    // lets the consumers use them (named barrier 5, which they take once x is
    // staged) and reads the worklist from global memory.
    if (wid == CW) {
        if (lane == 0) {
            for (int s = 0; s < nst; ++s) {
                ft::mbar_init(&full[s], 1);
                ft::mbar_init(&empty[s], CW);
            }
            ft::mbar_fence_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 5, %0;" ::"n"(CONS + 32) : "memory");
        if (lane == 0) {
            Steps sq;
            sq.c = c;
            sq.G = G;
            sq.cpe = cpe;
            sq.nA = nA;
            sq.nfill = q;
            sq.R = R;
            sq.TG = TG;
            sq.m_off = p.wl_off;
            sq.open(0);
            const uint64_t pol = ft::l2_policy_evict_first();
            // this CTA's W_d rows (values and scales) of the resident entries
            // go to L2 once the ring is primed, so phase B reads them from L2
            auto prefetch_wd = [&]() {
                if (R == 0) return;
                for (int e = 0; e < nA; ++e) {
                    const uint8_t* rec = p.slot_pool + (size_t)p.wl_slot[e] * p.rb;
                    ft::bulk_prefetch_l2(rec + VGU + (size_t)r0 * dvrow, (unsigned)R * dvrow);
                    ft::bulk_prefetch_l2(rec + VGU + VD + SGU + (size_t)r0 * dsrow, (unsigned)R * dsrow);
                }
            };
            int it = 0, counted = -1;  // the last group whose count this thread has seen complete
            int filled_a = 0, filled = 0;  // fills seen with W_gu / the whole record in their slots (in order)
            bool ok = true;
            int kind, ent, item, g0;
            while (ok && sq.next(kind, ent, item, g0)) {
                if (kind == STEP_SEAL) continue;
                const int st = it % nst;
                if (it == nst) prefetch_wd();
                if (it >= nst && !ft::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err)) { ok = false; break; }
                const uint8_t* rec = p.slot_pool + (size_t)p.wl_slot[ent] * p.rb;
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                // a fill's W_gu rows (phase A) or its whole record (phase B)
                // once every CTA has stored its share
                if (kind == STEP_A && ent - nA + 1 > filled_a) {
                    if (!wait_field(p.wdc + (ent - nA), 16, (unsigned)G, p.err)) { ok = false; break; }
                    filled_a = ent - nA + 1;
                }
                if (kind == STEP_B && ent - nA + 1 > filled) {
                    if (!wait_field(p.ready + (ent - nA), 32, (unsigned)G, p.err)) { ok = false; break; }
                    filled = ent - nA + 1;
                }
                if (kind == STEP_A) {
                    const int grow = (item - ent * cpe) * 2 * FPC;  // first gate row; up rows 16 later
                    ft::mbar_arrive_expect_tx(&full[st], 2u * FPC * (vrow + srow));
                    ft::bulk_g2s_hint(dst, rec + (size_t)grow * vrow, FPC * vrow, &full[st], pol);
                    ft::bulk_g2s_hint(dst + FPC * vrow, rec + (size_t)(grow + 16) * vrow, FPC * vrow, &full[st], pol);
                    ft::bulk_g2s_hint(dst + 2 * FPC * vrow, rec + VGU + VD + (size_t)grow * srow, FPC * srow,
                                      &full[st], pol);
                    ft::bulk_g2s_hint(dst + 2 * FPC * vrow + FPC * srow, rec + VGU + VD + (size_t)(grow + 16) * srow,
                                      FPC * srow, &full[st], pol);
                    ++it;
                    continue;
                }
                // phase-B item: this CTA's W_d rows of the entry, then the h
                // rows of the item once every CTA has sealed the entry's group
                const int off = p.wl_off[ent];
                const int ng = min(TG, p.wl_off[ent + 1] - off - g0);
                const unsigned wb = (unsigned)R * dvrow, sb = (unsigned)R * dsrow, hb = (unsigned)ng * F * 4u;
                ft::mbar_arrive_expect_tx(&full[st], wb + sb + hb);
                ft::bulk_g2s_hint(dst, rec + VGU + (size_t)r0 * dvrow, wb, &full[st], pol);
                ft::bulk_g2s_hint(dst + (size_t)RMAX * dvrow, rec + VGU + VD + SGU + (size_t)r0 * dsrow, sb,
                                  &full[st], pol);
                // (waited for once per group; after a timed-out wait the rows
                // are still copied, whatever they hold, so that the item
                // completes and the ring drains)
                const int gq = ent < nA ? 0 : ent - nA + 1;
                if (gq != counted) {
                    ok = wait_field(group_count(gq), gq == 0 ? 32u : 0u, (unsigned)G, p.err);
                    counted = gq;
                }
                ft::bulk_g2s(dst + wpart, p.hbuf + (size_t)(off + g0) * F, hb, &full[st]);
                ++it;
            }
            if (it <= nst && ok) prefetch_wd();
            ft::drain_ring(full, it, nst, p.err);
            count_out();
        }
        return;
    }

    // ------------------------------------------------- consumers: staging
    constexpr int STAGERS = CONS;
    for (int i = tid; i <= ugpu; i += STAGERS) m_off[i] = p.wl_off[i];
    for (int i = tid; i < ugpu; i += STAGERS) {
        m_slot[i] = p.wl_slot[i];
        m_gs[i] = p.gscale[p.wl_fid[i]];
    }
    for (int i = tid; i < nasg; i += STAGERS) {
        m_tok[i] = p.as_tok[i];
        m_gate[i] = p.as_gate[i];
    }
    for (int i = tid; i < TK; i += STAGERS) m_pos[i] = p.out_pos[i];
    // paired, scaled activations: in shared memory by every CTA, or one
    // token row per warp across the grid into the global block, then a grid
    // barrier
    const uint4* xin = reinterpret_cast<const uint4*>(p.x);
    if (XM == X_SMEM) {
        // all threads: per-token maxima (shared atomics on the magnitudes'
        // bits, which order like the values), then the scaled pairs
        unsigned* amax_bits = reinterpret_cast<unsigned*>(xf);
        for (int t = tid; t < T; t += STAGERS) amax_bits[t] = 0u;
        ft::named_bar_sync(4, STAGERS);
        const int qrow = H / 8;
        for (int i = tid; i < T * qrow; i += STAGERS) {
            float f[8];
            ft::bf16x8_to_f32(xin[i], f);
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
            atomicMax(&amax_bits[i / qrow], __float_as_uint(m));
        }
        ft::named_bar_sync(4, STAGERS);
        for (int i = tid; i < T * qrow; i += STAGERS) {
            const int t = i / qrow, q8 = i - t * qrow;
            const int a = x_exponent(__uint_as_float(amax_bits[t]));
            x_s[(size_t)t * qrow + xpos(q8)] = x_pairs(xin[i], ldexpf(1.f, a));
        }
        ft::named_bar_sync(4, STAGERS);
        for (int t = tid; t < T; t += STAGERS) xf[t] = ldexpf(1.f, -x_exponent(__uint_as_float(amax_bits[t])));
        ft::named_bar_sync(4, STAGERS);
    } else {
        for (int t = c + G * wid; t < T; t += G * (STAGERS / 32)) {
            const float fct = stage_x_row(xin + (size_t)t * (H / 8), H, p.x16 + (size_t)t * (H / 8), lane);
            if (lane == 0) p.xsc[t] = fct;
        }
        ft::named_bar_sync(4, STAGERS);
        if (tid == 0) ft::grid_barrier(p.gbar, (unsigned)G, p.err);
        ft::named_bar_sync(4, STAGERS);
        for (int t = tid; t < T; t += STAGERS) xf[t] = p.xsc[t];
        ft::named_bar_sync(4, STAGERS);
    }
    ft::named_bar_sync(5, CONS + 32);  // the producer has initialised the ring barriers

    Steps sq;
    sq.c = c;
    sq.G = G;
    sq.cpe = cpe;
    sq.nA = nA;
    sq.nfill = q;
    sq.R = R;
    sq.TG = TG;
    sq.m_off = m_off;
    sq.open(0);


    // ------------------------------------- consumers: phase-A and phase-B items
    // Phase-A items are taken by all 16 warps; phase-B items alternate
    // between the two halves of 8 warps (half 0 the even ones), so that two
    // items' conversions, barriers and short row chains overlap; each warp of
    // the taking half arrives twice on the slot's empty barrier (its count is
    // 16).  After a failed (timed-out) wait a warp stops waiting, computing
    // and releasing slots, but takes the same barriers and seals as the
    // others of its half.
    constexpr int HW = CW / 2;           // warps per half
    constexpr int HT = HW * 32;          // threads per half
    const int half = wid / HW;
    int it = 0, nb = 0;
    bool failed = false;
    int kind, ent, item, g0;
    while (sq.next(kind, ent, item, g0)) {
        if (kind == STEP_SEAL) {
            // every warp's h of the group's items on this CTA is written
            ft::named_bar_sync(3, CONS);
            if (tid == 0) ft::red_release_gpu_add(group_count(ent), 1u);
            continue;
        }
        const int st = it % nst;
        if (kind == STEP_B && (nb & 1) != half) {  // the other half's item
            ++it;
            ++nb;
            continue;
        }
        const bool ok = !failed && __all_sync(0xffffffffu, ft::mbar_wait(&full[st], (it / nst) & 1, p.err));
        failed = !ok;
        const unsigned char* sb = ring + (size_t)st * slot_bytes;
        const int off = m_off[ent];
        const int ntok = m_off[ent + 1] - off;
        if (kind == STEP_A) {
            // gate/up + SwiGLU: warp w computes feature w of the item
            const int f = (item - ent * cpe) * FPC + wid;
            const uint4* gv = reinterpret_cast<const uint4*>(sb + (size_t)wid * vrow);
            const uint4* uv = reinterpret_cast<const uint4*>(sb + (size_t)(FPC + wid) * vrow);
            const uint8_t* gs = sb + 2 * FPC * vrow + (size_t)wid * srow;
            const uint8_t* us = sb + 2 * FPC * vrow + FPC * srow + (size_t)wid * srow;
            if (ok) gu_feature4<XM, SB>(gv, uv, gs, us, xsrc, xf, H, m_tok, off, ntok, F, f, lane, m_gs[ent], p.hbuf);
            __syncwarp();
            if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
            ++it;
            continue;
        }
        // down rows [r0, r1) of one token group of the entry, by this half.
        // The staged fp32 h rows are converted to f16 pairs, each 16-value
        // block scaled by its own power of two, by the half's threads into
        // the slot's tail (past the W_d rows and the fp32 rows the copy
        // lands): the pairs, then the block factors; then the half's barrier
        // (warps whose wait failed still take it).  Consecutive items use
        // different slots, and a slot's tail is rewritten only after every
        // warp has released the slot.
        const int ng = min(TG, ntok - g0);
        const float* hs = reinterpret_cast<const float*>(sb + wpart);
        unsigned char* tail = ring + (size_t)st * slot_bytes + wpart + (size_t)TG * F * 4;
        uint4* hp = reinterpret_cast<uint4*>(tail);
        float* hfb = reinterpret_cast<float*>(tail + (size_t)TG * F * 2);
        if (ok) {
            // the two chunks of a block are lanes 2m and 2m + 1 of one step
            // (F/8 is a multiple of 32, so every lane of a warp takes the same
            // number of steps)
            for (int i = tid - half * HT; i < ng * (F / 8); i += HT) {
                const int n = i / (F / 8), q8 = i - n * (F / 8);
                float fb;
                hp[(size_t)n * (F / 8) + xpos(q8)] = h_pairs_block(hs + (size_t)n * F, q8, &fb);
                if ((q8 & 1) == 0) hfb[(size_t)n * (F / 16) + (q8 >> 1)] = fb;
            }
        }
        if (half)  // constant barrier ids (a computed id reserves every barrier of the CTA)
            ft::named_bar_sync(7, HT);
        else
            ft::named_bar_sync(6, HT);
        for (int rb = wid - half * HW; rb < R && ok; rb += RW * HW)
            down_rows4<SB, HW>(sb, sb + (size_t)RMAX * dvrow, dvrow, dsrow, hp, hfb, ng, F, lane, m_gs[ent], o_s,
                               off + g0, RMAX, rb, R);
        __syncwarp();
        if (ok && lane == 0) mbar_arrive_n(&empty[st], 2);
        ++it;
        ++nb;
    }
    ft::named_bar_sync(1, CONS);
    for (int idx = tid; idx < T * R; idx += CONS) {
        const int t = idx / R, rl = idx - t * R;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
            const int pos = m_pos[t * k + j];
            if (pos >= 0) acc = fmaf(m_gate[pos], o_s[(size_t)pos * RMAX + rl], acc);
        }
        const size_t oi = (size_t)t * H + r0 + rl;
        if (p.partial_C) acc += p.partial_C[oi];
        p.y[oi] = acc;
    }
    if (tid == 0) count_out();  // after this CTA's last seal
}

}  // namespace

bool expert_ffn_fp4_fits(int H, int F, int T, int k, int fmt, int num_sms) {
    Fp4Plan pl;
    return fp4_plan(H, F, T, k, fmt == FT_FMT_MXFP4 ? 32 : 16, num_sms, pl);
}

cudaError_t launch_expert_ffn_fp4(ExpertParams p, int fmt, int num_sms, cudaStream_t s) {
    if (fmt != FT_FMT_NVFP4 && fmt != FT_FMT_MXFP4) return cudaErrorInvalidValue;
    const int SB = fmt == FT_FMT_MXFP4 ? 32 : 16;
    Fp4Plan pl;
    if (!fp4_plan(p.H, p.F, p.T, p.k, SB, num_sms, pl)) return cudaErrorInvalidValue;
    const int xm = pl.xm;
    if (xm == X_GLOBAL && (!p.x16 || !p.xsc)) return cudaErrorInvalidValue;
    const size_t head = pl.head, slot = pl.slot, fch = pl.fch;
    const int nst = pl.nst, nf = pl.nf;
    p.nstage = nst;
    p.stage_bytes = (unsigned)slot;
    p.tgroup = pl.tg;
    p.fill_chunk = (unsigned)fch;
    p.fill_slots = nf;
    const size_t smem = head + slot * nst + (size_t)nf * fch;
    const void* fn = SB == 16 ? (xm == X_SMEM ? (const void*)expert_ffn_fp4_kernel<X_SMEM, 16>
                                              : (const void*)expert_ffn_fp4_kernel<X_GLOBAL, 16>)
                              : (xm == X_SMEM ? (const void*)expert_ffn_fp4_kernel<X_SMEM, 32>
                                              : (const void*)expert_ffn_fp4_kernel<X_GLOBAL, 32>);
    cudaError_t e = ensure_dynamic_smem(fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, fn, args);
}
