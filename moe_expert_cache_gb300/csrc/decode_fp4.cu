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
//     added in fp32; the row total is rescaled once by the token's power of
//     two and the expert's global.
// The per-token maximum of h is formed in phase A (shared-memory maxima,
// then one 64-bit atomic max per CTA and token, tagged with the grid
// barrier's generation so that values from earlier launches lose).
//
// Record (per layer-expert): [W_gu values 2F x H/2 bytes, low nibble first,
// gate/up rows interleaved in groups of 16][W_d values H x F/2]
// [W_gu scales 2F x H/SB][W_d scales H x F/SB].
//
// Layout of the work: 16 consumer warps, one producer warp (TMA ring) and one
// fill warp.  A phase-A item is 16 features (16 gate rows, the 16 up rows and
// their scale rows, one warp per feature); a phase-B item is (expert, group
// of at most TG tokens): the CTA's W_d rows, the staged fp32 h rows and, in
// the slot's tail, those rows converted to f16 pairs, two W_d rows per warp
// pass.  x is converted into shared memory when T*H*2 bytes fit, else into a
// global block behind a grid barrier.  A grid barrier separates phase A from
// phase B.
#include "ft_common.cuh"
#include "../../include/ft.h"

namespace {

constexpr int CW = 16;                // consumer warps
constexpr int CONS = CW * 32;
constexpr int FILL_WARPS = 1;         // fused cache fill (one TMA thread)
constexpr int THREADS = CONS + 32 + FILL_WARPS * 32;  // + producer warp + fill warps
constexpr int FPC = CW;               // features per phase-A chunk: one per consumer warp
constexpr int RW = 2;                 // W_d rows per warp pass in phase B
constexpr size_t HEAD = 256;
// Phase-A activations: f16 pairs in shared memory (X_SMEM, when T*H*2 bytes
// fit) or in a global scratch row block written at the start of the launch
// (X_GLOBAL).
enum { X_SMEM = 0, X_GLOBAL = 1 };
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
                                          int F, int f, int lane, float gsc, float* hbuf, unsigned* hmx) {
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
    // read only by phase B, as staged rows: swizzled for its fp32 loads; the
    // token's largest |h| of this CTA is kept for phase B's scaling
    if (lane < NT) {
        hbuf[(size_t)(off + g0 + lane) * F + swz_f32(f)] = mine;
        atomicMax(&hmx[tk[lane]], __float_as_uint(fabsf(mine)));
    }
}

template <int XM, int SB>
__device__ __noinline__ void gu_feature4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                            const uint4* xs, const float* xf, int H, const int* m_tok, int off,
                                            int ntok, int F, int f, int lane, float gsc, float* hbuf,
                                            unsigned* hmx) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 2) {
            gu_group4<2, XM, SB>(gv, uv, gs, us, xs, xf, H, m_tok, off, g0, F, f, lane, gsc, hbuf, hmx);
            g0 += 2;
        } else {
            gu_group4<1, XM, SB>(gv, uv, gs, us, xs, xf, H, m_tok, off, g0, F, f, lane, gsc, hbuf, hmx);
            g0 += 1;
        }
    }
}

// Phase B: the W_d rows rb + CW*r (r < RW, row < R) of a slot (values +
// scales) against NT h rows held as scaled f16 pairs (the layout of the
// phase-A activations, F/8 chunks per row; row factors hf).  Each h chunk is
// loaded once and applied to every row of the warp.
template <int NT, int SB>
__device__ __forceinline__ void down_group4(const uint8_t* wrows, const uint8_t* srows, unsigned dvrow,
                                            unsigned dsrow, const uint4* hp, const float* hfr, int g, int F,
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
            const int rl = rb + CW * r < R ? rb + CW * r : rb;  // rows past R repeat row rb (not stored)
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
#pragma unroll
            for (int r = 0; r < RW; ++r)
                acc[r][n] = fmaf(sc[r].x, dot16_h(d[r], hc[0], hc[1]),
                                 fmaf(sc[r].y, dot16_h(d[r] + 8, hc[2], hc[3]), acc[r][n]));
        }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int rl = rb + CW * r;
        if (rl < R) {  // warp-uniform
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float sv = ft::warp_sum(acc[r][n]) * hfr[g + n] * gsc;
                if (lane == 0) o_s[(size_t)(obase + g + n) * RMAX + rl] = sv;
            }
        }
    }
}

// The rows rb + CW*r (r < RW) of a slot against its ng h rows, two tokens
// at a time.
template <int SB>
__device__ __noinline__ void down_rows4(const uint8_t* wrows, const uint8_t* srows, unsigned dvrow,
                                        unsigned dsrow, const uint4* hp, const float* hfr, int ng, int F, int lane,
                                        float gsc, float* o_s, int obase, int RMAX, int rb, int R) {
    int g = 0;
    while (g < ng) {
        if (ng - g >= 2) {
            down_group4<2, SB>(wrows, srows, dvrow, dsrow, hp, hfr, g, F, lane, gsc, o_s, obase, RMAX, rb, R);
            g += 2;
        } else {
            down_group4<1, SB>(wrows, srows, dvrow, dsrow, hp, hfr, g, F, lane, gsc, o_s, obase, RMAX, rb, R);
            g += 1;
        }
    }
}

// Eight fp32 values (h elements 8q..8q+7 of a staged row, swizzled as
// swz_f32) times `up` as the chunk of four f16 pairs (h[2J], h[2J+1]).
__device__ __forceinline__ uint4 h_pairs(const float* hr, int q, float up) {
    const float4 lo = *reinterpret_cast<const float4*>(hr + swz_f32(8 * q));
    const float4 hi = *reinterpret_cast<const float4*>(hr + swz_f32(8 * q + 4));
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

template <int XM, int SB>
__global__ void __launch_bounds__(THREADS, 1) expert_ffn_fp4_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_gdone;
    __shared__ unsigned s_gen;  // grid barrier generation at the start of phase A
    const int H = p.H, F = p.F, T = p.T, k = p.k, TG = p.tgroup;
    const int nst = p.nstage;
    const unsigned slot_bytes = p.stage_bytes;
    const int ugpu = p.info[INFO_UGPU];
    const int nasg = p.info[INFO_NASSIGN];
    const int G = gridDim.x, c = blockIdx.x;
    const int cpe = F / FPC;
    const int NA = ugpu * cpe;
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
    int* m_fill = reinterpret_cast<int*>(m_gs + TK);      // fill index of each entry (or -1)
    float* xf = reinterpret_cast<float*>(m_fill + TK);    // row factor 2^-a_t of each token
    unsigned* hmx = reinterpret_cast<unsigned*>(xf + T);  // largest |h| of each token (this CTA, then all)
    float* hup = reinterpret_cast<float*>(hmx + T);       // h scale 2^b_t of each token
    float* hfr = hup + T;                                 // h row factor 2^-b_t of each staged row
    o += ((size_t)(7 * TK + 1 + 3 * T + 2 * TG) * 4 + 127) & ~(size_t)127;
    unsigned char* ring = smem + o;
    const unsigned wpart = ((unsigned)RMAX * (dvrow + dsrow) + 127u) & ~127u;
    const uint4* xsrc = XM == X_GLOBAL ? p.x16 : x_s;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            ft::mbar_init(&full[s], 1);
            ft::mbar_init(&empty[s], CW);
        }
        ft::mbar_fence_init();
        s_gdone = 0;
    }
    for (int i = tid; i <= ugpu; i += THREADS) m_off[i] = p.wl_off[i];
    for (int i = tid; i < ugpu; i += THREADS) {
        m_slot[i] = p.wl_slot[i];
        m_gs[i] = p.gscale[p.wl_fid[i]];
        m_fill[i] = p.do_fill ? p.wl_fill[i] : -1;
    }
    for (int i = tid; i < nasg; i += THREADS) {
        m_tok[i] = p.as_tok[i];
        m_gate[i] = p.as_gate[i];
    }
    for (int i = tid; i < TK; i += THREADS) m_pos[i] = p.out_pos[i];
    for (int i = tid; i < T; i += THREADS) hmx[i] = 0u;
    // paired, scaled activations: in shared memory by every CTA, or one
    // token row per warp across the grid into the global block, then a grid
    // barrier
    const uint4* xin = reinterpret_cast<const uint4*>(p.x);
    if (XM == X_SMEM) {
        // all threads: per-token maxima (shared atomics on the magnitudes'
        // bits, which order like the values), then the scaled pairs
        unsigned* amax_bits = reinterpret_cast<unsigned*>(xf);
        for (int t = tid; t < T; t += THREADS) amax_bits[t] = 0u;
        __syncthreads();
        const int qrow = H / 8;
        for (int i = tid; i < T * qrow; i += THREADS) {
            float f[8];
            ft::bf16x8_to_f32(xin[i], f);
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
            atomicMax(&amax_bits[i / qrow], __float_as_uint(m));
        }
        __syncthreads();
        for (int i = tid; i < T * qrow; i += THREADS) {
            const int t = i / qrow, q = i - t * qrow;
            const int a = x_exponent(__uint_as_float(amax_bits[t]));
            x_s[(size_t)t * qrow + xpos(q)] = x_pairs(xin[i], ldexpf(1.f, a));
        }
        __syncthreads();
        for (int t = tid; t < T; t += THREADS) xf[t] = ldexpf(1.f, -x_exponent(__uint_as_float(amax_bits[t])));
        __syncthreads();
    } else {
        for (int t = c + G * wid; t < T; t += G * (THREADS / 32)) {
            const float fct = stage_x_row(xin + (size_t)t * (H / 8), H, p.x16 + (size_t)t * (H / 8), lane);
            if (lane == 0) p.xsc[t] = fct;
        }
        __syncthreads();
        if (tid == 0) ft::grid_barrier(p.gbar, (unsigned)G, p.err);
        __syncthreads();
        for (int t = tid; t < T; t += THREADS) xf[t] = p.xsc[t];
        __syncthreads();
    }

    if (tid == 0) s_gen = ft::ld_acquire_gpu(&p.gbar[1]);  // no grid barrier can pass before phase A ends
    __syncthreads();

    // --------------------------------------------------------- fused fill
    if (wid > CW) {
        if (lane == 0 && p.do_fill)
            ft::fill_share_tma(reinterpret_cast<const uint8_t*>(p.host_pool), const_cast<uint8_t*>(p.slot_pool), p.rb,
                               p.info[INFO_Q], p.fill_slot, p.fill_fid, p.ready, c, G,
                               ring + (size_t)nst * slot_bytes, reinterpret_cast<uint64_t*>(smem + 128),
                               p.fill_chunk, p.fill_slots, p.err);
        return;
    }
    // ------------------------------------------------------------ producer
    if (wid == CW) {
        if (lane == 0) {
            const uint64_t pol = ft::l2_policy_evict_first();
            // this CTA's W_d rows (values and scales) of the resident entries
            // go to L2 once the ring is primed, so phase B reads them from L2
            auto prefetch_wd = [&]() {
                if (R == 0) return;
                for (int e = 0; e < ugpu; ++e) {
                    if (m_fill[e] >= 0) continue;
                    const uint8_t* rec = p.slot_pool + (size_t)m_slot[e] * p.rb;
                    ft::bulk_prefetch_l2(rec + VGU + (size_t)r0 * dvrow, (unsigned)R * dvrow);
                    ft::bulk_prefetch_l2(rec + VGU + VD + SGU + (size_t)r0 * dsrow, (unsigned)R * dsrow);
                }
            };
            int it = 0;
            bool ok = true;
            int waited = -1;
            for (int a = c; a < NA && ok; a += G, ++it) {
                const int st = it % nst;
                if (it == nst) prefetch_wd();
                if (it >= nst && !ft::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err)) { ok = false; break; }
                const int ent = a / cpe;
                if (m_fill[ent] >= 0 && m_fill[ent] != waited) {
                    if (!ft::wait_filled(p.ready, m_fill[ent], (unsigned)G, p.err)) { ok = false; break; }
                    waited = m_fill[ent];
                }
                const int f0 = (a - ent * cpe) * FPC;
                const uint8_t* rec = p.slot_pool + (size_t)m_slot[ent] * p.rb;
                const int grow = (f0 >> 4) * 32 + (f0 & 15);  // first gate row; up rows 16 later
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                ft::mbar_arrive_expect_tx(&full[st], 2u * FPC * (vrow + srow));
                ft::bulk_g2s_hint(dst, rec + (size_t)grow * vrow, FPC * vrow, &full[st], pol);
                ft::bulk_g2s_hint(dst + FPC * vrow, rec + (size_t)(grow + 16) * vrow, FPC * vrow, &full[st], pol);
                ft::bulk_g2s_hint(dst + 2 * FPC * vrow, rec + VGU + VD + (size_t)grow * srow, FPC * srow, &full[st], pol);
                ft::bulk_g2s_hint(dst + 2 * FPC * vrow + FPC * srow, rec + VGU + VD + (size_t)(grow + 16) * srow,
                                  FPC * srow, &full[st], pol);
            }
            if (it <= nst && ok) prefetch_wd();
            // phase B items = (expert, group of <= TG tokens); W_d rows stream
            // ahead of the grid barrier, h rows after it
            int nitems = 0;
            if (R > 0)
                for (int e = 0; e < ugpu; ++e) nitems += (m_off[e + 1] - m_off[e] + TG - 1) / TG;
            const int pre = nitems < nst ? nitems : nst;
            const int itB = it;
            bool gdone = false;
            int e = 0, g0 = 0, idx = 0;
            for (; idx < nitems && ok; ++idx, ++it) {
                const int st = it % nst;
                if (it >= nst && !ft::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err)) { ok = false; break; }
                const int off = m_off[e], ntok = m_off[e + 1] - off;
                const int ng = min(TG, ntok - g0);
                const uint8_t* rec = p.slot_pool + (size_t)m_slot[e] * p.rb;
                if (g0 == 0 && m_fill[e] >= 0 && !ft::wait_filled(p.ready, m_fill[e], (unsigned)G, p.err)) {
                    ok = false;
                    break;
                }
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                const unsigned wb = (unsigned)R * dvrow, sb = (unsigned)R * dsrow, hb = (unsigned)ng * F * 4u;
                ft::mbar_arrive_expect_tx(&full[st], wb + sb + hb);
                ft::bulk_g2s_hint(dst, rec + VGU + (size_t)r0 * dvrow, wb, &full[st], pol);
                ft::bulk_g2s_hint(dst + (size_t)RMAX * dvrow, rec + VGU + VD + SGU + (size_t)r0 * dsrow, sb, &full[st], pol);
                if (idx >= pre - 1) {
                    if (!gdone) {
                        const uint64_t t0 = ft::globaltimer();
                        while (!ft::ld_acquire_cta(&s_gdone)) {
                            if (ft::globaltimer() - t0 > FT_WAIT_LIMIT_NS) {
                                atomicOr(p.err, FT_DEVERR_TIMEOUT);
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        gdone = true;
                        // deferred h rows of the items prefetched before the barrier
                        int e2 = 0, g2 = 0;
                        for (int i2 = 0; i2 <= idx; ++i2) {
                            const int off2 = m_off[e2], nt2 = m_off[e2 + 1] - off2;
                            const int ng2 = min(TG, nt2 - g2);
                            const int st2 = (itB + i2) % nst;
                            ft::bulk_g2s(ring + (size_t)st2 * slot_bytes + wpart, p.hbuf + (size_t)(off2 + g2) * F,
                                         (unsigned)ng2 * F * 4u, &full[st2]);
                            g2 += TG;
                            if (g2 >= nt2) { g2 = 0; ++e2; }
                        }
                    } else {
                        ft::bulk_g2s(dst + wpart, p.hbuf + (size_t)(off + g0) * F, hb, &full[st]);
                    }
                }
                g0 += TG;
                if (g0 >= ntok) { g0 = 0; ++e; }
            }
            ft::drain_ring(full, it, nst, p.err);
        }
        return;
    }

    // ------------------------------------------------- phase A: gate/up + SwiGLU
    int it = 0;
    bool failed = false;
    for (int a = c; a < NA; a += G, ++it) {
        const int st = it % nst;
        const bool ok = !failed && ft::mbar_wait(&full[st], (it / nst) & 1, p.err);
        failed = !ok;
        const int ent = a / cpe;
        const int f = (a - ent * cpe) * FPC + wid;
        const int off = m_off[ent];
        const int ntok = m_off[ent + 1] - off;
        const unsigned char* sb = ring + (size_t)st * slot_bytes;
        const uint4* gv = reinterpret_cast<const uint4*>(sb + (size_t)wid * vrow);
        const uint4* uv = reinterpret_cast<const uint4*>(sb + (size_t)(FPC + wid) * vrow);
        const uint8_t* gs = sb + 2 * FPC * vrow + (size_t)wid * srow;
        const uint8_t* us = sb + 2 * FPC * vrow + FPC * srow + (size_t)wid * srow;
        if (ok)
            gu_feature4<XM, SB>(gv, uv, gs, us, xsrc, xf, H, m_tok, off, ntok, F, f, lane, m_gs[ent], p.hbuf, hmx);
        __syncwarp();
        if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
    }

    // per-token |h| maxima of the grid, tagged with the barrier generation of
    // this launch in the high word (older values lose every comparison)
    ft::named_bar_sync(1, CONS);
    const unsigned long long gen = (unsigned long long)s_gen << 32;
    for (int t = tid; t < T; t += CONS)
        atomicMax(reinterpret_cast<unsigned long long*>(p.hmax) + t, gen | hmx[t]);
    ft::named_bar_sync(1, CONS);
    if (tid == 0) {
        ft::grid_barrier(p.gbar, (unsigned)G, p.err);
        ft::st_release_cta(&s_gdone, 1);
    }
    ft::named_bar_sync(1, CONS);
    for (int t = tid; t < T; t += CONS) {
        const unsigned long long v = reinterpret_cast<const unsigned long long*>(p.hmax)[t];
        const int b = x_exponent((v >> 32) == (gen >> 32) ? __uint_as_float((unsigned)v) : 0.f);
        hup[t] = ldexpf(1.f, b);
        xf[t] = ldexpf(1.f, -b);  // phase A is done with the x factors
    }
    ft::named_bar_sync(1, CONS);

    // ---------------------------------------------------- phase B: down rows
    if (R > 0) {
        for (int e = 0; e < ugpu; ++e) {
            const int off = m_off[e], ntok = m_off[e + 1] - off;
            for (int g0 = 0; g0 < ntok; g0 += TG, ++it) {
                const int ng = min(TG, ntok - g0);
                const int st = it % nst;
                const bool ok = !failed && ft::mbar_wait(&full[st], (it / nst) & 1, p.err);
                failed = !ok;
                const unsigned char* sb = ring + (size_t)st * slot_bytes;
                const float* hs = reinterpret_cast<const float*>(sb + wpart);
                // the staged h rows as scaled f16 pairs, written by every
                // consumer thread into the slot's tail (past the W_d rows and
                // the fp32 rows the copy lands), then one barrier; warps whose
                // wait failed still take the barrier.  Consecutive items use
                // different slots, and a slot's tail is rewritten only after
                // every warp has passed the barrier of the item before.
                uint4* hp = reinterpret_cast<uint4*>(ring + (size_t)st * slot_bytes + wpart + (size_t)TG * F * 4);
                if (ok) {
                    for (int i = tid; i < ng * (F / 8); i += CONS) {
                        const int n = i / (F / 8), q = i - n * (F / 8);
                        hp[(size_t)n * (F / 8) + xpos(q)] = h_pairs(hs + (size_t)n * F, q, hup[m_tok[off + g0 + n]]);
                    }
                    if (tid < ng) hfr[(it & 1) * TG + tid] = xf[m_tok[off + g0 + tid]];
                }
                ft::named_bar_sync(2, CONS);
                for (int rb = wid; rb < R && ok; rb += RW * CW)
                    down_rows4<SB>(sb, sb + (size_t)RMAX * dvrow, dvrow, dsrow, hp, hfr + (it & 1) * TG, ng, F,
                                   lane, m_gs[e], o_s, off + g0, RMAX, rb, R);
                __syncwarp();
                if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
            }
        }
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
}

}  // namespace

static constexpr size_t kSmemLimit4 = 227 * 1024 - 256;  // dynamic; the rest is static shared memory

namespace {

// Shared-memory plan of one FP4 launch (T tokens), or false when no plan fits.
struct Fp4Plan {
    int xm, tg, nst, nf;
    size_t head, slot, fch;
};

bool fp4_plan(int H, int F, int T, int k, int SB, int G, Fp4Plan& pl) {
    const int RMAX = (H + G - 1) / G;
    const size_t TK = (size_t)T * k;
    pl.xm = (size_t)T * H * 2 <= 32768 ? X_SMEM : X_GLOBAL;
    const size_t xbytes = pl.xm == X_SMEM ? (size_t)T * H * 2 : 0;
    const size_t head0 = HEAD + ((xbytes + 127) & ~(size_t)127) + ((TK * RMAX * 4 + 127) & ~(size_t)127);
    const size_t chunk = (size_t)2 * FPC * (H / 2 + H / SB);
    const size_t wpart = ((size_t)RMAX * (F / 2 + F / SB) + 127) & ~(size_t)127;
    // The fill ring is kept small (3 x 4 KiB per SM): host reads queued beyond
    // the link's bandwidth-delay product delay every SM's HBM reads.
    pl.fch = 4096;
    // token group of phase B: the most h rows (at most 16) whose staging in a
    // slot (fp32 as copied, then f16 pairs) leaves room for two slots
    int tg = T < 16 ? T : 16;
    for (; tg >= 1; --tg) {
        pl.head = head0 + (((7 * TK + 1 + 3 * (size_t)T + 2 * (size_t)tg) * 4 + 127) & ~(size_t)127);
        pl.slot = wpart + (size_t)tg * F * 6;
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
