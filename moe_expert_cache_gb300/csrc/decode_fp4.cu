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
// Weight w = e2m1 * scale(block along K) * global(expert).  Each block is
// summed in fp32 against the fp32 activations, scaled by its scale, and the
// row total is multiplied by the expert's global once.  Activations are not
// quantised (W4A16).
//
// Record (per layer-expert): [W_gu values 2F x H/2 bytes, low nibble first,
// gate/up rows interleaved in groups of 16][W_d values H x F/2]
// [W_gu scales 2F x H/SB][W_d scales H x F/SB].
//
// Differences from the BF16 kernel: a phase-A slot holds 8 gate rows, the 8
// matching up rows and their scale rows (four bulk copies); a phase-B item is
// (expert, group of at most TG tokens) so that the staged h rows stay within
// a slot for any T; x is read from shared memory (fp32 or bf16) when it fits
// and from global memory otherwise.
#include "ft_common.cuh"
#include "../../include/ft.h"

namespace {

constexpr int CW = 8;                 // consumer warps
constexpr int CONS = CW * 32;
constexpr int FILL_WARPS = 1;         // fused cache fill (one TMA thread)
constexpr int THREADS = CONS + 32 + FILL_WARPS * 32;  // + producer warp + fill warps
constexpr int FPC = CW;               // features per phase-A chunk
constexpr size_t HEAD = 256;
enum { X_F32_SMEM = 0, X_BF16_SMEM = 1, X_BF16_GLOBAL = 2 };

// e2m1 decode by bit placement: code j of word w (nibble j, low nibble
// first) becomes the fp32 whose exponent field holds the code's two exponent
// bits, whose top mantissa bit holds its mantissa bit and whose sign is its
// sign.  That float equals value * 2^-126 exactly, for the subnormal code 1
// (0.5) as well; activations are held scaled by 2^64 (kActScale) so the
// products stay normal, and the row sums are rescaled by 2^62 (kSumScale).
// Four integer operations per value instead of a table lookup or a
// conversion instruction.
constexpr float kActScale = 18446744073709551616.0f;  // 2^64
constexpr float kSumScale = 4611686018427387904.0f;   // 2^62

template <int J>
__device__ __forceinline__ float e2m1_scaled(uint32_t w) {
    const uint32_t mag = (J * 4 <= 22 ? (w << (J * 4 <= 22 ? 22 - 4 * J : 0)) : (w >> (J * 4 > 22 ? 4 * J - 22 : 0))) &
                         0x01C00000u;
    const uint32_t sgn = (w << (28 - 4 * J)) & 0x80000000u;
    return __uint_as_float(mag | sgn);
}

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
// the exponent field, code 0 the subnormal 2^-127, code 255 NaN.
template <int SB>
__device__ __forceinline__ float2 scales32(const uint8_t* srow, int v) {
    if (SB == 16) return e4m3x2_f32(srow + 2 * v);
    const uint32_t c = srow[v];
    const float s = __uint_as_float(c == 255u ? 0x7FC00000u : c == 0u ? 0x00400000u : c << 23);
    return make_float2(s, s);
}

// Activation rows in shared memory (x and the staged h rows) are swizzled so
// that a warp's loads of its lanes' 32-value groups spread over all banks:
// within group v (128 bytes of fp32, or 64 bytes of bf16), 16-byte chunk i
// is stored at chunk (i + v) mod 8 (fp32) or (i + v) mod 4 (bf16).
__device__ __forceinline__ int swz_f32(int e) {  // element e of a row -> its stored position
    const int v = e >> 5, i = (e >> 2) & 7;
    return (v << 5) | (((i + v) & 7) << 2) | (e & 3);
}

// 32 activations of token row `xr` starting at element 32*v.
template <int XM>
__device__ __forceinline__ void load_x32(const void* xr, int v, float* x) {
    if (XM == X_F32_SMEM) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(xr) + (size_t)v * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = p[(i + v) & 7];
            x[4 * i] = q.x; x[4 * i + 1] = q.y; x[4 * i + 2] = q.z; x[4 * i + 3] = q.w;
        }
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(xr) + (size_t)v * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 q = XM == X_BF16_GLOBAL ? __ldg(p + i) : p[(i + v) & 3];
            ft::bf16x8_to_f32(q, x + 8 * i);
#pragma unroll
            for (int j = 0; j < 8; ++j) x[8 * i + j] *= kActScale;
        }
    }
}

// eight values of one word against x[0..7] (scaled), added to a / b (even / odd)
__device__ __forceinline__ void fp4_word(uint32_t w, const float* x, float& a, float& b) {
    a = fmaf(e2m1_scaled<0>(w), x[0], a);
    b = fmaf(e2m1_scaled<1>(w), x[1], b);
    a = fmaf(e2m1_scaled<2>(w), x[2], a);
    b = fmaf(e2m1_scaled<3>(w), x[3], b);
    a = fmaf(e2m1_scaled<4>(w), x[4], a);
    b = fmaf(e2m1_scaled<5>(w), x[5], b);
    a = fmaf(e2m1_scaled<6>(w), x[6], a);
    b = fmaf(e2m1_scaled<7>(w), x[7], b);
}

// sum over 32 values of one uint4 (two scale blocks): sc0 * block0 + sc1 * block1,
// in units of 2^-62 (activations scaled by 2^64, values by 2^-126)
__device__ __forceinline__ float fp4_dot32(const uint4& w, const float* x, float sc0, float sc1) {
    float a0 = 0.f, b0 = 0.f, a1 = 0.f, b1 = 0.f;
    fp4_word(w.x, x, a0, b0);
    fp4_word(w.y, x + 8, a0, b0);
    fp4_word(w.z, x + 16, a1, b1);
    fp4_word(w.w, x + 24, a1, b1);
    return fmaf(sc0, a0 + b0, sc1 * (a1 + b1));
}

// Phase A: gate and up rows of one feature against NT tokens; returns the
// un-globalled row sums in ag / au.
template <int NT, int XM, int SB>
__device__ __forceinline__ void gu_dots4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                         const void* xs, size_t xrow_elems, const int* tk, int H, int lane,
                                         float* ag, float* au) {
#pragma unroll
    for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
    const int nv = H >> 5;  // uint4 (32 values) per row
    for (int v = lane; v < nv; v += 32) {
        const uint4 wg = gv[v], wu = uv[v];
        const float2 gsc2 = scales32<SB>(gs, v), usc2 = scales32<SB>(us, v);
        const float g0 = gsc2.x, g1 = gsc2.y, u0 = usc2.x, u1 = usc2.y;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float x[32];
            const void* xr = XM == X_F32_SMEM
                                 ? (const void*)(static_cast<const float*>(xs) + (size_t)tk[n] * xrow_elems)
                                 : (const void*)(static_cast<const __nv_bfloat16*>(xs) + (size_t)tk[n] * xrow_elems);
            load_x32<XM>(xr, v, x);
            ag[n] += fp4_dot32(wg, x, g0, g1);
            au[n] += fp4_dot32(wu, x, u0, u1);
        }
    }
}

template <int NT, int XM, int SB>
__device__ __forceinline__ void gu_group4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                          const void* xs, int H, const int* m_tok, int off, int g0, int F, int f,
                                          int lane, float gsc, float* hbuf) {
    int tk[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) tk[n] = m_tok[off + g0 + n];
    float ag[NT], au[NT];
    gu_dots4<NT, XM, SB>(gv, uv, gs, us, xs, (size_t)H, tk, H, lane, ag, au);
    float mine = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float sg = ft::warp_sum(ag[n]) * kSumScale * gsc;
        const float su = ft::warp_sum(au[n]) * kSumScale * gsc;
        if (lane == n) mine = ft::silu_mul(sg, su);
    }
    // read only by phase B, as staged rows: scaled and swizzled like x
    if (lane < NT) hbuf[(size_t)(off + g0 + lane) * F + swz_f32(f)] = mine * kActScale;
}

template <int XM, int SB>
__device__ __forceinline__ void gu_feature4(const uint4* gv, const uint4* uv, const uint8_t* gs, const uint8_t* us,
                                            const void* xs, int H, const int* m_tok, int off, int ntok, int F, int f,
                                            int lane, float gsc, float* hbuf) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 4) {
            gu_group4<4, XM, SB>(gv, uv, gs, us, xs, H, m_tok, off, g0, F, f, lane, gsc, hbuf);
            g0 += 4;
        } else if (rem >= 2) {
            gu_group4<2, XM, SB>(gv, uv, gs, us, xs, H, m_tok, off, g0, F, f, lane, gsc, hbuf);
            g0 += 2;
        } else {
            gu_group4<1, XM, SB>(gv, uv, gs, us, xs, H, m_tok, off, g0, F, f, lane, gsc, hbuf);
            g0 += 1;
        }
    }
}

// Phase B: one W_d row (values + scales) against NT staged h rows (fp32).
template <int NT, int SB>
__device__ __forceinline__ void down_group4(const uint4* wv, const uint8_t* ws, const float* hs, int g, int F,
                                            int lane, float gsc, float* o_s, int obase, int RMAX,
                                            int rl) {
    float acc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.f;
    const int nv = F >> 5;
    for (int v = lane; v < nv; v += 32) {
        const uint4 w = wv[v];
        const float2 sc2 = scales32<SB>(ws, v);
        const float s0 = sc2.x, s1 = sc2.y;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float x[32];
            load_x32<X_F32_SMEM>(hs + (size_t)(g + n) * F, v, x);
            acc[n] += fp4_dot32(w, x, s0, s1);
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float sv = ft::warp_sum(acc[n]) * kSumScale * gsc;
        if (lane == 0) o_s[(size_t)(obase + g + n) * RMAX + rl] = sv;
    }
}

template <int SB>
__device__ __forceinline__ void down_row4(const uint4* wv, const uint8_t* ws, const float* hs, int ng, int F,
                                          int lane, float gsc, float* o_s, int obase, int RMAX,
                                          int rl) {
    int g = 0;
    while (g < ng) {
        const int rem = ng - g;
        if (rem >= 4) {
            down_group4<4, SB>(wv, ws, hs, g, F, lane, gsc, o_s, obase, RMAX, rl);
            g += 4;
        } else if (rem >= 2) {
            down_group4<2, SB>(wv, ws, hs, g, F, lane, gsc, o_s, obase, RMAX, rl);
            g += 2;
        } else {
            down_group4<1, SB>(wv, ws, hs, g, F, lane, gsc, o_s, obase, RMAX, rl);
            g += 1;
        }
    }
}

}  // namespace

namespace {

template <int XM, int SB>
__global__ void __launch_bounds__(THREADS, 1) expert_ffn_fp4_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_gdone;
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
    void* x_s = smem + o;
    if (XM != X_BF16_GLOBAL) o += ((size_t)T * H * (XM == X_F32_SMEM ? 4 : 2) + 127) & ~(size_t)127;
    float* o_s = reinterpret_cast<float*>(smem + o);
    o += ((size_t)TK * RMAX * 4 + 127) & ~(size_t)127;
    int* m_off = reinterpret_cast<int*>(smem + o);
    int* m_slot = m_off + TK + 1;
    int* m_tok = m_slot + TK;
    float* m_gate = reinterpret_cast<float*>(m_tok + TK);
    int* m_pos = reinterpret_cast<int*>(m_gate + TK);
    float* m_gs = reinterpret_cast<float*>(m_pos + TK);   // global scale of each entry
    int* m_fill = reinterpret_cast<int*>(m_gs + TK);      // fill index of each entry (or -1)
    o += ((size_t)(7 * TK + 1) * 4 + 127) & ~(size_t)127;
    unsigned char* ring = smem + o;
    const unsigned wpart = ((unsigned)RMAX * (dvrow + dsrow) + 127u) & ~127u;
    const void* xsrc = XM == X_BF16_GLOBAL ? static_cast<const void*>(p.x) : x_s;

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
    if (XM == X_F32_SMEM) {
        for (int i = tid; i < T * H / 8; i += THREADS) {
            float f8[8];
            ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(p.x)[i], f8);
            for (int j = 0; j < 8; ++j) f8[j] *= kActScale;
            const int t = (8 * i) / H, e = 8 * i - t * H;  // 8 values from element e of token t
            float* row = static_cast<float*>(x_s) + (size_t)t * H;
            *reinterpret_cast<float4*>(row + swz_f32(e)) = make_float4(f8[0], f8[1], f8[2], f8[3]);
            *reinterpret_cast<float4*>(row + swz_f32(e + 4)) = make_float4(f8[4], f8[5], f8[6], f8[7]);
        }
    } else if (XM == X_BF16_SMEM) {
        for (int i = tid; i < T * H / 8; i += THREADS) {
            const int t = (8 * i) / H, e = 8 * i - t * H;  // 8 values from element e of token t
            const int v = e >> 5, c = (e >> 3) & 3;
            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(x_s) + (size_t)t * H + 32 * v)[(c + v) & 3] =
                reinterpret_cast<const uint4*>(p.x)[i];
        }
    }
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
            int it = 0;
            bool ok = true;
            int waited = -1;
            for (int a = c; a < NA && ok; a += G, ++it) {
                const int st = it % nst;
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
        if (ok) gu_feature4<XM, SB>(gv, uv, gs, us, xsrc, H, m_tok, off, ntok, F, f, lane, m_gs[ent], p.hbuf);
        __syncwarp();
        if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
    }

    ft::named_bar_sync(1, CONS);
    if (tid == 0) {
        ft::grid_barrier(p.gbar, (unsigned)G, p.err);
        ft::st_release_cta(&s_gdone, 1);
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
                for (int rl = wid; rl < R && ok; rl += CW)
                    down_row4<SB>(reinterpret_cast<const uint4*>(sb + (size_t)rl * dvrow),
                              sb + (size_t)RMAX * dvrow + (size_t)rl * dsrow, hs, ng, F, lane, m_gs[e], o_s,
                              off + g0, RMAX, rl);
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

cudaError_t launch_expert_ffn_fp4(ExpertParams p, int fmt, int num_sms, cudaStream_t s) {
    if (fmt != FT_FMT_NVFP4 && fmt != FT_FMT_MXFP4) return cudaErrorInvalidValue;
    const int SB = fmt == FT_FMT_MXFP4 ? 32 : 16;
    const int G = num_sms;
    const int RMAX = (p.H + G - 1) / G;
    const size_t TK = (size_t)p.T * p.k;
    int xm = X_F32_SMEM;
    size_t xbytes = (size_t)p.T * p.H * 4;
    if (xbytes > 32768) {
        xm = X_BF16_SMEM;
        xbytes = (size_t)p.T * p.H * 2;
        if (xbytes > 32768) {
            xm = X_BF16_GLOBAL;
            xbytes = 0;
        }
    }
    const size_t head = HEAD + ((xbytes + 127) & ~(size_t)127) + ((TK * RMAX * 4 + 127) & ~(size_t)127) +
                        (((7 * TK + 1) * 4 + 127) & ~(size_t)127);
    const size_t chunk = (size_t)2 * FPC * (p.H / 2 + p.H / SB);
    const size_t wpart = ((size_t)RMAX * (p.F / 2 + p.F / SB) + 127) & ~(size_t)127;
    if (head + 2 * chunk > kSmemLimit4) return cudaErrorInvalidValue;
    // token group of phase B: as many h rows as fit next to the W_d rows in a
    // slot when two slots fill the shared memory
    int tg = (int)(((kSmemLimit4 - head - 16384) / 2 - wpart) / ((size_t)p.F * 4));
    if (tg > p.T) tg = p.T;
    if (tg > 16) tg = 16;
    if (tg < 1) return cudaErrorInvalidValue;
    size_t slot = wpart + (size_t)tg * p.F * 4;
    if (slot < chunk) slot = chunk;
    slot = (slot + 127) & ~(size_t)127;
    // The fill ring is kept small (3 x 4 KiB per SM): host reads queued beyond
    // the link's bandwidth-delay product delay every SM's HBM reads.
    const size_t fch = 4096;
    if (head + 2 * fch + 2 * slot > kSmemLimit4) return cudaErrorInvalidValue;
    int nst = (int)((kSmemLimit4 - head - 2 * fch) / slot);
    if (nst > 4) nst = 4;
    p.nstage = nst;
    p.stage_bytes = (unsigned)slot;
    p.tgroup = tg;
    int nf = (int)((kSmemLimit4 - head - slot * nst) / fch);
    if (nf > 3) nf = 3;
    p.fill_chunk = (unsigned)fch;
    p.fill_slots = nf;
    const size_t smem = head + slot * nst + (size_t)nf * fch;
    const void* fn;
    if (SB == 16)
        fn = xm == X_F32_SMEM    ? (const void*)expert_ffn_fp4_kernel<X_F32_SMEM, 16>
             : xm == X_BF16_SMEM ? (const void*)expert_ffn_fp4_kernel<X_BF16_SMEM, 16>
                                 : (const void*)expert_ffn_fp4_kernel<X_BF16_GLOBAL, 16>;
    else
        fn = xm == X_F32_SMEM    ? (const void*)expert_ffn_fp4_kernel<X_F32_SMEM, 32>
             : xm == X_BF16_SMEM ? (const void*)expert_ffn_fp4_kernel<X_BF16_SMEM, 32>
                                 : (const void*)expert_ffn_fp4_kernel<X_BF16_GLOBAL, 32>;
    static size_t smem_set[6] = {0, 0, 0, 0, 0, 0};  // per kernel variant: set only when it grows
    const int var = xm + (SB == 32 ? 3 : 0);
    if (smem > smem_set[var]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[var] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
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
