// Decode-phase kernels of the expert cache: cache fills, and the expert
// SwiGLU FFN over the resident slots merged with the CPU-set partial sum.
//
// Fill (deepmox "How residency follows demand without leaving the device"):
// for every selected miss, the complete record of its flat id is copied from
// the host pool into its victim slot, so every bank in a slot belongs to one
// layer-expert.  The victims and source rows are only known on the device, so
// the copy is device-driven: the kernel reads the page-locked host pool
// through its device mapping (NVLink-C2C on this machine) and writes HBM.
//
// Expert FFN (METAL MEDIA page, Figure 2 caption; explainer section 14):
// FFN(x) = W_d (SiLU(W_g x) * (W_u x)); y_t = sum_j g_tj FFN_{e_tj}(x_t) over
// the routes that run on the GPU, plus the supplied partial sum of the CPU set.
// Decode is bandwidth-bound (about one flop per weight byte at T = 1), so the
// layer is one persistent, cooperatively launched streaming kernel with one
// CTA per SM, and the fills the control pass left pending are performed by
// the same launch, overlapped with the resident experts' work:
//   * a producer warp streams weights into a ring of shared-memory slots with
//     1-D bulk (TMA) copies completing on mbarriers;
//   * phase A of the resident entries (gate/up + SwiGLU): items of (entry,
//     8 features); CTA c takes items c, c + G, ...; one slot holds 8 gate rows
//     and the 8 matching up rows (contiguous in the record thanks to the
//     16-row gate/up interleave); consumer warp w computes feature w of the
//     slot (both dot products, SiLU, product) and writes h in fp32;
//   * the fill copy warp copies fill items drawn from a counter of the launch
//     (each record's W_d pieces, then its gate/up units) host pool -> small
//     shared ring -> victim slot, and the fill math warp computes the SwiGLU
//     features of the units straight from the ring, so a fill's gate/up rows
//     are never read back from HBM;
//   * phase B (down + merge): CTA c owns output rows [c*H/G, (c+1)*H/G) of
//     every GPU expert, in stages of whole entries whose h rows the h warp
//     adds once they are complete (resident entries: every CTA has counted
//     its phase-A items; fills: the math warps have counted every feature,
//     and every CTA's W_d pieces of the fill are in its slot);
//     then it sums the gated expert outputs over j ascending and adds
//     partial_C, so the order of the sum is fixed and no atomics are needed.
#include "ft_common.cuh"

namespace {

constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int PRODUCER_WARP = CONSUMER_WARPS;   // TMA issue of the phase-A/B ring
constexpr int FILL_ISSUE_WARP = CONSUMER_WARPS + 1;  // fused cache fill: copies
constexpr int FILL_MATH_WARP = CONSUMER_WARPS + 2;   // fused cache fill: gate/up math
constexpr int H_WARP = CONSUMER_WARPS + 3;          // phase-B stages: h rows once complete
constexpr int EXPERT_THREADS = CONSUMERS + 4 * 32;
constexpr int FPC = CONSUMER_WARPS;             // features per phase-A chunk
constexpr size_t HEAD = 256;                    // barrier area

// ------------------------------------------------------------------- fill

__global__ void __launch_bounds__(512) fill_kernel(FillParams p) {
    const int q = p.info[INFO_Q];
    if (q <= 0) return;
    const unsigned long long n = p.rec16;
    const unsigned long long per = (n + gridDim.x - 1) / gridDim.x;
    const unsigned long long b0 = per * blockIdx.x;
    const unsigned long long b1 = b0 + per < n ? b0 + per : n;
    for (int r = 0; r < q; ++r) {
        const uint4* src = p.host_pool + (unsigned long long)p.fill_fid[r] * n;
        uint4* dst = p.slot_pool + (unsigned long long)p.fill_slot[r] * n;
        unsigned long long i = b0 + threadIdx.x;
        for (; i + 3ull * blockDim.x < b1; i += 4ull * blockDim.x) {
            uint4 v0 = src[i];
            uint4 v1 = src[i + blockDim.x];
            uint4 v2 = src[i + 2 * blockDim.x];
            uint4 v3 = src[i + 3 * blockDim.x];
            dst[i] = v0;
            dst[i + blockDim.x] = v1;
            dst[i + 2 * blockDim.x] = v2;
            dst[i + 3 * blockDim.x] = v3;
        }
        for (; i < b1; i += blockDim.x) dst[i] = src[i];
    }
}

// ------------------------------------------------------------- expert FFN

// fp32 activation rows in shared memory (x, and the h rows staged for phase
// B) swap the two 16-byte halves of every 32-byte group g with bit 2 of g set,
// so that a warp's lanes, which read consecutive groups, spread their 16-byte
// loads over all banks (no 2-way conflict).
__device__ __forceinline__ int swz8(int e) {  // element e of a row -> its stored position
    return e ^ (((e >> 5) & 1) << 2);
}

// ---- phase A inner loop: gate and up dot products of one feature over the
// K columns [k0, k0 + K) held in shared memory, for NT tokens.  x is read from
// shared memory as fp32 (XF) or bf16, row stride ldx.
template <int NT, bool XF>
__device__ __forceinline__ void gu_dots(const uint4* __restrict__ wg, const uint4* __restrict__ wu,
                                        const void* xs, const int* tk, int K, int ldx, int k0, int lane, float* ag,
                                        float* au) {
#pragma unroll
    for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
    const int nv = K >> 3;
    // several tokens already give independent chains: unroll only for few
#pragma unroll(NT >= 4 ? 1 : (NT == 2 ? 2 : 4))
    for (int v = lane; v < nv; v += 32) {
        float g8[8], u8[8];
        ft::bf16x8_to_f32(wg[v], g8);
        ft::bf16x8_to_f32(wu[v], u8);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float x8[8];
            const size_t xo = (size_t)tk[n] * ldx + k0;
            if (XF) {
                const float4* xp = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xs) + xo + v * 8);
                const int sw = ((k0 >> 3) + v) >> 2 & 1;  // halves swapped (swz8)
                const float4 x0 = xp[sw], x1 = xp[sw ^ 1];
                x8[0] = x0.x; x8[1] = x0.y; x8[2] = x0.z; x8[3] = x0.w;
                x8[4] = x1.x; x8[5] = x1.y; x8[6] = x1.z; x8[7] = x1.w;
            } else {
                ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(xs) + xo)[v],
                                  x8);
            }
            float sg = ag[n], su = au[n];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                sg = fmaf(g8[q], x8[q], sg);
                su = fmaf(u8[q], x8[q], su);
            }
            ag[n] = sg;
            au[n] = su;
        }
    }
}

// One token group of one feature.  With nseg K segments the two dot products
// are summed over the segments in order (segment sums kept per token in facc,
// by the lane that owns the token), and SwiGLU is applied after the last one.
template <int NT, bool XF>
__device__ __forceinline__ void gu_group(const uint4* wg, const uint4* wu, const void* xs, const int* m_tok, int off,
                                         int g0, int K, int H, int k0, int F, int f, int lane, float* hbuf, int seg,
                                         int nseg, float* facc) {
    int tk[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) tk[n] = m_tok[off + g0 + n];
    float ag[NT], au[NT];
    gu_dots<NT, XF>(wg, wu, xs, tk, K, H, k0, lane, ag, au);
    float mg = 0.f, mu = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float sg = ft::warp_sum(ag[n]);
        const float su = ft::warp_sum(au[n]);
        if (lane == n) {
            mg = sg;
            mu = su;
        }
    }
    if (lane < NT) {
        if (nseg > 1) {
            float* a = facc + 2 * (g0 + lane);
            if (seg > 0) {
                mg += a[0];
                mu += a[1];
            }
            if (seg < nseg - 1) {
                a[0] = mg;
                a[1] = mu;
                return;
            }
        }
        hbuf[(size_t)(off + g0 + lane) * F + swz8(f)] = ft::silu_mul(mg, mu);
    }
}

// Out of line: one copy serves the consumer warps and the fill math warp,
// which keeps the kernel's hot code small enough for the instruction cache.
template <bool XF>
__device__ __noinline__ void gu_feature(const uint4* wg, const uint4* wu, const void* xs, const int* m_tok,
                                           int off, int ntok, int K, int H, int k0, int F, int f, int lane,
                                           float* hbuf, int seg = 0, int nseg = 1, float* facc = nullptr) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 4) {
            gu_group<4, XF>(wg, wu, xs, m_tok, off, g0, K, H, k0, F, f, lane, hbuf, seg, nseg, facc);
            g0 += 4;
        } else if (rem >= 2) {
            gu_group<2, XF>(wg, wu, xs, m_tok, off, g0, K, H, k0, F, f, lane, hbuf, seg, nseg, facc);
            g0 += 2;
        } else {
            gu_group<1, XF>(wg, wu, xs, m_tok, off, g0, K, H, k0, F, f, lane, hbuf, seg, nseg, facc);
            g0 += 1;
        }
    }
}

// ---- phase B inner loop: the rows rb + rs * i (i < 4, row < R) of one
// entry's W_d block in shared memory against NT token rows of h (fp32, shared
// memory).  Each column chunk of h is read once and applied to all the rows
// of the warp, which gives independent accumulation chains.
template <int NT>
__device__ __forceinline__ void down_group(uint32_t wbase, uint32_t hs, int g0, int F, int R, int rb, int rs,
                                           int lane, float* o_s, int obase, int RMAX) {
    float acc[4][NT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[r][n] = 0.f;
    const int nv = F >> 3;
    for (int v = lane; v < nv; v += 32) {
        float hv[NT][8];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint32_t hp = hs + ((uint32_t)(g0 + n) * F + v * 8) * 4u;
            const uint32_t sw = (uint32_t)(v >> 2 & 1) * 16u;  // halves swapped (swz8)
            const float4 x0 = ft::lds128f(hp + sw), x1 = ft::lds128f(hp + (16u - sw));
            hv[n][0] = x0.x; hv[n][1] = x0.y; hv[n][2] = x0.z; hv[n][3] = x0.w;
            hv[n][4] = x1.x; hv[n][5] = x1.y; hv[n][6] = x1.z; hv[n][7] = x1.w;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int rl = rb + r * rs;
            if (rl < R) {
                float w8[8];
                ft::bf16x8_to_f32(ft::lds128(wbase + (uint32_t)rl * F * 2 + v * 16), w8);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float s2 = acc[r][n];
#pragma unroll
                    for (int q = 0; q < 8; ++q) s2 = fmaf(w8[q], hv[n][q], s2);
                    acc[r][n] = s2;
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int rl = rb + r * rs;
        if (rl < R) {  // warp-uniform
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float sv = ft::warp_sum(acc[r][n]);
                if (lane == 0) o_s[(size_t)(obase + g0 + n) * RMAX + rl] = sv;
            }
        }
    }
}

// The rows wi, wi + nw, wi + 2 nw, ... (< R) of one entry -- this warp is the
// wi-th of the nw warps serving the entry -- NT tokens at a time.  Out of
// line, like gu_feature, to keep the hot code small; W_d rows and h by shared
// address.
__device__ __noinline__ void down_entry(uint32_t wbase, uint32_t hs, int ntok, int F, int R, int wi, int nw,
                                        int lane, float* o_s, int obase, int RMAX) {
    for (int rb = wi; rb < R; rb += 4 * nw) {
        int g0 = 0;
        while (g0 < ntok) {
            const int rem = ntok - g0;
            if (rem >= 4) {
                down_group<4>(wbase, hs, g0, F, R, rb, nw, lane, o_s, obase, RMAX);
                g0 += 4;
            } else if (rem >= 2) {
                down_group<2>(wbase, hs, g0, F, R, rb, nw, lane, o_s, obase, RMAX);
                g0 += 2;
            } else {
                down_group<1>(wbase, hs, g0, F, R, rb, nw, lane, o_s, obase, RMAX);
                g0 += 1;
            }
        }
    }
}

__global__ void __launch_bounds__(EXPERT_THREADS, 1) expert_ffn_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_fitem[8], s_fsub[8];  // fill ring: item and K segment of the chunk in each slot (-1: end)
    __shared__ int s_armed;  // ring steps armed by the producer (-1 after a failure)
    const int H = p.H, F = p.F, T = p.T, k = p.k;
    const int nst = p.nstage;
    const unsigned slot_bytes = p.stage_bytes;
    const int ugpu = p.info[INFO_UGPU];
    const int nasg = p.info[INFO_NASSIGN];
    const int q = p.do_fill ? p.info[INFO_Q] : 0;  // fills performed here: the last q entries
    const int nA = ugpu - q;                        // entries streamed from their slots in phase A
    const int G = gridDim.x, c = blockIdx.x;
    const int cpe = F / FPC;  // phase-A chunks per expert
    const int NA = nA * cpe;
    const int r0 = (int)((long long)H * c / G), r1 = (int)((long long)H * (c + 1) / G);
    const int R = r1 - r0;
    const int RMAX = (H + G - 1) / G;
    const int nB = R > 0 ? ugpu : 0;
    const int TK = T * k;

    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + nst;
    uint64_t* ffull = reinterpret_cast<uint64_t*>(smem + 128);  // fill ring: chunk landed
    uint64_t* fcons = ffull + 4;                                 // fill ring: chunk's features computed
    const bool xf32 = (size_t)T * H * 4 <= 65536;  // x kept as fp32 in shared memory
    const size_t xbytes = (size_t)T * H * (xf32 ? 4 : 2);
    size_t o = HEAD;
    void* x_s = smem + o;
    o += (xbytes + 127) & ~(size_t)127;
    float* o_s = reinterpret_cast<float*>(smem + o);  // [T*k][RMAX] expert outputs of my rows
    o += ((size_t)TK * RMAX * 4 + 127) & ~(size_t)127;
    // worklist metadata, staged once
    int* m_off = reinterpret_cast<int*>(smem + o);    // [TK+1] entry offsets (ugpu+1 used)
    int* m_slot = m_off + TK + 1;                      // [TK]   entry slots (ugpu used)
    int* m_tok = m_slot + TK;                          // [TK]   token of each assignment
    float* m_gate = reinterpret_cast<float*>(m_tok + TK);  // [TK]
    int* m_pos = reinterpret_cast<int*>(m_gate + TK);      // [TK]   assignment of (t, j)
    o += ((size_t)(5 * TK + 1) * 4 + 127) & ~(size_t)127;
    float* facc = reinterpret_cast<float*>(smem + o);      // [T][2] segment sums of the fill math warp
    o += ((size_t)2 * T * 4 + 127) & ~(size_t)127;
    unsigned char* ring = smem + o;
    unsigned char* fring = ring + (size_t)nst * slot_bytes;
    const unsigned rowbytes = (unsigned)H * 2u;
    // phase-B stage: consecutive entries, each its W_d rows [r0, r1) then its
    // h rows, as many as fit in a slot (a stage never mixes resident entries
    // and fills, whose W_d rows this CTA stores itself)
    const unsigned wpad = ((unsigned)R * F * 2u + 127u) & ~127u;
    auto hbytes = [&](int e) { return (unsigned)(m_off[e + 1] - m_off[e]) * F * 4u; };
    auto stage_end = [&](int e0) {
        unsigned used = 0;
        int e1 = e0;
        while (e1 < nB) {
            const unsigned need = wpad + ((hbytes(e1) + 127u) & ~127u);
            if (e1 > e0 && (used + need > slot_bytes || e1 == nA)) break;
            used += need;
            ++e1;
        }
        return e1;
    };
    // One ring sequence for the producer, the h warp and the consumers: the
    // phase-A items c, c + G, ..., then the phase-B stages.
    auto stage_due = [&](int a, int e0) { return e0 < nB && a >= NA; };
    // h of the resident entries is complete once every CTA has counted its
    // phase-A items in hits_done; h of fill r once the math warps have counted
    // its F features in ready[r]
    unsigned* hits_done = p.gbar + 1;
    // Exit count: the consumers, the fill copy warp and the fill math warp of
    // every CTA each count out once they are done with the counters; whoever
    // completes the count returns the counters to zero for the next launch.
    auto count_out = [&]() {
        unsigned n;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(n) : "l"(p.gbar) : "memory");
        if (n == 3u * (unsigned)G - 1u) {
            for (int e = 0; e < ugpu; ++e) p.ready[e] = 0u;
            for (int r = 0; r < q; ++r) p.wdc[r] = 0u;
            p.gbar[2] = 0u;
            p.gbar[1] = 0u;
            p.gbar[0] = 0u;
        }
    };

    // fused-fill geometry.  Each fill record is cut into items: first its
    // W_d block in pieces of one ring chunk (NWD items), then its gate/up rows
    // in units of fpf features (upr items), a unit split into nks chunks of
    // KS columns.  The CTAs' copy warps draw items from one counter of the
    // launch (fill 0's items first), so a CTA whose host reads return sooner
    // copies more, and every CTA finishes its part at about the same time.
    const int nf = p.fill_slots;
    const unsigned fch = p.fill_chunk;
    const int fpf = p.fill_fpf, nks = p.fill_nks;
    const int KS = H / nks;
    const int upr = F / fpf;
    const unsigned long long wdt = (unsigned long long)H * F * 2;  // W_d bytes of a record
    const int NWD = (int)((wdt + fch - 1) / fch);
    const int ipf = NWD + upr;  // items per fill
    const int n_items = q * ipf;
    const unsigned partb = (unsigned)fpf * KS * 2u;  // gate (or up) bytes of one unit chunk
    // The fill copy warp owns its ring barriers and slot tags and starts at once;
    // the other warps stage the worklist and x meanwhile.  Named barrier 3:
    // the copy warp arrives once its state is initialised, the rest sync.
    if (wid == FILL_ISSUE_WARP) {
        if (lane == 0) {
            for (int s = 0; s < nf; ++s) {
                // one cp.async arrival per lane of the copy warp, and lane 0's
                // arrival that publishes the slot's tag
                ft::mbar_init(&ffull[s], 33);
                ft::mbar_init(&fcons[s], 1);
            }
            ft::mbar_fence_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 3, %0;" ::"n"(EXPERT_THREADS) : "memory");
    } else {
        if (tid == 0) {
            for (int s = 0; s < nst; ++s) {
                ft::mbar_init(&full[s], 1);
                ft::mbar_init(&empty[s], CONSUMER_WARPS);
            }
            ft::mbar_fence_init();
            s_armed = 0;
        }
        constexpr int NS = EXPERT_THREADS - 32;  // staging threads: every warp but the copy warp
        const int st0 = wid < FILL_ISSUE_WARP ? tid : tid - 32;
        for (int i = st0; i <= ugpu; i += NS) m_off[i] = p.wl_off[i];
        for (int i = st0; i < ugpu; i += NS) m_slot[i] = p.wl_slot[i];
        for (int i = st0; i < nasg; i += NS) {
            m_tok[i] = p.as_tok[i];
            m_gate[i] = p.as_gate[i];
        }
        for (int i = st0; i < TK; i += NS) m_pos[i] = p.out_pos[i];
        if (xf32) {
            for (int i = st0; i < T * H / 8; i += NS) {
                float f8[8];
                ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(p.x)[i], f8);
                const int sw = (i >> 2) & 1;  // halves swapped (swz8); rows start at multiples of 8 groups
                reinterpret_cast<float4*>(x_s)[2 * i + sw] = make_float4(f8[0], f8[1], f8[2], f8[3]);
                reinterpret_cast<float4*>(x_s)[2 * i + (sw ^ 1)] = make_float4(f8[4], f8[5], f8[6], f8[7]);
            }
        } else {
            for (int i = st0; i < (int)(xbytes / 16); i += NS)
                reinterpret_cast<uint4*>(x_s)[i] = reinterpret_cast<const uint4*>(p.x)[i];
        }
        ft::named_bar_sync(3, EXPERT_THREADS);
    }

    // ------------------------------------------------- fused fill: copy warp
    // host pool -> fill ring by per-lane cp.async (the load/store path, so the
    // slow host reads do not queue ahead of the ring's bulk copies from HBM),
    // then fill ring -> victim slot by one bulk store.  A chunk is released
    // for the next load once the math warp has used it and its store has read
    // it.  Lane 0 draws the next item one ahead, so the counter's latency
    // overlaps the chunks in flight.  The W_d pieces a CTA stored are
    // published in wdc[r] (GPU scope, after their stores complete) when its
    // sequence moves past them; the producers of every CTA wait for the
    // count before reading their W_d rows of the fill from its slot.
    if (wid == FILL_ISSUE_WARP) {
        const uint8_t* host = reinterpret_cast<const uint8_t*>(p.host_pool);
        uint8_t* pool = const_cast<uint8_t*>(p.slot_pool);
        const unsigned long long wd0 = (unsigned long long)4 * F * H;
        const unsigned long long upoff = (unsigned long long)16 * H * 2;  // up rows follow gate rows by 16 rows
        // offset within the record and bytes of one part of chunk (item, seg)
        auto locate = [&](int item, int seg, unsigned long long& off, unsigned& n) {
            const int li = item % ipf;
            if (li >= NWD) {
                const int f0 = (li - NWD) * fpf;
                const unsigned long long row = (unsigned long long)(f0 >> 4) * 32 + (f0 & 15);
                off = (row * H + (unsigned long long)seg * KS) * 2;
                n = partb;
            } else {
                const unsigned long long po = (unsigned long long)li * fch;
                off = wd0 + po;
                n = (unsigned)(wdt - po < fch ? wdt - po : fch);
            }
        };
        // CTA c takes item c first; every later item is drawn from the
        // counter (values from G on) right after the current item's first
        // chunk is issued, and read when that item is exhausted.
        unsigned* claims = p.gbar + 2;
        // the first fill's record, loaded beside the fill count rather than
        // after it (launches that perform fills have the array; unused when q = 0)
        const int fid0 = p.do_fill ? p.fill_fid[0] : 0;
        int ahead = 0;  // lane 0: the draw in flight
        int nxt = c;    // the next item to start, once `known`
        bool known = true;
        int cur = -1, sub = 0, nsub = 0;
        bool more = true;
        auto load = [&](int s) {  // all lanes: the next chunk into slot s, or the end tag
            bool started = false;
            if (more && sub == nsub) {
                if (!known) nxt = G + __shfl_sync(0xffffffffu, ahead, 0);
                if (nxt >= n_items) {
                    more = false;
                } else {
                    cur = nxt;
                    sub = 0;
                    nsub = cur % ipf < NWD ? 1 : nks;
                    known = false;
                    started = true;
                }
            }
            if (!more) {
                if (lane == 0) {
                    s_fitem[s] = -1;
                    ft::mbar_arrive(&ffull[s]);
                }
                ft::cp_async_arrive(&ffull[s]);
                return;
            }
            const int seg = sub++;
            unsigned long long off;
            unsigned n;
            locate(cur, seg, off, n);
            unsigned char* d = fring + (size_t)s * fch;
            const int fr = cur / ipf;
            const uint8_t* src = host + (unsigned long long)(fr == 0 ? fid0 : p.fill_fid[fr]) * p.rb + off;
            for (unsigned v = lane * 16u; v < n; v += 512u) ft::cp_async16(d + v, src + v);
            if (cur % ipf >= NWD)
                for (unsigned v = lane * 16u; v < n; v += 512u) ft::cp_async16(d + n + v, src + upoff + v);
            if (lane == 0) {
                s_fitem[s] = cur;
                s_fsub[s] = seg;
                ft::mbar_arrive(&ffull[s]);
                if (started) ahead = (int)atomicAdd(claims, 1u);
            }
            ft::cp_async_arrive(&ffull[s]);
        };
        auto store = [&](int item, int seg, int s) {  // lane 0
            unsigned long long off;
            unsigned n;
            locate(item, seg, off, n);
            const unsigned char* d = fring + (size_t)s * fch;
            uint8_t* dst = pool + (unsigned long long)p.fill_slot[item / ipf] * p.rb + off;
            ft::bulk_s2g(dst, d, n);
            if (item % ipf >= NWD) ft::bulk_s2g(dst + upoff, d + n, n);
            ft::bulk_commit();
        };
        auto publish_wd = [&](int r, int n) {  // lane 0
            ft::bulk_wait_all();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            ft::red_release_gpu_add(&p.wdc[r], (unsigned)n);
        };
        // prime the ring; `more` turns false once the end tag is in it
        int issued = 0;
        do load(issued++);
        while (issued < nf && more);
        int pend_r = 0, pend_n = 0;  // lane 0: W_d pieces stored, not yet published
        for (int g = 0; g < issued; ++g) {
            const int s = g % nf;
            const uint32_t par = (uint32_t)(g / nf) & 1u;
            int item = -1, w = 1;
            if (lane == 0) {
                item = s_fitem[s];
                if (item >= 0) {
                    w = ft::mbar_wait(&ffull[s], par, p.err, p.wait_ns);
                    if (w) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // cp.async data -> bulk store
                        store(item, s_fsub[s], s);
                        if (item % ipf < NWD) {
                            pend_r = item / ipf;
                            ++pend_n;
                            const int nx = s_fitem[(g + 1) % nf];  // the next chunk of this CTA, or the end tag
                            if (nx < 0 || nx / ipf != pend_r || nx % ipf >= NWD) {
                                publish_wd(pend_r, pend_n);
                                pend_n = 0;
                            }
                        }
                        w = ft::mbar_wait(&fcons[s], par, p.err, p.wait_ns);
                        ft::bulk_wait_read_all();
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, item, 0) < 0) break;  // the end tag
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            if (more) {
                load(s);
                ++issued;
            }
        }
        ft::cp_async_wait_all();  // nothing in flight into shared memory at exit
        __syncwarp();
        if (lane == 0) {
            ft::bulk_wait_all();
            count_out();
        }
        return;
    }

    // ------------------------------------------ fused fill: gate/up math warp
    // SwiGLU features of the fill units this CTA copied, from the fill ring,
    // in the copy warp's order, up to its end tag.
    if (wid == FILL_MATH_WARP) {
        for (int g = 0;; ++g) {
            const int s = g % nf;
            if (!__all_sync(0xffffffffu, ft::mbar_wait(&ffull[s], (uint32_t)(g / nf) & 1u, p.err, p.wait_ns))) break;
            const int item = s_fitem[s];
            if (item < 0) break;
            const int r = item / ipf, li = item - r * ipf;
            if (li < NWD) {  // a W_d piece: acknowledged so the ring cannot lap this warp
                __syncwarp();
                if (lane == 0) ft::mbar_arrive(&fcons[s]);
                continue;
            }
            const int seg = s_fsub[s];
            const int f0 = (li - NWD) * fpf;
            const int off = m_off[nA + r];
            const int ntok = m_off[nA + r + 1] - off;
            const unsigned char* d = fring + (size_t)s * fch;
            for (int fi = 0; fi < fpf; ++fi) {
                const uint4* wg = reinterpret_cast<const uint4*>(d + (size_t)fi * KS * 2);
                const uint4* wu = reinterpret_cast<const uint4*>(d + partb + (size_t)fi * KS * 2);
                if (xf32)
                    gu_feature<true>(wg, wu, x_s, m_tok, off, ntok, KS, H, seg * KS, F, f0 + fi, lane, p.hbuf, seg,
                                     nks, facc);
                else
                    gu_feature<false>(wg, wu, x_s, m_tok, off, ntok, KS, H, seg * KS, F, f0 + fi, lane, p.hbuf, seg,
                                      nks, facc);
            }
            __syncwarp();
            if (lane == 0) {
                ft::mbar_arrive(&fcons[s]);
                if (seg == nks - 1) ft::red_release_gpu_add(&p.ready[nA + r], (unsigned)fpf);
            }
        }
        __syncwarp();
        if (lane == 0) count_out();  // after the last release
        return;
    }

    // -------------------------------------------------------------- h warp
    // For each phase-B stage armed by the producer: the h rows of each entry,
    // once every feature of it is written (by whichever CTA computed it).
    // After a timed-out wait the rows are still copied (whatever they hold)
    // so that the stage completes and the ring drains.
    if (wid == H_WARP) {
        if (lane == 0) {
            for (int a = c, e0 = 0, it = 0;; ++it) {
                const bool isB = stage_due(a, e0);
                if (!isB && a >= NA) break;
                if (!isB) {
                    a += G;
                    continue;
                }
                const int e1 = stage_end(e0);
                const uint64_t t0 = ft::globaltimer();
                int armed;
                while ((armed = ft::ld_acquire_cta(&s_armed)) >= 0 && armed <= it) {
                    __nanosleep(128);  // leave the issue slots to the consumer warps
                    if (ft::globaltimer() - t0 > p.wait_ns) {
                        atomicOr(p.err, FT_DEVERR_TIMEOUT);
                        armed = -1;
                        break;
                    }
                }
                if (armed < 0) break;
                const int st = it % nst;
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                unsigned o = 0;
                for (int e = e0; e < e1; ++e) {
                    if (e < nA)
                        ft::wait_count(hits_done, (unsigned)G, p.err, p.wait_ns);
                    else
                        ft::wait_count(&p.ready[e], (unsigned)F, p.err, p.wait_ns);
                    ft::bulk_g2s(dst + o + wpad, p.hbuf + (size_t)m_off[e] * F, hbytes(e), &full[st]);
                    o += wpad + ((hbytes(e) + 127u) & ~127u);
                }
                e0 = e1;
            }
        }
        return;
    }

    // ------------------------------------------------------------ producer
    if (wid == PRODUCER_WARP) {
        if (lane == 0) {
            const uint64_t pol = ft::l2_policy_evict_first();
            const unsigned wb = (unsigned)R * F * 2u;
            // W_d rows of the resident entries go to L2 while phase A streams
            auto prefetch_wd = [&]() {
                for (int e = 0; e < nA && wb > 0; ++e)
                    ft::bulk_prefetch_l2(p.slot_pool + (size_t)m_slot[e] * p.rb + (size_t)4 * F * H + (size_t)r0 * F * 2,
                                         wb);
            };
            int it = 0;
            bool ok = true;
            for (int a = c, e0 = 0; ok; ++it) {
                const bool isB = stage_due(a, e0);
                if (!isB && a >= NA) break;
                const int st = it % nst;
                if (it == nst) prefetch_wd();
                if (it >= nst && !ft::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err, p.wait_ns)) { ok = false; break; }
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                if (!isB) {
                    const int ent = a / cpe;
                    const int f0 = (a - ent * cpe) * FPC;
                    const uint8_t* rec = p.slot_pool + (size_t)m_slot[ent] * p.rb;
                    const int grp = f0 >> 4, i = f0 & 15;
                    ft::mbar_arrive_expect_tx(&full[st], 2u * FPC * rowbytes);
                    ft::bulk_g2s_hint(dst, rec + (size_t)(grp * 32 + i) * rowbytes, FPC * rowbytes, &full[st], pol);
                    ft::bulk_g2s_hint(dst + (size_t)FPC * rowbytes, rec + (size_t)(grp * 32 + 16 + i) * rowbytes,
                                      FPC * rowbytes, &full[st], pol);
                    a += G;
                    continue;
                }
                // phase-B stage: the W_d rows of its entries (those of a fill
                // once every piece of its W_d block is in the slot), then the
                // h rows of each entry once every feature of it is written
                const int e1 = stage_end(e0);
                for (int e = e0 > nA ? e0 : nA; e < e1 && ok; ++e)
                    ok = ft::wait_count(&p.wdc[e - nA], (unsigned)NWD, p.err, p.wait_ns);
                if (!ok) break;
                unsigned tx = 0;
                for (int e = e0; e < e1; ++e) tx += wb + hbytes(e);
                ft::mbar_arrive_expect_tx(&full[st], tx);
                unsigned o = 0;
                for (int e = e0; e < e1; ++e) {
                    const uint8_t* wd = p.slot_pool + (size_t)m_slot[e] * p.rb + (size_t)4 * F * H + (size_t)r0 * F * 2;
                    ft::bulk_g2s_hint(dst + o, wd, wb, &full[st], pol);
                    o += wpad + ((hbytes(e) + 127u) & ~127u);
                }
                ft::st_release_cta(&s_armed, it + 1);  // the h warp adds the h rows
                e0 = e1;
            }
            if (!ok) ft::st_release_cta(&s_armed, -1);
            if (it <= nst) prefetch_wd();
            ft::drain_ring(full, it, nst, p.err);
        }
        return;
    }

    // ------------------------------- consumers: phase-A items and phase-B stages
    // After a failed (timed-out) wait a warp stops waiting, computing and
    // releasing slots, but keeps the same barrier sequence as the others.
    int it = 0;
    bool failed = false;
    if (c >= NA && tid == 0) ft::red_release_gpu_add(hits_done, 1u);
    for (int a = c, e0 = 0;; ++it) {
        const bool isB = stage_due(a, e0);
        if (!isB && a >= NA) break;
        const int st = it % nst;
        const bool ok = !failed && __all_sync(0xffffffffu, ft::mbar_wait(&full[st], (it / nst) & 1, p.err, p.wait_ns));
        failed = !ok;
        const unsigned char* sb = ring + (size_t)st * slot_bytes;
        if (!isB) {
            // gate/up + SwiGLU: warp w computes feature w of the item
            const int ent = a / cpe;
            const int f = (a - ent * cpe) * FPC + wid;
            const int off = m_off[ent];
            const int ntok = m_off[ent + 1] - off;
            const uint4* wg = reinterpret_cast<const uint4*>(sb + (size_t)wid * rowbytes);
            const uint4* wu = reinterpret_cast<const uint4*>(sb + (size_t)(FPC + wid) * rowbytes);
            if (ok) {
                if (xf32)
                    gu_feature<true>(wg, wu, x_s, m_tok, off, ntok, H, H, 0, F, f, lane, p.hbuf);
                else
                    gu_feature<false>(wg, wu, x_s, m_tok, off, ntok, H, H, 0, F, f, lane, p.hbuf);
            }
            __syncwarp();
            if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
            a += G;
            if (a >= NA) {  // this CTA's h of the resident entries is written
                ft::named_bar_sync(2, CONSUMERS);
                if (tid == 0) ft::red_release_gpu_add(hits_done, 1u);
            }
            continue;
        }
        // down rows [r0, r1) of the stage's entries.  The warps split over the
        // entries so that they proceed at the same time: with cls = min(ne, 8)
        // classes, warp w serves the entries e0 + (w mod cls) + j cls, as the
        // (w / cls)-th of the nw warps of its class.
        const int e1 = stage_end(e0);
        if (ok) {
            const int ne = e1 - e0;
            const int cls = ne < CONSUMER_WARPS ? ne : CONSUMER_WARPS;
            const int my = wid % cls, wi = wid / cls;
            const int nw = (CONSUMER_WARPS - my + cls - 1) / cls;
            unsigned so = 0;
            int e = e0;
            for (; e < e0 + my; ++e) so += wpad + ((hbytes(e) + 127u) & ~127u);
            while (e < e1) {
                const int off = m_off[e];
                const unsigned char* eb = sb + so;
                down_entry(ft::smem_addr(eb), ft::smem_addr(eb + wpad), m_off[e + 1] - off, F, R, wi, nw, lane, o_s,
                           off, RMAX);
                for (int n = 0; n < cls && e < e1; ++n, ++e) so += wpad + ((hbytes(e) + 127u) & ~127u);
            }
        }
        __syncwarp();
        if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
        e0 = e1;
    }
    ft::named_bar_sync(1, CONSUMERS);
    // gated merge in fixed order: j ascending, then the CPU-set partial sum
    for (int idx = tid; idx < T * R; idx += CONSUMERS) {
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
    // every read of the counters by this CTA's consumers, producer and h warp
    // precedes the end of its phase B
    ft::named_bar_sync(1, CONSUMERS);
    if (tid == 0) count_out();
}

}  // namespace

cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s) {
    fill_kernel<<<grid, 512, 0, s>>>(p);
    return cudaGetLastError();
}

static constexpr size_t kSmemLimit = 227 * 1024 - 256;  // dynamic; the rest is static shared memory
static constexpr size_t kFillChunk = 4096;               // bytes of one fused-fill ring chunk
static constexpr int kFillSlots = 3;                     // fused-fill ring chunks per CTA

// Shared-memory plan: barriers, x (if it fits in 64 KiB), the per-CTA output
// block, the worklist metadata and the fill math warp's segment sums, then the
// ring (as many slots as fit, at most 4) and the fused-fill ring.  A ring slot
// holds one phase-A chunk (16 rows of H) or one phase-B stage (R rows of W_d
// followed by the h rows of the entry's tokens).  The fill ring has 3 chunks
// of 4 KiB; a fill unit chunk holds the gate and up rows of fpf features, or
// of one feature over H / nks columns when one feature does not fit.
struct Bf16Plan {
    size_t smem, slot;
    int nstage, fpf, nks;
};

static bool bf16_plan(int H, int F, int T, int k, int G, Bf16Plan& pl) {
    const int RMAX = (H + G - 1) / G;
    const bool xf32 = (size_t)T * H * 4 <= 65536;
    const size_t xbytes = (size_t)T * H * (xf32 ? 4 : 2);
    const size_t TK = (size_t)T * k;
    const size_t head = HEAD + ((xbytes + 127) & ~(size_t)127) + ((TK * RMAX * 4 + 127) & ~(size_t)127) +
                        (((5 * TK + 1) * 4 + 127) & ~(size_t)127) + (((size_t)2 * T * 4 + 127) & ~(size_t)127);
    size_t slot = (size_t)2 * FPC * H * 2;
    const size_t down = (((size_t)RMAX * F * 2 + 127) & ~(size_t)127) + (size_t)T * F * 4;
    if (down > slot) slot = down;
    slot = (slot + 127) & ~(size_t)127;
    // The fill ring is deliberately small: the host link's bandwidth-delay
    // product is well under 1 MB, and host reads queued beyond it delay the
    // HBM reads of every other SM behind them in the memory system.
    const size_t fch = kFillChunk;
    const int nf = kFillSlots;
    if (head >= kSmemLimit || head + nf * fch + 2 * slot > kSmemLimit) return false;
    int nst = (int)((kSmemLimit - head - nf * fch) / slot);
    if (nst > 4) nst = 4;
    // fill unit: fpf whole features (a power of two up to 16, so a unit stays
    // inside one 16-row gate/up group), or one feature in nks K segments
    int fpf = 1, nks = 1;
    while (4ull * H * (2 * fpf) <= fch && 2 * fpf <= 16) fpf *= 2;
    while (4ull * (H / nks) > fch) nks *= 2;
    if (H % nks || (H / nks) % 8) return false;
    pl.smem = head + slot * nst + (size_t)nf * fch;
    pl.slot = slot;
    pl.nstage = nst;
    pl.fpf = fpf;
    pl.nks = nks;
    return true;
}

bool expert_ffn_fits(int H, int F, int T, int k, int num_sms) {
    Bf16Plan pl;
    return bf16_plan(H, F, T, k, num_sms, pl);
}

cudaError_t launch_expert_ffn(ExpertParams p, int num_sms, cudaStream_t s) {
    const int G = num_sms;
    if (p.wait_ns == 0) p.wait_ns = FT_WAIT_LIMIT_NS;
    Bf16Plan pl;
    if (!bf16_plan(p.H, p.F, p.T, p.k, G, pl)) return cudaErrorInvalidValue;
    p.nstage = pl.nstage;
    p.stage_bytes = (unsigned)pl.slot;
    p.fill_chunk = (unsigned)kFillChunk;
    p.fill_slots = kFillSlots;
    p.fill_fpf = pl.fpf;
    p.fill_nks = pl.nks;
    const size_t smem = pl.smem;
    cudaError_t e = ensure_dynamic_smem((const void*)expert_ffn_kernel, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(EXPERT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, expert_ffn_kernel, p);
}
