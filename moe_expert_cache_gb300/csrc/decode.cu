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
// CTA per SM:
//   * a producer warp streams weights into a ring of shared-memory slots with
//     1-D bulk (TMA) copies completing on mbarriers;
//   * phase A (gate/up + SwiGLU): the work is the flat list of (GPU expert,
//     group of 8 features), hits first, then the fills in fill order; CTA c
//     takes items c, c + G, ...; one slot holds
//     8 gate rows and the 8 matching up rows (contiguous in the record thanks
//     to the 16-row gate/up interleave); consumer warp w computes feature w of
//     the slot alone (both dot products, SiLU, product) and writes h in fp32;
//   * a grid barrier makes every h visible; the producer does not wait for it
//     and keeps streaming the W_d rows of phase B meanwhile;
//   * phase B (down + merge): CTA c owns output rows [c*H/G, (c+1)*H/G) of
//     every GPU expert; then it sums the gated expert outputs over j ascending
//     and adds partial_C, so the order of the sum is fixed and no atomics are
//     needed.
#include "ft_common.cuh"

namespace {

constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int FILL_WARPS = 1;                   // fused cache fill (one TMA thread)
constexpr int EXPERT_THREADS = CONSUMERS + 32 + FILL_WARPS * 32;  // + producer warp + fill warps
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

// ---- phase A inner loop: gate and up dot products of one feature (full K)
// for NT tokens.  x is read from shared memory as fp32 (XF) or bf16.
template <int NT, bool XF>
__device__ __forceinline__ void gu_dots(const uint4* __restrict__ wg, const uint4* __restrict__ wu,
                                        const void* xs, const int* tk, int H, int lane, float* ag, float* au) {
#pragma unroll
    for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
    const int nv = H >> 3;
#pragma unroll 4
    for (int v = lane; v < nv; v += 32) {
        float g8[8], u8[8];
        ft::bf16x8_to_f32(wg[v], g8);
        ft::bf16x8_to_f32(wu[v], u8);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float x8[8];
            if (XF) {
                const float4* xp = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xs) +
                                                                   (size_t)tk[n] * H + v * 8);
                const float4 x0 = xp[0], x1 = xp[1];
                x8[0] = x0.x; x8[1] = x0.y; x8[2] = x0.z; x8[3] = x0.w;
                x8[4] = x1.x; x8[5] = x1.y; x8[6] = x1.z; x8[7] = x1.w;
            } else {
                ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(xs) +
                                                                 (size_t)tk[n] * H)[v], x8);
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

template <int NT, bool XF>
__device__ __forceinline__ void gu_group(const uint4* wg, const uint4* wu, const void* xs, const int* m_tok, int off,
                                         int g0, int H, int F, int f, int lane, float* hbuf) {
    int tk[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) tk[n] = m_tok[off + g0 + n];
    float ag[NT], au[NT];
    gu_dots<NT, XF>(wg, wu, xs, tk, H, lane, ag, au);
    float mine = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float sg = ft::warp_sum(ag[n]);
        const float su = ft::warp_sum(au[n]);
        if (lane == n) mine = ft::silu_mul(sg, su);
    }
    if (lane < NT) hbuf[(size_t)(off + g0 + lane) * F + f] = mine;
}

template <bool XF>
__device__ __forceinline__ void gu_feature(const uint4* wg, const uint4* wu, const void* xs, const int* m_tok,
                                           int off, int ntok, int H, int F, int f, int lane, float* hbuf) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 8) {
            gu_group<8, XF>(wg, wu, xs, m_tok, off, g0, H, F, f, lane, hbuf);
            g0 += 8;
        } else if (rem >= 4) {
            gu_group<4, XF>(wg, wu, xs, m_tok, off, g0, H, F, f, lane, hbuf);
            g0 += 4;
        } else if (rem >= 2) {
            gu_group<2, XF>(wg, wu, xs, m_tok, off, g0, H, F, f, lane, hbuf);
            g0 += 2;
        } else {
            gu_group<1, XF>(wg, wu, xs, m_tok, off, g0, H, F, f, lane, hbuf);
            g0 += 1;
        }
    }
}

// ---- phase B inner loop: one W_d row against NT token rows of h (fp32, smem)
template <int NT>
__device__ __forceinline__ void down_group(const uint4* __restrict__ wrow, const float* hs, int g0, int F, int lane,
                                           float* o_s, int obase, int RMAX, int rl) {
    float acc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.f;
    const int nv = F >> 3;
#pragma unroll 3
    for (int v = lane; v < nv; v += 32) {
        float w8[8];
        ft::bf16x8_to_f32(wrow[v], w8);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const float4* hp = reinterpret_cast<const float4*>(hs + (size_t)(g0 + n) * F + v * 8);
            const float4 x0 = hp[0], x1 = hp[1];
            float s = acc[n];
            s = fmaf(w8[0], x0.x, s);
            s = fmaf(w8[1], x0.y, s);
            s = fmaf(w8[2], x0.z, s);
            s = fmaf(w8[3], x0.w, s);
            s = fmaf(w8[4], x1.x, s);
            s = fmaf(w8[5], x1.y, s);
            s = fmaf(w8[6], x1.z, s);
            s = fmaf(w8[7], x1.w, s);
            acc[n] = s;
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float sv = ft::warp_sum(acc[n]);
        if (lane == 0) o_s[(size_t)(obase + g0 + n) * RMAX + rl] = sv;
    }
}

__device__ __forceinline__ void down_row(const uint4* wrow, const float* hs, int ntok, int F, int lane, float* o_s,
                                         int off, int RMAX, int rl) {
    int g0 = 0;
    while (g0 < ntok) {
        const int rem = ntok - g0;
        if (rem >= 8) {
            down_group<8>(wrow, hs, g0, F, lane, o_s, off, RMAX, rl);
            g0 += 8;
        } else if (rem >= 4) {
            down_group<4>(wrow, hs, g0, F, lane, o_s, off, RMAX, rl);
            g0 += 4;
        } else if (rem >= 2) {
            down_group<2>(wrow, hs, g0, F, lane, o_s, off, RMAX, rl);
            g0 += 2;
        } else {
            down_group<1>(wrow, hs, g0, F, lane, o_s, off, RMAX, rl);
            g0 += 1;
        }
    }
}

__global__ void __launch_bounds__(EXPERT_THREADS, 1) expert_ffn_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_gdone;
    const int H = p.H, F = p.F, T = p.T, k = p.k;
    const int nst = p.nstage;
    const unsigned slot_bytes = p.stage_bytes;
    const int ugpu = p.info[INFO_UGPU];
    const int nasg = p.info[INFO_NASSIGN];
    const int G = gridDim.x, c = blockIdx.x;
    const int cpe = F / FPC;  // phase-A chunks per expert
    const int NA = ugpu * cpe;
    const int r0 = (int)((long long)H * c / G), r1 = (int)((long long)H * (c + 1) / G);
    const int R = r1 - r0;
    const int RMAX = (H + G - 1) / G;
    const int nB = R > 0 ? ugpu : 0;
    const int TK = T * k;

    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + nst;
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
    int* m_fill = m_pos + TK;                              // [TK]   fill index of entry (or -1)
    o += ((size_t)(6 * TK + 1) * 4 + 127) & ~(size_t)127;
    unsigned char* ring = smem + o;
    const unsigned rowbytes = (unsigned)H * 2u;
    const unsigned wpart = ((unsigned)RMAX * F * 2u + 127u) & ~127u;  // h rows follow the W_d rows

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            ft::mbar_init(&full[s], 1);
            ft::mbar_init(&empty[s], CONSUMER_WARPS);
        }
        ft::mbar_fence_init();
        s_gdone = 0;
    }
    for (int i = tid; i <= ugpu; i += EXPERT_THREADS) m_off[i] = p.wl_off[i];
    for (int i = tid; i < ugpu; i += EXPERT_THREADS) {
        m_slot[i] = p.wl_slot[i];
        m_fill[i] = p.do_fill ? p.wl_fill[i] : -1;
    }
    for (int i = tid; i < nasg; i += EXPERT_THREADS) {
        m_tok[i] = p.as_tok[i];
        m_gate[i] = p.as_gate[i];
    }
    for (int i = tid; i < TK; i += EXPERT_THREADS) m_pos[i] = p.out_pos[i];
    if (xf32) {
        for (int i = tid; i < T * H / 8; i += EXPERT_THREADS) {
            float f8[8];
            ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(p.x)[i], f8);
            reinterpret_cast<float4*>(x_s)[2 * i] = make_float4(f8[0], f8[1], f8[2], f8[3]);
            reinterpret_cast<float4*>(x_s)[2 * i + 1] = make_float4(f8[4], f8[5], f8[6], f8[7]);
        }
    } else {
        for (int i = tid; i < (int)(xbytes / 16); i += EXPERT_THREADS)
            reinterpret_cast<uint4*>(x_s)[i] = reinterpret_cast<const uint4*>(p.x)[i];
    }
    __syncthreads();

    // --------------------------------------------------------- fused fill
    if (wid > CONSUMER_WARPS) {
        if (lane == 0 && p.do_fill)
            ft::fill_share_tma(reinterpret_cast<const uint8_t*>(p.host_pool), const_cast<uint8_t*>(p.slot_pool), p.rb,
                               p.info[INFO_Q], p.fill_slot, p.fill_fid, p.ready, c, G,
                               ring + (size_t)nst * slot_bytes, reinterpret_cast<uint64_t*>(smem + 128),
                               p.fill_chunk, p.fill_slots, p.err);
        return;
    }
    // ------------------------------------------------------------ producer
    if (wid == CONSUMER_WARPS) {
        if (lane == 0) {
            const uint64_t pol = ft::l2_policy_evict_first();
            int it = 0;
            bool ok = true;
            int waited = -1;  // last fill index known complete
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
                const int grp = f0 >> 4, i = f0 & 15;
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                ft::mbar_arrive_expect_tx(&full[st], 2u * FPC * rowbytes);
                ft::bulk_g2s_hint(dst, rec + (size_t)(grp * 32 + i) * rowbytes, FPC * rowbytes, &full[st], pol);
                ft::bulk_g2s_hint(dst + (size_t)FPC * rowbytes, rec + (size_t)(grp * 32 + 16 + i) * rowbytes,
                                  FPC * rowbytes, &full[st], pol);
            }
            // phase B: W_d rows stream ahead of the grid barrier; the h rows of
            // an entry are copied once every CTA has written its h.
            const unsigned wb = (unsigned)R * F * 2u;
            const int pre = nB < nst ? nB : nst;
            const int itB = it;
            bool gdone = false;
            for (int e = 0; e < nB && ok; ++e, ++it) {
                const int st = it % nst;
                if (it >= nst && !ft::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err)) { ok = false; break; }
                const int off = m_off[e];
                const unsigned hb = (unsigned)(m_off[e + 1] - off) * F * 4u;
                unsigned char* dst = ring + (size_t)st * slot_bytes;
                if (m_fill[e] >= 0 && !ft::wait_filled(p.ready, m_fill[e], (unsigned)G, p.err)) { ok = false; break; }
                const uint8_t* wd = p.slot_pool + (size_t)m_slot[e] * p.rb + (size_t)2 * F * H * 2 + (size_t)r0 * F * 2;
                ft::mbar_arrive_expect_tx(&full[st], wb + hb);
                ft::bulk_g2s_hint(dst, wd, wb, &full[st], pol);
                if (e == pre - 1 || e >= pre) {
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
                        for (int e2 = 0; e2 < pre; ++e2) {  // deferred h rows of the prefetched entries
                            const int st2 = (itB + e2) % nst;
                            const int off2 = m_off[e2];
                            const unsigned hb2 = (unsigned)(m_off[e2 + 1] - off2) * F * 4u;
                            ft::bulk_g2s(ring + (size_t)st2 * slot_bytes + wpart, p.hbuf + (size_t)off2 * F, hb2,
                                         &full[st2]);
                        }
                    } else {
                        ft::bulk_g2s(dst + wpart, p.hbuf + (size_t)off * F, hb, &full[st]);
                    }
                }
            }
            ft::drain_ring(full, it, nst, p.err);
        }
        return;
    }

    // ------------------------------------------------- phase A: gate/up + SwiGLU
    // After a failed (timed-out) wait a warp stops waiting, computing and
    // releasing slots, but keeps the same barrier sequence as the others.
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
        const uint4* wg = reinterpret_cast<const uint4*>(ring + (size_t)st * slot_bytes + (size_t)wid * rowbytes);
        const uint4* wu = reinterpret_cast<const uint4*>(ring + (size_t)st * slot_bytes +
                                                         (size_t)(FPC + wid) * rowbytes);
        if (ok) {
            if (xf32)
                gu_feature<true>(wg, wu, x_s, m_tok, off, ntok, H, F, f, lane, p.hbuf);
            else
                gu_feature<false>(wg, wu, x_s, m_tok, off, ntok, H, F, f, lane, p.hbuf);
        }
        __syncwarp();
        if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
    }

    // every h of this layer is written before any CTA starts phase B
    ft::named_bar_sync(1, CONSUMERS);
    if (tid == 0) {
        ft::grid_barrier(p.gbar, (unsigned)G, p.err);
        ft::st_release_cta(&s_gdone, 1);
    }
    ft::named_bar_sync(1, CONSUMERS);

    // ---------------------------------------------------- phase B: down rows
    for (int e = 0; e < nB; ++e, ++it) {
        const int st = it % nst;
        const bool ok = !failed && ft::mbar_wait(&full[st], (it / nst) & 1, p.err);
        failed = !ok;
        const int off = m_off[e];
        const int ntok = m_off[e + 1] - off;
        const unsigned char* sb = ring + (size_t)st * slot_bytes;
        const float* hs = reinterpret_cast<const float*>(sb + wpart);
        for (int rl = wid; rl < R && ok; rl += CONSUMER_WARPS)
            down_row(reinterpret_cast<const uint4*>(sb + (size_t)rl * F * 2), hs, ntok, F, lane, o_s, off, RMAX, rl);
        __syncwarp();
        if (ok && lane == 0) ft::mbar_arrive(&empty[st]);
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
}

}  // namespace

cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s) {
    fill_kernel<<<grid, 512, 0, s>>>(p);
    return cudaGetLastError();
}

static constexpr size_t kSmemLimit = 227 * 1024;

// Shared-memory plan: barriers, x (if it fits in 64 KiB), the per-CTA output
// block, the worklist metadata, then as many ring slots as fit (at most 4).  A
// slot holds one phase-A chunk (16 rows of H) or one phase-B stage (R rows of
// W_d followed by the h rows of the entry's tokens).
cudaError_t launch_expert_ffn(ExpertParams p, int num_sms, cudaStream_t s) {
    const int G = num_sms;
    const int RMAX = (p.H + G - 1) / G;
    const bool xf32 = (size_t)p.T * p.H * 4 <= 65536;
    const size_t xbytes = (size_t)p.T * p.H * (xf32 ? 4 : 2);
    const size_t TK = (size_t)p.T * p.k;
    const size_t head = HEAD + ((xbytes + 127) & ~(size_t)127) +
                        ((TK * RMAX * 4 + 127) & ~(size_t)127) + (((6 * TK + 1) * 4 + 127) & ~(size_t)127);
    size_t slot = (size_t)2 * FPC * p.H * 2;
    const size_t down = (((size_t)RMAX * p.F * 2 + 127) & ~(size_t)127) + (size_t)p.T * p.F * 4;
    if (down > slot) slot = down;
    slot = (slot + 127) & ~(size_t)127;
    if (head >= kSmemLimit) return cudaErrorInvalidValue;
    // two fused-fill ring slots after the main ring: 16 KiB each, smaller if
    // that would leave fewer than two main slots
    size_t fch = 16384;
    int nst = 0;
    for (; fch >= 4096; fch /= 2) {
        if (head + 2 * fch >= kSmemLimit) continue;
        nst = (int)((kSmemLimit - head - 2 * fch) / slot);
        if (nst >= 2) break;
    }
    if (nst > 4) nst = 4;
    if (nst < 2) return cudaErrorInvalidValue;
    p.nstage = nst;
    p.stage_bytes = (unsigned)slot;
    int nf = (int)((kSmemLimit - head - slot * nst) / fch);
    if (nf > 4) nf = 4;
    p.fill_chunk = (unsigned)fch;
    p.fill_slots = nf;
    const size_t smem = head + slot * nst + (size_t)nf * fch;
    static size_t smem_set = 0;
    if (smem != smem_set) {
        cudaError_t e = cudaFuncSetAttribute(expert_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
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
