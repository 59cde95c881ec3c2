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
// kernels are streaming GEMVs: a persistent grid of one CTA per SM, weights
// staged through a ring of shared-memory buffers by 1-D bulk (TMA) copies
// completing on mbarriers, consumed by 8 warps with fp32 accumulation.
//   gate/up: the work is the flat list of (GPU expert, feature pair); CTA c
//            takes a contiguous 1/G share; one stage = gate rows f, f+1 and
//            up rows f, f+1 (contiguous in the record thanks to the 16-row
//            gate/up interleave); h is written in fp32.
//   down:    CTA c owns output rows [c*H/G, (c+1)*H/G) for every GPU expert:
//            one stage = those W_d rows of one expert plus the h rows of its
//            tokens; the gated merge over j (ascending) and partial_C is then
//            done in the same CTA, so the sum order is fixed and no atomics
//            are needed.
#include "ft_common.cuh"

namespace {

constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int EXPERT_THREADS = CONSUMERS + 32;  // + one producer warp
constexpr int MAXTOK = 16;                      // tokens per register block

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

// ---------------------------------------------------------- gate/up + SwiGLU

__device__ __forceinline__ float silu_mul(float a, float b) { return a / (1.f + expf(-a)) * b; }

struct RingBars {
    uint64_t* full;
    uint64_t* empty;
};

// Producer-side drain: wait (bounded) for the last phase of every stage that
// received a copy, so no bulk copy is in flight into shared memory at exit.
__device__ void drain_ring(RingBars rb, int issued, int nst, unsigned* err) {
    for (int it = issued - nst; it < issued; ++it) {
        if (it < 0) continue;
        ft::mbar_wait(&rb.full[it % nst], (it / nst) & 1, err);
    }
}

__global__ void __launch_bounds__(EXPERT_THREADS, 1) gateup_swiglu_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int H = p.H, F = p.F, T = p.T;
    const int nst = p.nstage;
    const int ugpu = p.info[INFO_UGPU];
    const int upe = F / 2;  // feature pairs per expert
    const int N = ugpu * upe;
    const int G = gridDim.x, c = blockIdx.x;
    const int u0 = (int)((long long)N * c / G), u1 = (int)((long long)N * (c + 1) / G);
    if (u0 >= u1) return;

    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    RingBars bars{reinterpret_cast<uint64_t*>(smem), reinterpret_cast<uint64_t*>(smem) + nst};
    float* red = reinterpret_cast<float*>(smem + 256);                       // [2][8][MAXTOK]
    const size_t xbytes = (size_t)T * H * 2;
    const bool x_in_smem = xbytes <= 65536;
    __nv_bfloat16* x_s = reinterpret_cast<__nv_bfloat16*>(smem + 256 + 2 * 8 * MAXTOK * 4);
    unsigned char* stages = smem + 256 + 2 * 8 * MAXTOK * 4 + (x_in_smem ? ((xbytes + 127) & ~(size_t)127) : 0);
    const __nv_bfloat16* xsrc = x_in_smem ? x_s : p.x;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            ft::mbar_init(&bars.full[s], 1);
            ft::mbar_init(&bars.empty[s], CONSUMER_WARPS);
        }
        ft::mbar_fence_init();
    }
    if (x_in_smem)
        for (int i = tid; i < (int)(xbytes / 16); i += EXPERT_THREADS)
            reinterpret_cast<uint4*>(x_s)[i] = reinterpret_cast<const uint4*>(p.x)[i];
    __syncthreads();

    const unsigned rowbytes = (unsigned)H * 2u;
    if (wid == CONSUMER_WARPS) {
        if (lane == 0) {
            const uint64_t pol = ft::l2_policy_evict_first();
            int it = 0;
            for (int u = u0; u < u1; ++u, ++it) {
                const int st = it % nst;
                if (it >= nst && !ft::mbar_wait(&bars.empty[st], ((it / nst) - 1) & 1, p.err)) break;
                const int ent = u / upe;
                const int f0 = (u - ent * upe) * 2;
                const uint8_t* rec = p.slot_pool + (size_t)p.wl_slot[ent] * p.rb;
                const int grp = f0 >> 4, i = f0 & 15;
                const uint8_t* gsrc = rec + (size_t)(grp * 32 + i) * rowbytes;
                const uint8_t* usrc = rec + (size_t)(grp * 32 + 16 + i) * rowbytes;
                unsigned char* dst = stages + (size_t)st * p.stage_bytes;
                ft::mbar_arrive_expect_tx(&bars.full[st], 4u * rowbytes);
                ft::bulk_g2s_hint(dst, gsrc, 2u * rowbytes, &bars.full[st], pol);
                ft::bulk_g2s_hint(dst + 2u * rowbytes, usrc, 2u * rowbytes, &bars.full[st], pol);
            }
            drain_ring(bars, it, nst, p.err);
        }
        return;
    }

    // consumers: warp w handles row (w >> 1) of the stage (g0, g1, u0, u1) and K half (w & 1).
    // After a failed (timed-out) wait a warp stops waiting and computing but
    // keeps the same named-barrier sequence as the others; it no longer
    // releases stages, so the producer's own bounded wait ends the ring.
    const int r = wid >> 1, kh = wid & 1;
    const int nv = H / 16;  // 16-byte vectors per K half
    int buf = 0;
    int it = 0;
    bool failed = false;
    for (int u = u0; u < u1; ++u, ++it) {
        const int st = it % nst;
        const bool ok = !failed && ft::mbar_wait(&bars.full[st], (it / nst) & 1, p.err);
        failed = !ok;
        const int ent = u / upe;
        const int f0 = (u - ent * upe) * 2;
        const int off = p.wl_off[ent];
        const int ntok = p.wl_off[ent + 1] - off;
        const uint4* wrow = reinterpret_cast<const uint4*>(stages + (size_t)st * p.stage_bytes +
                                                           (size_t)r * rowbytes + (size_t)kh * (rowbytes / 2));
        for (int g0 = 0; g0 < ntok; g0 += MAXTOK) {
            const int ng = min(MAXTOK, ntok - g0);
            int tk[MAXTOK];
#pragma unroll
            for (int n = 0; n < MAXTOK; ++n) tk[n] = n < ng ? p.as_tok[off + g0 + n] : 0;
            float acc[MAXTOK];
#pragma unroll
            for (int n = 0; n < MAXTOK; ++n) acc[n] = 0.f;
            if (ok) {
                for (int v = lane; v < nv; v += 32) {
                    float w8[8];
                    ft::bf16x8_to_f32(wrow[v], w8);
#pragma unroll
                    for (int n = 0; n < MAXTOK; ++n) {
                        if (n < ng) {
                            const uint4 xv = reinterpret_cast<const uint4*>(xsrc + (size_t)tk[n] * H +
                                                                            (size_t)kh * (H / 2))[v];
                            float x8[8];
                            ft::bf16x8_to_f32(xv, x8);
                            float s = acc[n];
#pragma unroll
                            for (int q = 0; q < 8; ++q) s = fmaf(w8[q], x8[q], s);
                            acc[n] = s;
                        }
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < MAXTOK; ++n) {
                if (n < ng) {
                    const float sum = ft::warp_sum(acc[n]);
                    if (lane == 0) red[(buf * 8 + wid) * MAXTOK + n] = sum;
                }
            }
            if (ok && g0 + MAXTOK >= ntok) {
                __syncwarp();
                if (lane == 0) ft::mbar_arrive(&bars.empty[st]);
            }
            ft::named_bar_sync(1, CONSUMERS);
            if (tid < 2 * ng) {
                const int fi = tid / ng, n = tid - fi * ng;
                const float* R = red + buf * 8 * MAXTOK;
                const float a = R[(2 * fi) * MAXTOK + n] + R[(2 * fi + 1) * MAXTOK + n];
                const float b = R[(4 + 2 * fi) * MAXTOK + n] + R[(5 + 2 * fi) * MAXTOK + n];
                p.hbuf[(size_t)(off + g0 + n) * F + f0 + fi] = silu_mul(a, b);
            }
            buf ^= 1;
        }
        if (ntok == 0) {
            __syncwarp();
            if (ok && lane == 0) ft::mbar_arrive(&bars.empty[st]);
            ft::named_bar_sync(1, CONSUMERS);
        }
    }
}

// ------------------------------------------------ down + gated merge + partial_C

__global__ void __launch_bounds__(EXPERT_THREADS, 1) down_combine_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int H = p.H, F = p.F, T = p.T, k = p.k;
    const int nst = p.nstage;
    const int ugpu = p.info[INFO_UGPU];
    const int G = gridDim.x, c = blockIdx.x;
    const int r0 = (int)((long long)H * c / G), r1 = (int)((long long)H * (c + 1) / G);
    const int R = r1 - r0;
    if (R <= 0) return;
    const int RMAX = (H + G - 1) / G;
    const int nasg_max = T * k;

    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    RingBars bars{reinterpret_cast<uint64_t*>(smem), reinterpret_cast<uint64_t*>(smem) + nst};
    float* o_s = reinterpret_cast<float*>(smem + 256);  // [T*k][RMAX]
    unsigned char* stages = smem + 256 + (((size_t)nasg_max * RMAX * 4 + 127) & ~(size_t)127);
    const unsigned wbytes_max = (unsigned)(((size_t)RMAX * F * 2 + 127) & ~(size_t)127);

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            ft::mbar_init(&bars.full[s], 1);
            ft::mbar_init(&bars.empty[s], CONSUMER_WARPS);
        }
        ft::mbar_fence_init();
    }
    __syncthreads();

    if (wid == CONSUMER_WARPS) {
        if (lane == 0) {
            const uint64_t pol = ft::l2_policy_evict_first();
            int it = 0;
            for (int ent = 0; ent < ugpu; ++ent, ++it) {
                const int st = it % nst;
                if (it >= nst && !ft::mbar_wait(&bars.empty[st], ((it / nst) - 1) & 1, p.err)) break;
                const int off = p.wl_off[ent];
                const int ntok = p.wl_off[ent + 1] - off;
                const uint8_t* wd = p.slot_pool + (size_t)p.wl_slot[ent] * p.rb + (size_t)2 * F * H * 2 +
                                    (size_t)r0 * F * 2;
                unsigned char* dst = stages + (size_t)st * p.stage_bytes;
                const unsigned wb = (unsigned)R * F * 2, hb = (unsigned)ntok * F * 4;
                ft::mbar_arrive_expect_tx(&bars.full[st], wb + hb);
                ft::bulk_g2s_hint(dst, wd, wb, &bars.full[st], pol);
                if (hb) ft::bulk_g2s(dst + wbytes_max, p.hbuf + (size_t)off * F, hb, &bars.full[st]);
            }
            drain_ring(bars, it, nst, p.err);
        }
        return;
    }

    const int nv = F / 8;  // 16-byte weight vectors per row
    int it = 0;
    for (int ent = 0; ent < ugpu; ++ent, ++it) {
        const int st = it % nst;
        const bool ok = ft::mbar_wait(&bars.full[st], (it / nst) & 1, p.err);
        const int off = p.wl_off[ent];
        const int ntok = p.wl_off[ent + 1] - off;
        const unsigned char* sb = stages + (size_t)st * p.stage_bytes;
        const float* hs = reinterpret_cast<const float*>(sb + wbytes_max);
        if (ok) {
            for (int rl = wid; rl < R; rl += CONSUMER_WARPS) {
                const uint4* wrow = reinterpret_cast<const uint4*>(sb + (size_t)rl * F * 2);
                for (int g0 = 0; g0 < ntok; g0 += MAXTOK) {
                    const int ng = min(MAXTOK, ntok - g0);
                    float acc[MAXTOK];
#pragma unroll
                    for (int n = 0; n < MAXTOK; ++n) acc[n] = 0.f;
                    for (int v = lane; v < nv; v += 32) {
                        float w8[8];
                        ft::bf16x8_to_f32(wrow[v], w8);
#pragma unroll
                        for (int n = 0; n < MAXTOK; ++n) {
                            if (n < ng) {
                                const float4* h4 = reinterpret_cast<const float4*>(hs + (size_t)(g0 + n) * F + v * 8);
                                const float4 a = h4[0], b = h4[1];
                                float s = acc[n];
                                s = fmaf(w8[0], a.x, s);
                                s = fmaf(w8[1], a.y, s);
                                s = fmaf(w8[2], a.z, s);
                                s = fmaf(w8[3], a.w, s);
                                s = fmaf(w8[4], b.x, s);
                                s = fmaf(w8[5], b.y, s);
                                s = fmaf(w8[6], b.z, s);
                                s = fmaf(w8[7], b.w, s);
                                acc[n] = s;
                            }
                        }
                    }
#pragma unroll
                    for (int n = 0; n < MAXTOK; ++n) {
                        if (n < ng) {
                            const float sum = ft::warp_sum(acc[n]);
                            if (lane == 0) o_s[(size_t)(off + g0 + n) * RMAX + rl] = sum;
                        }
                    }
                }
            }
        }
        if (!ok) break;  // stop releasing stages: the producer's bounded wait ends the ring
        __syncwarp();
        if (lane == 0) ft::mbar_arrive(&bars.empty[st]);
    }
    ft::named_bar_sync(1, CONSUMERS);
    // gated merge in fixed order: j ascending, then the CPU-set partial sum
    for (int idx = tid; idx < T * R; idx += CONSUMERS) {
        const int t = idx / R, rl = idx - t * R;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
            const int pos = p.out_pos[t * k + j];
            if (pos >= 0) acc = fmaf(p.as_gate[pos], o_s[(size_t)pos * RMAX + rl], acc);
        }
        const size_t o = (size_t)t * H + r0 + rl;
        if (p.partial_C) acc += p.partial_C[o];
        p.y[o] = acc;
    }
}

}  // namespace

cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s) {
    fill_kernel<<<grid, 512, 0, s>>>(p);
    return cudaGetLastError();
}

static cudaError_t set_smem(const void* fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

static constexpr size_t kSmemLimit = 227 * 1024;

// Shared-memory plan of the gate/up kernel: fixed header, x (if it fits in
// 64 KiB), then as many 4-row stages as fit (at most 8).
cudaError_t launch_gateup(ExpertParams p, int num_sms, cudaStream_t s) {
    const size_t xbytes = (size_t)p.T * p.H * 2;
    const size_t head = 256 + 2 * 8 * MAXTOK * 4 + (xbytes <= 65536 ? ((xbytes + 127) & ~(size_t)127) : 0);
    const size_t stage = (size_t)4 * p.H * 2;
    int nst = (int)((kSmemLimit - head) / stage);
    if (nst > 8) nst = 8;
    if (nst < 2) return cudaErrorInvalidValue;
    p.nstage = nst;
    p.stage_bytes = (unsigned)stage;
    const size_t smem = head + stage * nst;
    cudaError_t e = set_smem((const void*)gateup_swiglu_kernel, smem);
    if (e != cudaSuccess) return e;
    gateup_swiglu_kernel<<<num_sms, EXPERT_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_down(ExpertParams p, int num_sms, cudaStream_t s) {
    const int G = num_sms;
    const int RMAX = (p.H + G - 1) / G;
    const size_t head = 256 + (((size_t)p.T * p.k * RMAX * 4 + 127) & ~(size_t)127);
    const size_t wpart = ((size_t)RMAX * p.F * 2 + 127) & ~(size_t)127;
    const size_t stage = wpart + (size_t)p.T * p.F * 4;
    int nst = (int)((kSmemLimit - head) / stage);
    if (nst > 8) nst = 8;
    if (nst < 2) return cudaErrorInvalidValue;
    p.nstage = nst;
    p.stage_bytes = (unsigned)stage;
    const size_t smem = head + stage * nst;
    cudaError_t e = set_smem((const void*)down_combine_kernel, smem);
    if (e != cudaSuccess) return e;
    down_combine_kernel<<<G, EXPERT_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}
