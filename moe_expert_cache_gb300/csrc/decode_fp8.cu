// Decode expert FFN over block-FP8 records (W8A16).
//
// deepmox "One logical expert, two physical levels of memory": a block-FP8
// bank keeps FP8 weights and block-scale data.  Here the values are OCP FP8
// E4M3 codes and every 128 x 128 block (rows x K) of each weight matrix has
// one fp32 scale: w = e4m3(code) * scale(row / 128, k / 128).
//
// Record (per layer-expert): [W_gu values 2F x H bytes, gate/up rows
// interleaved in groups of 16] [W_d values H x F] [W_g scales F/128 x H/128
// fp32] [W_u scales F/128 x H/128] [W_d scales H/128 x F/128].
//
// Two kernels:
//   * fp8_gateup_kernel (cooperative, two CTAs per SM): every warp takes
//     (entry, feature) units; a unit streams the feature's gate and up rows
//     with 16-byte loads that skip L1, against every token of the entry, and
//     writes SwiGLU(h) to the fp32 scratch [assignment, F].  The fills the
//     control pass left pending stream in the same launch: the first thread
//     of each CTA's last warp copies the CTA's share of every fill record
//     from the host pool through a small TMA ring into the victim slot and
//     counts itself in the fill's counter, then that warp joins the others,
//     which claim the CTA's units one at a time; the units of a fill entry
//     wait (bounded) until every CTA has counted, while the resident
//     entries' units go ahead, so the host-link time overlaps the HBM-bound
//     work;
//   * fp8_down_kernel: CTA c owns output rows [c*H/G, (c+1)*H/G); its warps
//     take (entry, row) units against the h rows, then the CTA merges the
//     gated sum with the CPU-set partial sum in fixed order.
// E4M3 pairs are converted by the hardware (cvt.rn.f16x2.e4m3x2, exact),
// widened to fp32 and accumulated in fp32 per 16-value chunk, then scaled
// by the chunk's block scale (16 divides 128).
#include "ft_common.cuh"
#include "../../include/ft.h"

#include <cuda_fp16.h>

namespace {

constexpr int A_WARPS = 8;                  // warps of the gate/up kernel (the last one fills first)
constexpr int A_THREADS = A_WARPS * 32;
constexpr int A_FILL_SLOTS = 2;             // fused-fill ring chunks per CTA (two CTAs per SM)
constexpr unsigned A_FILL_CHUNK = 4096;     // bytes of one fused-fill ring chunk
constexpr int B_THREADS = 512;
constexpr int FP8_BLK = 128;

// 16-byte load of streamed weights, bypassing L1.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two e4m3 codes (the low and high byte of `b`) to fp32, exactly.
__device__ __forceinline__ float2 e4m3x2(uint32_t b) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)b));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Dot of 16 e4m3 values (one uint4, in K order) with 16 fp32 activations.
__device__ __forceinline__ float dot16(const uint4& w, const float* x) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 lo = e4m3x2(ww[i]), hi = e4m3x2(ww[i] >> 16);
        a = fmaf(lo.x, x[4 * i], a);
        b = fmaf(lo.y, x[4 * i + 1], b);
        a = fmaf(hi.x, x[4 * i + 2], a);
        b = fmaf(hi.y, x[4 * i + 3], b);
    }
    return a + b;
}

// Activations staged in shared memory as fp32, each 16-value chunk's four
// float4 rotated by (chunk / 2) mod 4 so that the eight lanes of a quarter
// warp (consecutive chunks) read eight different bank quads.
__device__ __forceinline__ int xrot(int e) {  // element e of a row -> its stored position
    const int q = e >> 4, i = (e >> 2) & 3;
    return (q << 4) | (((i + (q >> 1)) & 3) << 2) | (e & 3);
}

// The 16 activations of chunk c of a token row: from the rotated fp32 copy
// in shared memory (XS), or from the bf16 input in global memory.
template <bool XS>
__device__ __forceinline__ void load_x16(const float* xs, const __nv_bfloat16* xg, int t, int H, int c, float* x) {
    if (XS) {
        const float4* p = reinterpret_cast<const float4*>(xs + (size_t)t * H + (size_t)c * 16);
        const int r = (c >> 1) & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 q = p[(i + r) & 3];
            x[4 * i] = q.x; x[4 * i + 1] = q.y; x[4 * i + 2] = q.z; x[4 * i + 3] = q.w;
        }
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(xg + (size_t)t * H + (size_t)c * 16);
        ft::bf16x8_to_f32(__ldg(p), x);
        ft::bf16x8_to_f32(__ldg(p + 1), x + 8);
    }
}

// Gate and up rows of one feature against NT tokens (token rows tk).
template <int NT, bool XS>
__device__ __forceinline__ void gu_rows(const uint8_t* wg, const uint8_t* wu, const float* sg, const float* su,
                                        const float* xs, const __nv_bfloat16* xg, const int* tk, int H, int lane,
                                        float* ag, float* au) {
#pragma unroll
    for (int n = 0; n < NT; ++n) ag[n] = au[n] = 0.f;
    const int nc = H >> 4;
    // BT chunks of both rows are loaded before any is used (2 BT 16-byte
    // loads in flight per lane; fewer when more tokens share them, for the
    // registers)
    constexpr int BT = NT >= 4 ? 1 : (XS ? 4 : 2);
    for (int c0 = lane; c0 < nc; c0 += 32 * BT) {
        uint4 a[BT], b[BT];
#pragma unroll
        for (int j = 0; j < BT; ++j) {
            const int c = c0 + 32 * j;
            if (c < nc) {
                a[j] = ld_stream(wg + (size_t)c * 16);
                b[j] = ld_stream(wu + (size_t)c * 16);
            }
        }
#pragma unroll
        for (int j = 0; j < BT; ++j) {
            const int c = c0 + 32 * j;
            if (c < nc) {
                const float s1 = sg[c >> 3], s2 = su[c >> 3];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float x[16];
                    load_x16<XS>(xs, xg, tk[n], H, c, x);
                    ag[n] = fmaf(s1, dot16(a[j], x), ag[n]);
                    au[n] = fmaf(s2, dot16(b[j], x), au[n]);
                }
            }
        }
    }
}

template <int NT, bool XS>
__device__ __forceinline__ void gu_group(const uint8_t* wg, const uint8_t* wu, const float* sg, const float* su,
                                         const float* xs, const __nv_bfloat16* xg, const int* as_tok, int H, int F,
                                         int f, int pos0, int lane, float* hbuf) {
    int tk[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) tk[n] = as_tok[pos0 + n];
    float ag[NT], au[NT];
    gu_rows<NT, XS>(wg, wu, sg, su, xs, xg, tk, H, lane, ag, au);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float g = ft::warp_sum(ag[n]), u = ft::warp_sum(au[n]);
        if (lane == 0) hbuf[(size_t)(pos0 + n) * F + f] = ft::silu_mul(g, u);
    }
}

// Dynamic shared memory of the gate/up kernel: x as fp32 when XS, then the
// fused-fill ring.
__host__ __device__ inline size_t fp8_a_xbytes(int T, int H, bool xs) {
    return xs ? (((size_t)T * H * 4 + 127) & ~(size_t)127) : 0;
}

template <bool XS>
__global__ void __launch_bounds__(A_THREADS, 2) fp8_gateup_kernel(ExpertParams p) {
    extern __shared__ __align__(128) unsigned char smem_a[];
    __shared__ uint64_t fbar[A_FILL_SLOTS];
    __shared__ int s_xready, s_next;
    float* xs_dyn = reinterpret_cast<float*>(smem_a);
    const int H = p.H, F = p.F, T = p.T;
    const int ugpu = p.info[INFO_UGPU];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        s_xready = 0;
        s_next = 0;
    }
    __syncthreads();
    if (wid == A_WARPS - 1) {
        // ------------------------------------------- fused fill, then compute
        // this CTA's share of every fill record (nothing when q = 0), then
        // this warp's own units once x is staged
        if (lane == 0 && p.do_fill)
            ft::fill_share_tma(reinterpret_cast<const uint8_t*>(p.host_pool), const_cast<uint8_t*>(p.slot_pool), p.rb,
                               p.info[INFO_Q], p.fill_slot, p.fill_fid, p.ready, blockIdx.x, gridDim.x,
                               smem_a + fp8_a_xbytes(T, H, XS), fbar, A_FILL_CHUNK, A_FILL_SLOTS, p.err);
        if (XS && lane == 0) {
            const uint64_t t0 = ft::globaltimer();
            while (!ft::ld_acquire_cta(&s_xready)) {
                if (ft::globaltimer() - t0 > FT_WAIT_LIMIT_NS) {
                    atomicOr(p.err, FT_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (XS) {
        for (int i = tid; i < T * H / 8; i += (A_WARPS - 1) * 32) {
            float f8[8];
            ft::bf16x8_to_f32(reinterpret_cast<const uint4*>(p.x)[i], f8);
            const int t = (8 * i) / H, e = 8 * i - t * H;
            float* row = xs_dyn + (size_t)t * H;
            *reinterpret_cast<float4*>(row + xrot(e)) = make_float4(f8[0], f8[1], f8[2], f8[3]);
            *reinterpret_cast<float4*>(row + xrot(e + 4)) = make_float4(f8[4], f8[5], f8[6], f8[7]);
        }
        ft::named_bar_sync(1, (A_WARPS - 1) * 32);  // every warp but the fill warp
        if (tid == 0) ft::st_release_cta(&s_xready, 1);
    }
    const size_t nbg = (size_t)(F / FP8_BLK) * (H / FP8_BLK);  // scale blocks of W_g (and of W_u)
    int waited = -1;  // the last fill whose record this warp saw complete
    // this CTA's units c, c + G, ... (resident entries first, fills last),
    // claimed one at a time by whichever warp is free, so the fill warp
    // takes what is left once its copies are done
    for (;;) {
        int i = 0;
        if (lane == 0) i = atomicAdd(&s_next, 1);
        const int u = blockIdx.x + __shfl_sync(0xffffffffu, i, 0) * gridDim.x;
        if (u >= ugpu * F) break;
        const int e = u / F, f = u - e * F;
        if (p.do_fill) {
            const int fi = p.wl_fill[e];
            if (fi >= 0 && fi != waited) {
                int ok = 1;
                if (lane == 0) ok = ft::wait_filled(p.ready, fi, gridDim.x, p.err) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) continue;  // gave up: the status reports it
                waited = fi;
            }
        }
        const int off = p.wl_off[e], ntok = p.wl_off[e + 1] - off;
        const uint8_t* rec = p.slot_pool + (size_t)p.wl_slot[e] * p.rb;
        const int grow = (f >> 4) * 32 + (f & 15);  // gate row; the up row is 16 later
        const uint8_t* wg = rec + (size_t)grow * H;
        const uint8_t* wu = wg + (size_t)16 * H;
        const float* sc = reinterpret_cast<const float*>(rec + (size_t)3 * H * F);
        const float* sg = sc + (size_t)(f / FP8_BLK) * (H / FP8_BLK);
        const float* su = sg + nbg;
        int g0 = 0;
        while (g0 < ntok) {
            const int rem = ntok - g0;
            if (!XS && rem >= 4) {  // four-token groups where x comes from global memory (large T)
                gu_group<4, XS>(wg, wu, sg, su, xs_dyn, p.x, p.as_tok, H, F, f, off + g0, lane, p.hbuf);
                g0 += 4;
            } else if (rem >= 2) {
                gu_group<2, XS>(wg, wu, sg, su, xs_dyn, p.x, p.as_tok, H, F, f, off + g0, lane, p.hbuf);
                g0 += 2;
            } else {
                gu_group<1, XS>(wg, wu, sg, su, xs_dyn, p.x, p.as_tok, H, F, f, off + g0, lane, p.hbuf);
                g0 += 1;
            }
        }
    }
}

// One W_d row against NT h rows (fp32 rows of F values: the rotated copy in
// shared memory when HS, else the plain [assignment, F] scratch in global
// memory).
template <int NT, bool HS>
__device__ __forceinline__ void down_row(const uint8_t* wd, const float* sd, const float* hsrc, int pos0, int F,
                                         int lane, float* acc) {
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.f;
    const int nc = F >> 4;
    constexpr int BT = NT >= 4 ? 1 : 2;  // chunks loaded ahead (fewer with four tokens)
    for (int c0 = lane; c0 < nc; c0 += 32 * BT) {
        uint4 w[BT];
#pragma unroll
        for (int j = 0; j < BT; ++j)
            if (c0 + 32 * j < nc) w[j] = ld_stream(wd + (size_t)(c0 + 32 * j) * 16);
#pragma unroll
        for (int j = 0; j < BT; ++j) {
            const int c = c0 + 32 * j;
            if (c < nc) {
                const float s = sd[c >> 3];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float x[16];
                    if (HS) {
                        load_x16<true>(hsrc, nullptr, pos0 + n, F, c, x);
                    } else {
                        const float4* hp =
                            reinterpret_cast<const float4*>(hsrc + (size_t)(pos0 + n) * F + (size_t)c * 16);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 q = hp[i];
                            x[4 * i] = q.x; x[4 * i + 1] = q.y; x[4 * i + 2] = q.z; x[4 * i + 3] = q.w;
                        }
                    }
                    acc[n] = fmaf(s, dot16(w[j], x), acc[n]);
                }
            }
        }
    }
}

template <int NT, bool HS>
__device__ __forceinline__ void down_group(const uint8_t* wd, const float* sd, const float* hsrc, int pos0, int F,
                                           int lane, float* o_s, int RMAX, int rl) {
    float acc[NT];
    down_row<NT, HS>(wd, sd, hsrc, pos0, F, lane, acc);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float v = ft::warp_sum(acc[n]);
        if (lane == 0) o_s[(size_t)(pos0 + n) * RMAX + rl] = v;
    }
}

// HS: the h rows of every assignment (T*k rows of F fp32) are staged once per
// CTA in shared memory, rotated like x, so that the CTA's (entry, row) units
// read them from there instead of L2.
template <bool HS>
__global__ void __launch_bounds__(B_THREADS, 1) fp8_down_kernel(ExpertParams p) {
    extern __shared__ __align__(16) float o_s[];  // [assignment, RMAX], then the h rows (HS)
    const int H = p.H, F = p.F, T = p.T, k = p.k;
    const int ugpu = p.info[INFO_UGPU];
    const int G = gridDim.x, c = blockIdx.x;
    const int r0 = (int)((long long)H * c / G), r1 = (int)((long long)H * (c + 1) / G);
    const int R = r1 - r0;
    const int RMAX = (H + G - 1) / G;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    float* hs = o_s + (((size_t)T * k * RMAX + 3) & ~(size_t)3);
    if (HS) {
        const int nasg = p.info[INFO_NASSIGN];
        for (int i = tid; i < nasg * F / 4; i += B_THREADS) {
            const int a = (4 * i) / F, e = 4 * i - a * F;
            *reinterpret_cast<float4*>(hs + (size_t)a * F + xrot(e)) =
                reinterpret_cast<const float4*>(p.hbuf)[i];
        }
        __syncthreads();
    }
    const float* hsrc = HS ? hs : p.hbuf;
    const size_t nbg = (size_t)(F / FP8_BLK) * (H / FP8_BLK);
    for (int u = wid; u < ugpu * R; u += B_THREADS / 32) {
        const int e = u / R, rl = u - e * R;
        const int off = p.wl_off[e], ntok = p.wl_off[e + 1] - off;
        const uint8_t* rec = p.slot_pool + (size_t)p.wl_slot[e] * p.rb;
        const int r = r0 + rl;
        const uint8_t* wd = rec + (size_t)2 * F * H + (size_t)r * F;
        const float* sd = reinterpret_cast<const float*>(rec + (size_t)3 * H * F) + 2 * nbg +
                          (size_t)(r / FP8_BLK) * (F / FP8_BLK);
        int g0 = 0;
        while (g0 < ntok) {
            const int rem = ntok - g0;
            if (rem >= 4) {
                down_group<4, HS>(wd, sd, hsrc, off + g0, F, lane, o_s, RMAX, rl);
                g0 += 4;
            } else if (rem >= 2) {
                down_group<2, HS>(wd, sd, hsrc, off + g0, F, lane, o_s, RMAX, rl);
                g0 += 2;
            } else {
                down_group<1, HS>(wd, sd, hsrc, off + g0, F, lane, o_s, RMAX, rl);
                g0 += 1;
            }
        }
    }
    __syncthreads();
    // gated merge in fixed order: j ascending, then the CPU-set partial sum
    for (int idx = tid; idx < T * R; idx += B_THREADS) {
        const int t = idx / R, rl = idx - t * R;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
            const int pos = p.out_pos[t * k + j];
            if (pos >= 0) acc = fmaf(p.as_gate[pos], o_s[(size_t)pos * RMAX + rl], acc);
        }
        const size_t oi = (size_t)t * H + r0 + rl;
        if (p.partial_C) acc += p.partial_C[oi];
        p.y[oi] = acc;
    }
}

}  // namespace

cudaError_t launch_expert_ffn_fp8(ExpertParams p, int num_sms, cudaStream_t s) {
    const bool xs = (size_t)p.T * p.H * 4 <= 96 * 1024;
    const size_t smem_a = fp8_a_xbytes(p.T, p.H, xs) + (size_t)A_FILL_SLOTS * A_FILL_CHUNK;
    const void* fa = xs ? (const void*)fp8_gateup_kernel<true> : (const void*)fp8_gateup_kernel<false>;
    cudaError_t e = ensure_dynamic_smem(fa, smem_a);
    if (e != cudaSuccess) return e;
    // cooperative: the units of a fill entry wait for every CTA's share of
    // the record, so all CTAs must be resident together
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fa, A_THREADS, smem_a);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((per_sm < 2 ? per_sm : 2) * num_sms);
    cfg.blockDim = dim3(A_THREADS);
    cfg.dynamicSmemBytes = smem_a;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    e = cudaLaunchKernelExC(&cfg, fa, args);
    if (e != cudaSuccess) return e;
    const int RMAX = (p.H + num_sms - 1) / num_sms;
    const size_t o_bytes = (((size_t)p.T * p.k * RMAX + 3) & ~(size_t)3) * 4;
    const size_t h_bytes = (size_t)p.T * p.k * p.F * 4;
    const bool hs = o_bytes + h_bytes <= 200 * 1024;
    const size_t smem_b = o_bytes + (hs ? h_bytes : 0);
    if (smem_b > 227 * 1024) return cudaErrorInvalidValue;
    const void* fb = hs ? (const void*)fp8_down_kernel<true> : (const void*)fp8_down_kernel<false>;
    e = ensure_dynamic_smem(fb, smem_b);
    if (e != cudaSuccess) return e;
    if (hs)
        fp8_down_kernel<true><<<num_sms, B_THREADS, smem_b, s>>>(p);
    else
        fp8_down_kernel<false><<<num_sms, B_THREADS, smem_b, s>>>(p);
    return cudaGetLastError();
}
