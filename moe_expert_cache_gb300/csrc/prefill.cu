// Prefill path of the expert cache: full-layer double buffer and grouped
// GEMMs on the tensor cores.
//
// FreeToken explainer section 2 "Prefill: Stream the Entire Layer" and the
// deepmox chapter "The Expert Cache That Follows the Router": during prefill
// the union of the routes covers almost every expert, so whole layers are
// streamed through two full-layer buffers carved from the first two
// expert-layer regions of the slot pool, the next layer copied by a transfer
// stream while the current one computes; a release event makes a buffer's
// reuse wait for the GEMMs reading it, a begin fence orders the first copy
// after earlier decode work, and the previous owners of a buffer's slots are
// invalidated before it is overwritten.
//
// Per layer, on the compute stream:
//   pf_route    top-k + softmax gates per token, routed-token count per expert
//   pf_permute  per expert: its routes in token order (stable counting sort),
//               offsets, the route -> row map and the per-row gate
//   pf_gather   x rows into expert order (bf16)
//   GEMM1       per expert, X_e [M_e x H] . W_gu^T [H x 2F] on tcgen05, SwiGLU
//               epilogue -> h [M_e x F] bf16
//   GEMM2       per expert, h_e . W_d^T [F x H] -> gate * out [M_e x H] f16
//               (fp32 accumulation; the f16 rounding adds about 1e-5 relative
//               to the bf16 rounding of h, and halves the bytes of the per-route
//               outputs written here and read back by the combine)
//   pf_combine  y_t = sum_j (gate * out)[row(t, j)] in fp32, j ascending
#include "ft_common.cuh"
#include "ft_prefill.cuh"
#include "ft_tc.cuh"

#include <math.h>

namespace {

// ----------------------------------------------------------------- routing

// One warp per token: top-k of E <= 256 logits (value descending, lower id
// first), softmax over the k selected; counts[e] += 1 for every route.
__global__ void __launch_bounds__(256) pf_route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                       int* __restrict__ ids, float* __restrict__ gates,
                                                       int* __restrict__ counts, unsigned* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    constexpr int RV = 8;
    float vals[RV];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < RV; ++i) {
        const int e = lane + 32 * i;
        vals[i] = e < E ? row[e] : -INFINITY;
        if (e < E && !isfinite(vals[i])) bad = true;
    }
    bad = __any_sync(0xffffffffu, bad);
    unsigned used = 0;
    float sel_v = 0.f;
    int sel_e = lane;
    for (int j = 0; j < k && !bad; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < RV; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((used >> i) & 1u)) {
                const float v = vals[i];
                if (v > bv || (v == bv && e < be)) {
                    bv = v;
                    be = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) used |= 1u << (be >> 5);
        if (lane == j) {
            sel_v = bv;
            sel_e = be;
        }
    }
    float g;
    if (bad) {
        // invalid token: latch the error; its routes keep distinct in-range ids
        // and zero gates so the rest of the layer stays well formed
        if (lane == 0) atomicOr(err, FT_DEVERR_ARG);
        sel_e = lane;
        g = 0.f;
    } else {
        const float v0 = __shfl_sync(0xffffffffu, sel_v, 0);
        const float ex = lane < k ? expf(sel_v - v0) : 0.f;
        const float den = ft::warp_sum(ex);
        g = ex / den;
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = sel_e;
        gates[(size_t)t * k + lane] = g;
        atomicAdd(&counts[sel_e], 1);
    }
}

// One CTA per expert: offset = sum of the counts of lower experts; the
// expert's routes in ascending token order get consecutive rows.
__global__ void __launch_bounds__(1024) pf_permute_kernel(const int* __restrict__ ids, const float* __restrict__ gates,
                                                          const int* __restrict__ counts, int T, int E, int k,
                                                          int* __restrict__ offsets, int* __restrict__ perm_tok,
                                                          int* __restrict__ pos, float* __restrict__ row_gate) {
    __shared__ int warp_tot[32];
    __shared__ int s_off, s_carry;
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        int o = 0;
        for (int i = 0; i < e; ++i) o += counts[i];
        s_off = o;
        s_carry = 0;
        offsets[e] = o;
        if (e == E - 1) offsets[E] = o + counts[e];
    }
    __syncthreads();
    const int off = s_off;
    for (int t0 = 0; t0 < T; t0 += 1024) {
        const int t = t0 + tid;
        int jj = -1;
        if (t < T) {
            for (int j = 0; j < k; ++j)
                if (ids[(size_t)t * k + j] == e) jj = j;
        }
        const int f = jj >= 0 ? 1 : 0;
        int x = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;
        }
        __syncthreads();
        const int excl = (wid ? warp_tot[wid - 1] : 0) + x - f;
        if (f) {
            const int r = off + s_carry + excl;
            perm_tok[r] = t;
            pos[(size_t)t * k + jj] = r;
            row_gate[r] = gates[(size_t)t * k + jj];
        }
        __syncthreads();
        if (tid == 0) s_carry += warp_tot[31];
        __syncthreads();
    }
}

// One warp per expert-ordered row: X_perm[r] = x[perm_tok[r]] (bf16 rows).
__global__ void __launch_bounds__(256) pf_gather_kernel(const uint4* __restrict__ x, const int* __restrict__ perm_tok,
                                                        const int* __restrict__ offsets, int E, int H,
                                                        uint4* __restrict__ xperm) {
    const int rows = offsets[E];
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int lane = threadIdx.x & 31;
    const int nv = H / 8;
    const uint4* src = x + (size_t)perm_tok[r] * nv;
    uint4* dst = xperm + (size_t)r * nv;
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
}

// One CTA per token: y_t = sum_j out[pos(t, j)] in j order, in fp32 (out
// already carries the gate; f16 values).
__global__ void __launch_bounds__(256) pf_combine_kernel(const __half* __restrict__ outp, const int* __restrict__ pos,
                                                         int k, int H, float* __restrict__ y) {
    const int t = blockIdx.x;
    int rows[16];
    for (int j = 0; j < k; ++j) rows[j] = pos[(size_t)t * k + j];
    for (int c = threadIdx.x * 4; c < H; c += 256 * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const uint2 raw = *reinterpret_cast<const uint2*>(outp + (size_t)rows[j] * H + c);
            const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            const float4 v = make_float4(lo.x, lo.y, hi.x, hi.y);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        *reinterpret_cast<float4*>(y + (size_t)t * H + c) = acc;
    }
}

// Clear the owners of slots [s0, s0+n): slot_for_id of the owner, the owner
// and the stamp (the buffer's contents are about to be overwritten).
__global__ void pf_invalidate_kernel(int s0, int n, int* __restrict__ slot_for_id, int* __restrict__ id_for_slot,
                                     unsigned* __restrict__ stamps) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int s = s0 + i;
        const int o = id_for_slot[s];
        if (o >= 0) slot_for_id[o] = -1;
        id_for_slot[s] = -1;
        stamps[s] = 0u;
    }
}

}  // namespace

// ------------------------------------------------------- grouped GEMM (tcgen05)
//
// Tiles of 128 rows (one expert's rows in expert order) x 256 output columns;
// K in blocks of 64 bf16 (128 bytes, the 128-byte swizzle span).  Persistent:
// CTA c takes tiles c, c + G, ...  Warp roles:
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] per stage
//   warp 1      TMEM allocation (512 columns = two 256-column accumulators) and
//               the MMA issuer (one thread, 4 x K=16 MMAs per stage)
//   warps 2-5   epilogue: thread = accumulator row, tcgen05.ld 32 columns at a
//               time (the next load in flight while one is processed); mode 0 =
//               SwiGLU of the interleaved gate/up columns to bf16 h, mode 1 =
//               gate * value to f16 out.  Each warp transposes its 32 rows x
//               128 bytes through a padded shared-memory block, so every store
//               instruction writes four whole 128-byte lines.
// All waits are bounded; after a failed wait every role stops, the MMA thread
// waits for its issued MMAs, and TMEM is freed before exit.
namespace {

constexpr int GM = 128, GN = 256, GK = 64;
constexpr int GSTAGES = 4;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t A_BYTES = GM * GK * 2;   // 16 KiB
constexpr uint32_t B_BYTES = GN * GK * 2;   // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t EPI_ROW = 144;                 // 128 bytes of a row + 16 bytes of padding
constexpr uint32_t EPI_WARP = 32 * EPI_ROW;       // one epilogue warp's staging block
constexpr size_t GEMM_SMEM = 1024 + (size_t)GSTAGES * STAGE_BYTES + 4 * EPI_WARP + 1024;

struct GemmArgs {
    int E;                 // experts of the layer (tensor-map z extent)
    int nk;                // K blocks
    int n_tiles;           // 256-column tiles per expert
    int mode;              // 0: SwiGLU -> bf16 h; 1: gate * out -> f16
    const int* offsets;    // [E+1] expert row offsets
    __nv_bfloat16* hout;   // mode 0: [rows, F]
    int F;
    __half* fout;          // mode 1: [rows, ldo] f16
    int ldo;
    const float* row_gate; // mode 1: gate of each expert-ordered row
    const float* escale;   // per-expert factor of the weights (NVFP4 global) or null
    unsigned* err;
};

struct TileInfo {
    int e, m0, rows, nt;
};

__device__ __forceinline__ TileInfo decode_tile(int i, const int* s_mt, const int* offsets, int E, int n_tiles) {
    TileInfo ti;
    const int mt = i / n_tiles;
    ti.nt = i - mt * n_tiles;
    int lo = 0, hi = E;  // largest e with s_mt[e] <= mt
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_mt[mid] <= mt) lo = mid; else hi = mid;
    }
    ti.e = lo;
    ti.m0 = offsets[lo] + (mt - s_mt[lo]) * GM;
    ti.rows = min(GM, offsets[lo + 1] - ti.m0);
    return ti;
}

__global__ void __launch_bounds__(GEMM_THREADS, 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                                                                      const __grid_constant__ CUtensorMap mapB,
                                                                      GemmArgs p) {
    extern __shared__ __align__(1024) unsigned char gsm_raw[];
    __shared__ uint64_t full[GSTAGES], empty[GSTAGES], tfull[2], tempty[2], done_bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_mt[1025];
    __shared__ volatile int s_fail;
    unsigned char* gsm = reinterpret_cast<unsigned char*>(((uintptr_t)gsm_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int E = p.E;

    if (tid == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            ft::mbar_init(&full[s], 1);
            ft::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ft::mbar_init(&tfull[a], 1);
            ft::mbar_init(&tempty[a], 4);
        }
        ft::mbar_init(&done_bar, 1);
        ft::mbar_fence_init();
        s_fail = 0;
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            s_mt[e] = acc;
            acc += (p.offsets[e + 1] - p.offsets[e] + GM - 1) / GM;
        }
        s_mt[E] = acc;
    }
    if (wid == 0 && lane == 0) {
        tc::prefetch_map(&mapA);
        tc::prefetch_map(&mapB);
    }
    if (wid == 1) tc::tmem_alloc(&s_tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const int ntiles = s_mt[E] * p.n_tiles;

    if (wid == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int it = 0;
            for (int i = blockIdx.x; i < ntiles && !s_fail; i += gridDim.x) {
                const TileInfo ti = decode_tile(i, s_mt, p.offsets, E, p.n_tiles);
                for (int kb = 0; kb < p.nk; ++kb, ++it) {
                    const int st = it % GSTAGES;
                    if (it >= GSTAGES && !ft::mbar_wait(&empty[st], ((it / GSTAGES) - 1) & 1, p.err)) {
                        s_fail = 1;
                        break;
                    }
                    unsigned char* sa = gsm + (size_t)st * STAGE_BYTES;
                    ft::mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
                    tc::tma_load_2d(sa, &mapA, kb * GK, ti.m0, &full[st]);
                    tc::tma_load_3d(sa + A_BYTES, &mapB, kb * GK, ti.nt * GN, ti.e, &full[st]);
                }
            }
            // every issued stage has landed before exit (bounded)
            for (int j = it - GSTAGES; j < it; ++j)
                if (j >= 0) ft::mbar_wait(&full[j % GSTAGES], (j / GSTAGES) & 1, p.err);
        }
    } else if (wid == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16_f32(GM, GN);
            int it = 0, t = 0;
            for (int i = blockIdx.x; i < ntiles && !s_fail; i += gridDim.x, ++t) {
                const int acc = t & 1;
                if (t >= 2 && !ft::mbar_wait(&tempty[acc], ((t >> 1) - 1) & 1, p.err)) {
                    s_fail = 1;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(acc * GN);
                bool ok = true;
                for (int kb = 0; kb < p.nk; ++kb, ++it) {
                    const int st = it % GSTAGES;
                    if (!ft::mbar_wait(&full[st], (it / GSTAGES) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const unsigned char* sa = gsm + (size_t)st * STAGE_BYTES;
                    const uint64_t ad = tc::sdesc_k_sw128(sa);
                    const uint64_t bd = tc::sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < GK / 16; ++k)
                        tc::mma_bf16(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, (kb | k) ? 1u : 0u);
                    tc::mma_commit(&empty[st]);
                }
                if (!ok) {
                    s_fail = 1;
                    break;
                }
                tc::mma_commit(&tfull[acc]);
            }
            tc::mma_commit(&done_bar);
            ft::mbar_wait(&done_bar, 0, p.err);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = wid & 3;  // TMEM lane quarter of this warp
        const int r = q * 32 + lane;
        unsigned char* eb = gsm + (size_t)GSTAGES * STAGE_BYTES + (size_t)q * EPI_WARP;
        const int rsub = lane >> 3, cq = (lane & 7) * 16;  // read-back: row within 4, byte offset in the line
        int t = 0;
        for (int i = blockIdx.x; i < ntiles && !s_fail; i += gridDim.x, ++t) {
            const int acc = t & 1;
            if (!ft::mbar_wait(&tfull[acc], (t >> 1) & 1, p.err)) {
                s_fail = 1;
                break;
            }
            tc::fence_after_sync();
            const TileInfo ti = decode_tile(i, s_mt, p.offsets, E, p.n_tiles);
            const int row = ti.m0 + r;
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * GN);
            const float es = p.escale ? p.escale[ti.e] : 1.f;
            const float gate = (p.mode == 1 && r < ti.rows) ? p.row_gate[row] * es : 0.f;
            const int wrow0 = ti.m0 + q * 32;  // first row of this warp's block
            // one 32-column chunk of the accumulator row -> this lane's row of the
            // staging block; mode 1: 128 bytes per chunk, mode 0: 32 bytes per
            // chunk (four chunks fill the 128 bytes)
            auto stage = [&](const uint32_t* v, int c) {
                if (p.mode == 0) {
                    uint32_t packed[8];
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) {
                        // columns: 16 gate rows then the 16 matching up rows of
                        // features f0 .. f0+15, f0 = nt*128 + c*16
                        const float g0 = es * __uint_as_float(v[2 * i2]), g1 = es * __uint_as_float(v[2 * i2 + 1]);
                        const float u0 = es * __uint_as_float(v[16 + 2 * i2]);
                        const float u1 = es * __uint_as_float(v[16 + 2 * i2 + 1]);
                        const float h0 = g0 / (1.f + expf(-g0)) * u0;
                        const float h1 = g1 / (1.f + expf(-g1)) * u1;
                        const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                        packed[i2] = *reinterpret_cast<const uint32_t*>(&hb);
                    }
                    uint4* d = reinterpret_cast<uint4*>(eb + lane * EPI_ROW + (c & 3) * 32);
                    d[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    d[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                } else {
                    // gate * value as f16: a chunk's 32 columns are 64 bytes,
                    // half (c & 1) of the staged 128-byte line
                    uint32_t packed[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) {
                        const __half2 hv = __floats2half2_rn(gate * __uint_as_float(v[2 * i2]),
                                                             gate * __uint_as_float(v[2 * i2 + 1]));
                        packed[i2] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    uint4* d = reinterpret_cast<uint4*>(eb + lane * EPI_ROW + (c & 1) * 64);
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2)
                        d[i2] = make_uint4(packed[4 * i2], packed[4 * i2 + 1], packed[4 * i2 + 2], packed[4 * i2 + 3]);
                }
            };
            // the staged 32 rows x 128 bytes -> global, four whole lines per store
            auto flush = [&](int c) {
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int rr = j * 4 + rsub;
                    const int grow = wrow0 + rr;
                    const uint4 v4 = *reinterpret_cast<const uint4*>(eb + rr * EPI_ROW + cq);
                    if (q * 32 + rr < ti.rows) {
                        unsigned char* g =
                            p.mode == 0
                                ? reinterpret_cast<unsigned char*>(p.hout + (size_t)grow * p.F + ti.nt * (GN / 2) +
                                                                   (c >> 2) * 64)
                                : reinterpret_cast<unsigned char*>(p.fout + (size_t)grow * p.ldo + ti.nt * GN +
                                                                   (c >> 1) * 64);
                        *reinterpret_cast<uint4*>(g + cq) = v4;
                    }
                }
                __syncwarp();
            };
            uint32_t va[32], vb[32];
            tc::tmem_ld32(base, va);
#pragma unroll 1
            for (int c = 0; c < GN / 32; c += 2) {
                tc::tmem_wait_ld(va);
                tc::tmem_ld32(base + (uint32_t)((c + 1) * 32), vb);
                stage(va, c);  // c is even: the first half of a line in both modes
                tc::tmem_wait_ld(vb);
                if (c + 2 < GN / 32) tc::tmem_ld32(base + (uint32_t)((c + 2) * 32), va);
                stage(vb, c + 1);
                if (p.mode == 1 || ((c + 1) & 3) == 3) flush(c + 1);  // mode 1: a line per two chunks
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ft::mbar_arrive(&tempty[acc]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (wid == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// ------------------------------------------------------------------ host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// bf16 row-major matrix [rows, cols] (cols contiguous) as a 2-D map with a
// [box_rows x 64] box and 128-byte swizzle (K-major operand tiles).
bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E matrices [rows, cols] bf16, one per record, `record_bytes` apart: a 3-D
// map with a [box_rows x 64 x 1] box.
bool encode_3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t E, uint64_t record_bytes,
               uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {cols, rows, E};
    const cuuint64_t strides[2] = {cols * 2, record_bytes};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

ft_status prefill_alloc(PrefillState& pf, int T_max, int k, int H, int F, int E, int fmt) {
    pf.T_max = T_max;
    pf.E = E; pf.k = k; pf.H = H; pf.F = F;
    pf.fmt = fmt;
    if ((fmt == FT_FMT_NVFP4 || fmt == FT_FMT_MXFP4 || fmt == FT_FMT_FP8) &&
        cudaMalloc(&pf.staging, (size_t)E * 3 * H * F * 2) != cudaSuccess) {
        cudaGetLastError();
        return FT_ERR_OOM;
    }
    const size_t TK = (size_t)T_max * k;
    if (cudaMalloc(&pf.xperm, TK * H * 2) != cudaSuccess || cudaMalloc(&pf.hperm, TK * F * 2) != cudaSuccess ||
        cudaMalloc(&pf.outp, TK * H * 2) != cudaSuccess || cudaMalloc(&pf.ids, TK * 4) != cudaSuccess ||
        cudaMalloc(&pf.gates, TK * 4) != cudaSuccess || cudaMalloc(&pf.perm_tok, TK * 4) != cudaSuccess ||
        cudaMalloc(&pf.pos, TK * 4) != cudaSuccess || cudaMalloc(&pf.row_gate, TK * 4) != cudaSuccess ||
        cudaMalloc(&pf.counts, (size_t)E * 4) != cudaSuccess ||
        cudaMalloc(&pf.offsets, (size_t)(E + 1) * 4) != cudaSuccess) {
        cudaGetLastError();
        return FT_ERR_OOM;
    }
    // rows of the gathered operands that no expert owns stay finite
    if (cudaMemset(pf.xperm, 0, TK * H * 2) != cudaSuccess || cudaMemset(pf.hperm, 0, TK * F * 2) != cudaSuccess)
        return FT_ERR_CUDA;
    for (int b = 0; b < 2; ++b) {
        if (cudaEventCreateWithFlags(&pf.loaded[b], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&pf.released[b], cudaEventDisableTiming) != cudaSuccess)
            return FT_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&pf.fence, cudaEventDisableTiming) != cudaSuccess) return FT_ERR_CUDA;
    if (!encode_2d(&pf.mapA1, pf.xperm, TK, H, GM) || !encode_2d(&pf.mapA2, pf.hperm, TK, F, GM)) return FT_ERR_CUDA;
    return FT_OK;
}

ft_status prefill_set_pool(PrefillState& pf, const uint8_t* pool, size_t rb) {
    const uint64_t E = pf.E, H = pf.H, F = pf.F;
    pf.rb = rb;
    for (int b = 0; b < 2; ++b) {
        // BF16: the GEMMs read the buffer's records in place; NVFP4 and
        // MXFP4: the bf16 staging copy of the layer (one, reused by both
        // buffers in turn)
        const bool staged = pf.fmt == FT_FMT_NVFP4 || pf.fmt == FT_FMT_MXFP4 || pf.fmt == FT_FMT_FP8;
        const uint8_t* base = staged ? static_cast<const uint8_t*>(pf.staging) : pool + (size_t)b * E * rb;
        const uint64_t rbb = staged ? 3 * H * F * 2 : rb;
        if (!encode_3d(&pf.mapB1[b], base, 2 * F, H, E, rbb, GN) ||
            !encode_3d(&pf.mapB2[b], base + 2 * F * H * 2, H, F, E, rbb, GN))
            return FT_ERR_CUDA;
    }
    pf.maps_pool = pool;
    return FT_OK;
}

void prefill_free(PrefillState& pf) {
    cudaFree(pf.xperm);
    cudaFree(pf.hperm);
    cudaFree(pf.outp);
    cudaFree(pf.ids);
    cudaFree(pf.gates);
    cudaFree(pf.perm_tok);
    cudaFree(pf.pos);
    cudaFree(pf.row_gate);
    cudaFree(pf.counts);
    cudaFree(pf.offsets);
    cudaFree(pf.staging);
    for (int b = 0; b < 2; ++b) {
        if (pf.loaded[b]) cudaEventDestroy(pf.loaded[b]);
        if (pf.released[b]) cudaEventDestroy(pf.released[b]);
    }
    if (pf.fence) cudaEventDestroy(pf.fence);
    pf = PrefillState();
}

cudaError_t launch_pf_invalidate(int s0, int n, int* slot_for_id, int* id_for_slot, unsigned* stamps,
                                 cudaStream_t s) {
    pf_invalidate_kernel<<<(n + 255) / 256, 256, 0, s>>>(s0, n, slot_for_id, id_for_slot, stamps);
    return cudaGetLastError();
}

cudaError_t launch_pf_route(PrefillState& pf, const float* logits, int T, unsigned* err, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(pf.counts, 0, (size_t)pf.E * 4, s);
    if (e != cudaSuccess) return e;
    pf_route_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, pf.E, pf.k, pf.ids, pf.gates, pf.counts, err);
    return cudaGetLastError();
}

cudaError_t launch_pf_permute(PrefillState& pf, int T, cudaStream_t s) {
    pf_permute_kernel<<<pf.E, 1024, 0, s>>>(pf.ids, pf.gates, pf.counts, T, pf.E, pf.k, pf.offsets, pf.perm_tok,
                                            pf.pos, pf.row_gate);
    return cudaGetLastError();
}

cudaError_t launch_pf_gather(PrefillState& pf, const void* x, int T, cudaStream_t s) {
    const int rows = T * pf.k;
    pf_gather_kernel<<<(rows + 7) / 8, 256, 0, s>>>(static_cast<const uint4*>(x), pf.perm_tok, pf.offsets, pf.E,
                                                    pf.H, static_cast<uint4*>(pf.xperm));
    return cudaGetLastError();
}

static cudaError_t launch_gemm(const CUtensorMap& A, const CUtensorMap& B, const GemmArgs& a, int num_sms,
                               cudaStream_t s) {
    cudaError_t e = ensure_dynamic_smem((const void*)grouped_gemm_kernel, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<<<num_sms, GEMM_THREADS, GEMM_SMEM, s>>>(A, B, a);
    return cudaGetLastError();
}

cudaError_t launch_pf_gemm1(PrefillState& pf, int buffer, const float* escale, int num_sms, unsigned* err,
                            cudaStream_t s) {
    GemmArgs a{};
    a.escale = escale;
    a.E = pf.E;
    a.nk = pf.H / GK;
    a.n_tiles = 2 * pf.F / GN;
    a.mode = 0;
    a.offsets = pf.offsets;
    a.hout = static_cast<__nv_bfloat16*>(pf.hperm);
    a.F = pf.F;
    a.err = err;
    return launch_gemm(pf.mapA1, pf.mapB1[buffer], a, num_sms, s);
}

cudaError_t launch_pf_gemm2(PrefillState& pf, int buffer, const float* escale, int num_sms, unsigned* err,
                            cudaStream_t s) {
    GemmArgs a{};
    a.escale = escale;
    a.E = pf.E;
    a.nk = pf.F / GK;
    a.n_tiles = pf.H / GN;
    a.mode = 1;
    a.offsets = pf.offsets;
    a.fout = pf.outp;
    a.ldo = pf.H;
    a.row_gate = pf.row_gate;
    a.err = err;
    return launch_gemm(pf.mapA2, pf.mapB2[buffer], a, num_sms, s);
}

cudaError_t launch_pf_combine(PrefillState& pf, int T, float* y, cudaStream_t s) {
    pf_combine_kernel<<<T, 256, 0, s>>>(pf.outp, pf.pos, pf.k, pf.H, y);
    return cudaGetLastError();
}

// ------------------------------------------- NVFP4 / MXFP4 -> bf16 staging

namespace {

// Expand E FP4 records into the bf16 record layout: every weight becomes
// e2m1(value) * block scale, which bf16 holds exactly (at most 6 significant
// bits for an e4m3 scale, 2 for a power-of-two E8M0 scale, within bf16's
// exponent range for every scale a finite weight of magnitude < 2^127 takes);
// the NVFP4 per-expert fp32 global is applied by the GEMM epilogues.  SB is
// the scale block: 16 (e4m3 scales, NVFP4) or 32 (E8M0 scales, MXFP4).  One
// thread per 32 values (one 16-byte group of codes).
template <int SB>
__global__ void __launch_bounds__(256) pf_dequant_kernel(const uint8_t* __restrict__ src, size_t rb4, int E, int H,
                                                         int F, uint8_t* __restrict__ dst) {
    __shared__ float e2m1[16];
    __shared__ float sct[256];  // scale code -> value
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        if (SB == 16) {
            const int e = (i >> 3) & 15, m = i & 7;
            const float v = e == 0 ? ldexpf((float)m / 8.f, -6) : ldexpf(1.f + (float)m / 8.f, e - 7);
            sct[i] = (i & 0x7F) == 0x7F ? __int_as_float(0x7FC00000) : ((i & 0x80) ? -v : v);
        } else {
            // E8M0: 2^(i-127) as its IEEE single bit pattern (code 0: the
            // subnormal 2^-127), code 255 NaN
            sct[i] = __uint_as_float(i == 255 ? 0x7FC00000u : i == 0 ? 0x00400000u : (uint32_t)i << 23);
        }
        if (i < 16) {
            const int c = i & 7;
            const float mag = c < 2 ? 0.5f * (float)c : (1.f + 0.5f * (float)(c & 1)) * (float)(1 << ((c >> 1) - 1));
            e2m1[i] = (i & 8) ? -mag : mag;
        }
    }
    __syncthreads();
    const size_t VGU = (size_t)F * H, VD = (size_t)H * F / 2, SGU = (size_t)2 * F * H / SB;
    const size_t rb16 = (size_t)3 * H * F * 2;
    const size_t gu_units = (size_t)2 * F * H / 32, units = (size_t)3 * H * F / 32;
    const size_t total = units * E;
    constexpr int SPU = 32 / SB;  // scales per unit of 32 values
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (size_t)gridDim.x * blockDim.x) {
        const size_t e = u / units, w = u - e * units;
        const uint8_t* rec = src + e * rb4;
        uint8_t* out = dst + e * rb16;
        const uint8_t* codes;
        const uint8_t* sc;
        uint8_t* o;
        if (w < gu_units) {  // W_gu: value group w of row w / (H/32)
            const size_t r = w / (H / 32), c = w - r * (H / 32);
            codes = rec + r * (H / 2) + c * 16;
            sc = rec + VGU + VD + r * (H / SB) + c * SPU;
            o = out + (r * H + c * 32) * 2;
        } else {
            const size_t w2 = w - gu_units, r = w2 / (F / 32), c = w2 - r * (F / 32);
            codes = rec + VGU + r * (F / 2) + c * 16;
            sc = rec + VGU + VD + SGU + r * (F / SB) + c * SPU;
            o = out + (size_t)2 * F * H * 2 + (r * F + c * 32) * 2;
        }
        const uint4 q = *reinterpret_cast<const uint4*>(codes);
        const float s0 = sct[sc[0]], s1 = SPU == 2 ? sct[sc[SPU - 1]] : s0;
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t b = (wd[i >> 2] >> (8 * (i & 3))) & 255u;
            const float s = i < 8 ? s0 : s1;
            const __nv_bfloat162 v = __floats2bfloat162_rn(e2m1[b & 15] * s, e2m1[b >> 4] * s);
            packed[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
        uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
        for (int i = 0; i < 4; ++i) o4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    }
}

// Expand E block-FP8 records into the bf16 record layout: every weight
// becomes bf16(e4m3(code) * scale(row / 128, k / 128)), one rounding (the
// product of a 4-bit significand and an fp32 scale is not a bf16 in general).
// One thread per 16 values (one 16-byte group of codes).
__global__ void __launch_bounds__(256) pf_dequant_fp8_kernel(const uint8_t* __restrict__ src, size_t rb8, int E,
                                                             int H, int F, uint8_t* __restrict__ dst) {
    const size_t rb16 = (size_t)3 * H * F * 2;
    const size_t units = (size_t)3 * H * F / 16;  // W_gu then W_d, 16 values per unit
    const size_t gu_units = (size_t)2 * F * H / 16;
    const size_t nbg = (size_t)(F / 128) * (H / 128);
    const size_t total = units * E;
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (size_t)gridDim.x * blockDim.x) {
        const size_t e = u / units, w = u - e * units;
        const uint8_t* rec = src + e * rb8;
        const float* sc = reinterpret_cast<const float*>(rec + (size_t)3 * H * F);
        float s;
        if (w < gu_units) {  // W_gu row r (interleaved gate/up groups of 16), columns c*16..
            const size_t r = w / (H / 16), c = w - r * (H / 16);
            const size_t grp = r / 32, i = r - grp * 32;  // i < 16: gate row grp*16+i, else up row grp*16+i-16
            const size_t frow = grp * 16 + (i & 15);
            s = sc[(i < 16 ? 0 : nbg) + (frow / 128) * (H / 128) + (c * 16) / 128];
        } else {
            const size_t w2 = w - gu_units, r = w2 / (F / 16), c = w2 - r * (F / 16);
            s = sc[2 * nbg + (r / 128) * (F / 128) + (c * 16) / 128];
        }
        const uint4 q = *reinterpret_cast<const uint4*>(rec + w * 16);
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t h;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)(wd[i >> 1] >> (16 * (i & 1)))));
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
            const __nv_bfloat162 v = __floats2bfloat162_rn(f.x * s, f.y * s);
            packed[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
        uint4* o4 = reinterpret_cast<uint4*>(dst + e * rb16 + w * 32);
        o4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        o4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
}

}  // namespace

cudaError_t launch_pf_dequant(PrefillState& pf, const uint8_t* layer_records, cudaStream_t s) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (pf.fmt == FT_FMT_FP8)
        pf_dequant_fp8_kernel<<<sms * 8, 256, 0, s>>>(layer_records, pf.rb, pf.E, pf.H, pf.F,
                                                      static_cast<uint8_t*>(pf.staging));
    else if (pf.fmt == FT_FMT_MXFP4)
        pf_dequant_kernel<32><<<sms * 8, 256, 0, s>>>(layer_records, pf.rb, pf.E, pf.H, pf.F,
                                                      static_cast<uint8_t*>(pf.staging));
    else
        pf_dequant_kernel<16><<<sms * 8, 256, 0, s>>>(layer_records, pf.rb, pf.E, pf.H, pf.F,
                                                      static_cast<uint8_t*>(pf.staging));
    return cudaGetLastError();
}
