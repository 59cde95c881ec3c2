// Internal helpers shared by the libft kernels: PTX wrappers for mbarriers,
// bulk (TMA) copies and the global timer, the sticky device error word, and
// the parameter blocks passed to the kernels.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

// Device error bits (latched in ctx->err, read by ft_get_status).
#define FT_DEVERR_ARG      1u   // invalid ids / non-finite logits
#define FT_DEVERR_TIMEOUT  2u   // a bounded wait gave up

// Every spin wait in this library gives up after this many nanoseconds of
// global time, latches FT_DEVERR_TIMEOUT and lets the kernel wind down.
#define FT_WAIT_LIMIT_NS 2000000000ull

// Slots of the int32 info block written by the control kernel.
enum {
    INFO_LAYER = 0, INFO_T, INFO_U, INFO_H, INFO_M, INFO_Q0, INFO_Q1, INFO_Q, INFO_NC,
    INFO_UGPU, INFO_NASSIGN, INFO_CLOCK, INFO_VALID, INFO_WORDS
};
// Cumulative counters (uint64): calls, unique, hits, misses, fills, cpu, assign.
enum { CNT_CALLS = 0, CNT_UNIQUE, CNT_HITS, CNT_MISSES, CNT_FILLS, CNT_CPU, CNT_ASSIGN, CNT_WORDS };

namespace ft {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy and the CTA.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; bounded by limit_ns
// of global time.  Returns false (and latches the timeout bit) on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          uint64_t limit_ns = FT_WAIT_LIMIT_NS) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 0 && globaltimer() - t0 > limit_ns) {
            atomicOr(err, FT_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 evict-first hint for data read once (streamed weights).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// 1-D bulk copy this CTA's shared memory -> global, in the thread's current
// bulk async-group (close it with bulk_commit).  Same alignment rules.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk store of this thread has completed its writes
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 16-byte asynchronous copy global -> shared through the load/store path
// (not the bulk-copy unit), L1 bypassed.  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async issued so far by this thread has landed
// (the arrival is not pre-counted: the barrier's count includes it).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Counter increment that releases this thread's prior writes (and, through
// a preceding warp or CTA barrier, its peers') at GPU scope.
__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Prefetch `bytes` of global memory into L2 (no completion tracking).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Explicit shared-memory loads by 32-bit shared address (for out-of-line
// helpers, where a generic pointer would compile to generic loads).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

// 8 bf16 packed in a uint4 -> 8 floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu_mul(float a, float b) { return a / (1.f + expf(-a)) * b; }


__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Sense-reversing grid barrier over all CTAs of a cooperative launch:
// bar[0] counts arrivals, bar[1] is the generation.  Bounded: gives up after
// FT_WAIT_LIMIT_NS and latches the timeout bit.  Called by one thread per CTA
// between CTA-wide barriers.
__device__ __forceinline__ void grid_barrier(unsigned* bar, unsigned G, unsigned* err) {
    const unsigned gen0 = ld_acquire_gpu(&bar[1]);
    unsigned c;
    // arrival: releases this CTA's writes; the last arrival also acquires everyone's
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(c) : "l"(bar) : "memory");
    if (c == G - 1) {
        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(bar) : "memory");
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(bar + 1), "r"(gen0 + 1u) : "memory");
    } else {
        const uint64_t t0 = globaltimer();
        for (unsigned it = 0; ld_acquire_gpu(&bar[1]) == gen0; ++it) {
            if ((it & 63u) == 63u && globaltimer() - t0 > FT_WAIT_LIMIT_NS) {
                atomicOr(err, FT_DEVERR_TIMEOUT);
                break;
            }
        }
    }
}

// Producer-side drain: wait (bounded) for the last phase of every slot that
// received a copy, so no bulk copy is in flight into shared memory at exit.
// Always the full FT_WAIT_LIMIT_NS, whatever limit the kernel's other waits
// use: a copy still in flight must land before the CTA may exit.
__device__ __forceinline__ void drain_ring(uint64_t* full, int issued, int nst, unsigned* err) {
    for (int it = issued - nst; it < issued; ++it)
        if (it >= 0) mbar_wait(&full[it % nst], (it / nst) & 1, err);
}

__device__ __forceinline__ void st_release_cta(int* p, int v) {
    asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}


// Producer side: wait (bounded) until all G CTAs have copied their part of
// fill i, then order the async proxy after those generic writes.
// Bounded wait until *c >= target (acquire at GPU scope), then order the
// async proxy (bulk copies) after the acquired writes.
__device__ __forceinline__ bool wait_count(const unsigned* c, unsigned target, unsigned* err,
                                           uint64_t limit_ns = FT_WAIT_LIMIT_NS) {
    const uint64_t t0 = globaltimer();
    for (unsigned it = 0;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        if (v >= target) break;
        __nanosleep(64);  // a poll of L2: leave the issue slots to the math warps
        if ((it & 15u) == 15u && globaltimer() - t0 > limit_ns) {
            atomicOr(err, FT_DEVERR_TIMEOUT);
            return false;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

__device__ __forceinline__ bool wait_filled(unsigned* ready, int i, unsigned G, unsigned* err) {
    const uint64_t t0 = globaltimer();
    for (unsigned it = 0;; ++it) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ready + i) : "memory");
        if (v >= G) break;
        if ((it & 63u) == 63u && globaltimer() - t0 > FT_WAIT_LIMIT_NS) {
            atomicOr(err, FT_DEVERR_TIMEOUT);
            return false;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Fused cache fill by TMA, run by ONE thread of CTA c (of G): part c of every
// fill record goes host pool -> shared ring (bulk loads on mbarriers, up to
// `nf` in flight) -> victim slot (bulk stores).  The chunks of all records
// form one stream, so the next record's loads are in flight while a record's
// last stores complete; then the thread orders those async-proxy writes
// before a release and counts the CTA in ready[r].  Ring: nf (<= 4) slots of
// `fch` bytes, barriers fbar[nf]; every wait is bounded.
__device__ __forceinline__ void fill_share_tma(const uint8_t* host, uint8_t* pool, unsigned long long rb, int q,
                                               const int* fslot, const int* ffid, unsigned* ready, int c, int G,
                                               uint8_t* fring, uint64_t* fbar, unsigned fch, int nf, unsigned* err) {
    for (int s = 0; s < nf; ++s) mbar_init(&fbar[s], 1);
    mbar_fence_init();
    const unsigned long long rec16 = rb / 16;
    const unsigned long long per = ((rec16 + G - 1) / G) * 16;
    const unsigned long long b0 = per * (unsigned long long)c;
    const unsigned long long b1 = b0 + per < rb ? b0 + per : rb;
    const int nch = b1 > b0 ? (int)((b1 - b0 + fch - 1) / fch) : 0;  // chunks per record part
    const int total = nch * q;
    auto chunk = [&](int g, const uint8_t*& src, uint8_t*& dst, unsigned& n) {
        const int r = g / nch, j = g - r * nch;
        const unsigned long long o = b0 + (unsigned long long)j * fch;
        n = (unsigned)((b1 - o) < fch ? (b1 - o) : fch);
        src = host + (unsigned long long)ffid[r] * rb + o;
        dst = pool + (unsigned long long)fslot[r] * rb + o;
    };
    int issued = 0, done = 0;
    for (; issued < total && issued < nf; ++issued) {
        const uint8_t* src; uint8_t* dst; unsigned n;
        chunk(issued, src, dst, n);
        mbar_arrive_expect_tx(&fbar[issued], n);
        bulk_g2s(fring + (size_t)issued * fch, src, n, &fbar[issued]);
    }
    bool ok = true;
    for (int r = 0; r < q; ++r) {
        for (int j = 0; j < nch && ok; ++j, ++done) {
            const int g = done, s = g % nf;
            if (!mbar_wait(&fbar[s], (uint32_t)(g / nf) & 1u, err)) { ok = false; break; }
            const uint8_t* src; uint8_t* dst; unsigned n;
            chunk(g, src, dst, n);
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                         "r"(smem_addr(fring + (size_t)s * fch)), "r"(n) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            if (issued < total) {
                chunk(issued, src, dst, n);
                mbar_arrive_expect_tx(&fbar[s], n);
                bulk_g2s(fring + (size_t)s * fch, src, n, &fbar[s]);
                ++issued;
            }
        }
        if (!ok) break;
        // record r's part has landed: publish (async proxy -> generic release)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        atomicAdd(&ready[r], 1u);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    // after a failed wait, loads still in flight land before the CTA may exit (bounded)
    for (int g = done + (ok ? 0 : 1); g < issued; ++g) mbar_wait(&fbar[g % nf], (uint32_t)(g / nf) & 1u, err);
}

}  // namespace ft

// ------------------------------------------------------------- host side

// Raise `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes`.  The attribute belongs to one (kernel, device) pair, so the
// largest size set so far is remembered per pair; the lock makes concurrent
// host threads safe.  A pair that finds the table full is set on every call.
inline cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
    struct Set {
        const void* fn;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static Set tab[256];
    static int n = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    Set* hit = nullptr;
    for (int i = 0; i < n && !hit; ++i)
        if (tab[i].fn == kernel && tab[i].dev == dev) hit = &tab[i];
    if (hit && hit->bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (!hit && n < (int)(sizeof(tab) / sizeof(tab[0]))) {
        hit = &tab[n++];
        hit->fn = kernel;
        hit->dev = dev;
    }
    if (hit) hit->bytes = bytes;
    return cudaSuccess;
}

// ------------------------------------------------------------------ params

struct CtlParams {
    int layer, T, E, k, L, S;
    const float* logits;      // [T,E] or null
    const int* topk_ids;      // [T,k] or null
    const float* topk_w;      // [T,k] or null
    double B_P, B_H;
    int q0_n;                 // q0tab holds q0 for m < q0_n (0: compute on the device)
    int q0tab[257];           // q0 = round((m * B_P) / B_H) in fp64, per miss count m
    int* slot_for_id;         // [L*E]
    int* id_for_slot;         // [S]
    unsigned* stamps;         // [S]
    unsigned* clock;          // [1]
    int* out_ids;             // [T*k]
    float* out_gates;         // [T*k]
    int* out_slots;           // [T*k]  slot or -1
    int* out_pos;             // [T*k]  row of (t,j) in the assignment arrays or -1
    int* wl_slot;             // [E]    slot of GPU entry i (entries ascending expert id)
    int* wl_off;              // [E+1]  first assignment of entry i
    int* wl_fid;              // [E]    flat id of entry i
    int* wl_fill;             // [E]    fill index of entry i, or -1 for a hit
    unsigned* ready;          // [E]    per-fill / per-entry counters of the expert kernel (reset here)
    int* as_tok;              // [T*k]  token of each assignment (entry-major, token ascending)
    float* as_gate;           // [T*k]
    int* fill_slot;           // [E]
    int* fill_fid;            // [E]
    int* out_F;               // [E]
    int* out_C;               // [E]
    int* out_victims;         // [E]
    int* info;                // [INFO_WORDS]
    unsigned long long* counters;  // [CNT_WORDS]
    unsigned* err;
};

struct FillParams {
    const uint4* host_pool;   // device-accessible address of the host pool
    uint4* slot_pool;
    unsigned long long rec16; // record bytes / 16
    const int* info;
    const int* fill_slot;
    const int* fill_fid;
};

struct ExpertParams {
    const uint8_t* slot_pool;
    unsigned long long rb;    // record bytes
    int H, F, T, k;
    const __nv_bfloat16* x;   // [T,H]
    const float* partial_C;   // [T,H] or null
    float* y;                 // [T,H]
    const int* info;
    const int* wl_slot;
    const int* wl_off;
    const int* as_tok;
    const float* as_gate;
    const int* out_pos;
    float* hbuf;              // [T*k, F] fp32
    unsigned* err;
    unsigned* gbar;           // [4] FP4: grid barrier of the x staging (arrivals, generation), exit count,
                              // CTAs done with the resident entries' phase-A items (zero at rest);
                              // BF16: exit count, hits done, fill items drawn; zero at rest
    const int* wl_fid;        // [E] flat id of each GPU entry (NVFP4 global lookup)
    // fused cache fill (performed by this launch when do_fill != 0)
    int do_fill;
    const uint4* host_pool;   // device-accessible address of the host pool
    const int* fill_slot;     // [q] victim slot of fill i
    const int* fill_fid;      // [q] flat id of fill i
    const int* wl_fill;       // [E] fill index of entry i, or -1 for a hit
    unsigned* ready;          // FP4 and block-FP8: [q] CTAs that finished their part of fill i (zeroed by
                              // the control pass); BF16: [ugpu] h features written per entry (zero at rest)
    unsigned* wdc;            // BF16: [q] W_d pieces of fill i stored in its slot; FP4: [q] CTAs done with
                              // the phase-A items of fill i (low half-word) and CTAs whose share of fill
                              // i's W_gu is stored (high half-word) (zero at rest)
    unsigned fill_chunk;      // bytes of one fused-fill ring slot
    int fill_slots;           // fused-fill ring slots (2..4)
    int fill_fpf;             // BF16: features per fused-fill unit
    int fill_nks;             // BF16: K segments per fused-fill unit
    const float* gscale;      // [L*E] FP4 per-expert fp32 global (all 1 for MXFP4), or null
    uint4* x16;               // FP4 decode scratch: T_max x H activations as scaled f16 pairs
    float* xsc;               // FP4 decode scratch: T_max row factors
    unsigned long long wait_ns;  // BF16: limit of the waits on other warps' or CTAs' progress
                                 // (waits for a thread's own copies keep FT_WAIT_LIMIT_NS)
    int tgroup;               // NVFP4: tokens per phase-B item
    int nstage;               // pipeline depth (stages in shared memory)
    unsigned stage_bytes;     // bytes of one stage
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_route_ctl(const CtlParams& p, cudaStream_t s);
cudaError_t launch_fill(const FillParams& p, int grid, cudaStream_t s);
cudaError_t launch_expert_ffn(ExpertParams p, int num_sms, cudaStream_t s);
// whether the BF16 decode kernel has a shared-memory plan for T tokens
bool expert_ffn_fits(int H, int F, int T, int k, int num_sms);
// fmt: FT_FMT_NVFP4 (e4m3 block-16 scales) or FT_FMT_MXFP4 (E8M0 block-32 scales)
cudaError_t launch_expert_ffn_fp4(ExpertParams p, int fmt, int num_sms, cudaStream_t s);
// whether the FP4 kernel has a shared-memory plan for T tokens (checked at init for T_max)
bool expert_ffn_fp4_fits(int H, int F, int T, int k, int fmt, int num_sms);
// block-FP8 records: gate/up + SwiGLU kernel, then down + merge kernel (no fused fill)
cudaError_t launch_expert_ffn_fp8(ExpertParams p, int num_sms, cudaStream_t s);
size_t route_ctl_smem_bytes(int T, int k, int E, int S);
constexpr size_t kCtlSmemMax = 200 * 1024;
