// libft host side: the C ABI declared in include/ft.h.
//
// Owns the context (slot pool, residency maps, LRU stamps, worklists,
// scratch), validates arguments on the host, and enqueues the kernels on the
// caller's streams.  The decode path (ft_route_ctl, ft_moe_forward) performs
// no host synchronisation and no allocation, so a whole decode step can be
// captured into a CUDA graph by the caller.
#include "ft_common.cuh"
#include "ft_prefill.cuh"
#include "../../include/ft.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <cmath>
#include <vector>

// Per-kernel event records of the optional profile.
struct ProfRec {
    int kid;
    cudaEvent_t a, b;
};
struct Profiler {
    bool on = false;
    bool paused = false;
    std::vector<cudaEvent_t> pool;
    std::vector<ProfRec> pending;
    double ms[FT_K_COUNT] = {};
    uint64_t n[FT_K_COUNT] = {};
};

struct ft_ctx {
    int L, E, k, H, F, S, fmt, T_max, T_prefill_max;
    size_t rb;
    int device, num_sms;
    cudaStream_t cs, ts;
    const void* host_pool;
    const uint8_t* host_pool_dev;
    uint8_t* slot_pool;
    int* slot_for_id;
    int* id_for_slot;
    unsigned* stamps;
    float* nvfp4_global;
    uint4* x16;      // FP4 decode: activations as scaled f16 pairs (T_max x H)
    float* xsc;      // FP4 decode: row factors (T_max)
    // fixed-size control outputs and worklists (one arena)
    void* arena;
    unsigned* clock;
    int *ids, *slots_topk, *pos, *as_tok, *wl_slot, *wl_off, *wl_fid, *wl_fill, *fill_slot, *fill_fid, *Fl, *Cl, *victims, *info;
    float *gates, *as_gate;
    unsigned long long* counters;
    unsigned* err;
    unsigned* gbar;
    unsigned* ready;
    unsigned* wdc;
    float* hbuf;
    bool fill_pending;
    unsigned long long wait_ns;  // limit of the BF16 decode kernel's progress waits
    int last_T;
    bool have_ctl;
    PrefillState pf;
    Profiler prof;
};

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

#define FT_CUDA(call)                                                                          \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess) {                                                               \
            if (getenv("FT_DEBUG")) fprintf(stderr, "libft: %s -> %s\n", #call, cudaGetErrorString(e_)); \
            return e_ == cudaErrorMemoryAllocation ? FT_ERR_OOM : FT_ERR_CUDA;                 \
        }                                                                                      \
    } while (0)

cudaEvent_t prof_event(Profiler& pr) {
    if (!pr.pool.empty()) {
        cudaEvent_t e = pr.pool.back();
        pr.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Records an event pair around the launches made in its scope (profile on).
// Inside a stream capture the records become external event-record nodes of
// the graph, so they time every replay of the captured launch.
inline void prof_record(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
        cudaEventRecord(e, s);
}

struct ProfScope {
    Profiler& pr;
    cudaStream_t s;
    ProfRec r{};
    bool rec = false;
    ProfScope(Profiler& p, int kid, cudaStream_t st) : pr(p), s(st) {
        if (!pr.on || pr.paused) return;
        rec = true;
        r.kid = kid;
        r.a = prof_event(pr);
        r.b = prof_event(pr);
        if (r.a) prof_record(r.a, s);
    }
    ~ProfScope() {
        if (!rec || !r.a || !r.b) return;
        prof_record(r.b, s);
        pr.pending.push_back(r);
    }
};

void prof_release(Profiler& pr) {
    for (auto& r : pr.pending) {
        pr.pool.push_back(r.a);
        pr.pool.push_back(r.b);
    }
    pr.pending.clear();
    for (auto e : pr.pool) cudaEventDestroy(e);
    pr.pool.clear();
}

void free_ctx(ft_ctx* c) {
    if (!c) return;
    prof_release(c->prof);
    prefill_free(c->pf);
    cudaFree(c->slot_pool);
    cudaFree(c->slot_for_id);
    cudaFree(c->id_for_slot);
    cudaFree(c->stamps);
    cudaFree(c->nvfp4_global);
    cudaFree(c->x16);
    cudaFree(c->xsc);
    cudaFree(c->arena);
    cudaFree(c->hbuf);
    delete c;
}

// Run a pending cache fill with the standalone kernel (the fill of a control
// pass is normally fused into the following ft_moe_forward).
cudaError_t flush_fill(ft_ctx* c) {
    if (!c->fill_pending) return cudaSuccess;
    c->fill_pending = false;
    FillParams fp{};
    fp.host_pool = (const uint4*)c->host_pool_dev;
    fp.slot_pool = (uint4*)c->slot_pool;
    fp.rec16 = c->rb / 16;
    fp.info = c->info;
    fp.fill_slot = c->fill_slot;
    fp.fill_fid = c->fill_fid;
    ProfScope ps(c->prof, FT_K_FILL, c->cs);
    return launch_fill(fp, 2 * c->num_sms, c->cs);
}

}  // namespace

extern "C" {

int32_t ft_abi_version(void) { return FT_ABI_VERSION; }

const char* ft_status_str(ft_status s) {
    switch (s) {
        case FT_OK: return "ok";
        case FT_ERR_ARG: return "invalid argument";
        case FT_ERR_CUDA: return "CUDA call failed";
        case FT_ERR_OOM: return "out of memory";
        case FT_ERR_CAPACITY: return "cache too small for the request";
        case FT_ERR_TIMEOUT: return "bounded device wait gave up";
        case FT_ERR_STATE: return "call not allowed in the current state";
        case FT_ERR_DEVICE: return "invalid input detected on the device";
        default: return "unknown status";
    }
}

size_t ft_record_bytes(int32_t H, int32_t F, int32_t fmt) {
    const size_t n = (size_t)3 * H * F;
    if (fmt == FT_FMT_BF16) return 2 * n;
    if (fmt == FT_FMT_NVFP4) return n / 2 + n / 16;
    if (fmt == FT_FMT_MXFP4) return n / 2 + n / 32;
    if (fmt == FT_FMT_FP8) return n + (size_t)12 * (H / 128) * (F / 128);
    return 0;
}

ft_status ft_layer_init(ft_ctx** out, int32_t L, int32_t E, int32_t k, int32_t H, int32_t F, int32_t S,
                        int32_t fmt, int32_t T_max, int32_t T_prefill_max, const void* host_pool,
                        const float* nvfp4_global, void* compute_stream, void* transfer_stream) {
    if (!out) return FT_ERR_ARG;
    *out = nullptr;
    if (L < 1 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E || H < 64 || H % 64 || F < 64 || F % 64 || S < 1 ||
        T_max < 1 || T_max > 256 || T_max * k > 4096 || T_prefill_max < 0 || !host_pool)
        return FT_ERR_ARG;
    if (fmt != FT_FMT_BF16 && fmt != FT_FMT_NVFP4 && fmt != FT_FMT_MXFP4 && fmt != FT_FMT_FP8) return FT_ERR_ARG;
    // FP8 records (3HF value bytes + 4 bytes per 128 x 128 block of W_g, W_u and
    // W_d) and their scale matrices must start on 16-byte boundaries
    if (fmt == FT_FMT_FP8 && (nvfp4_global || H % 128 || F % 128 || ((H / 128) * (F / 128)) % 4)) return FT_ERR_ARG;
    if (fmt == FT_FMT_NVFP4 && (!nvfp4_global || H % 256 || F % 256)) return FT_ERR_ARG;
    if (fmt == FT_FMT_MXFP4 && (nvfp4_global || H % 256 || F % 512)) return FT_ERR_ARG;
    if (fmt == FT_FMT_BF16 && nvfp4_global) return FT_ERR_ARG;
    if (route_ctl_smem_bytes(T_max, k, E, S) > kCtlSmemMax) return FT_ERR_ARG;
    if (fmt == FT_FMT_BF16 && (size_t)T_max * H * 2 > 65536) return FT_ERR_ARG;  // BF16 decode stages x in smem
    // prefill: 256-column GEMM tiles over 2F and H, top-k of at most 256 logits
    if (T_prefill_max > 0 && (H % 256 || (2 * F) % 256 || E > 256 || (size_t)T_prefill_max * k > (1u << 30)))
        return FT_ERR_ARG;
    ft_ctx* c = new (std::nothrow) ft_ctx();
    if (!c) return FT_ERR_OOM;
    c->L = L; c->E = E; c->k = k; c->H = H; c->F = F; c->S = S; c->fmt = fmt;
    c->T_max = T_max; c->T_prefill_max = T_prefill_max;
    c->rb = ft_record_bytes(H, F, fmt);
    c->cs = (cudaStream_t)compute_stream;
    c->ts = (cudaStream_t)transfer_stream;
    c->host_pool = host_pool;
    c->wait_ns = FT_WAIT_LIMIT_NS;
    ft_status st = FT_OK;
    auto fail = [&](ft_status s) { free_ctx(c); return s; };
#define INIT_CUDA(call)                                                                        \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess) {                                                               \
            if (getenv("FT_DEBUG")) fprintf(stderr, "libft: %s -> %s\n", #call, cudaGetErrorString(e_)); \
            return fail(e_ == cudaErrorMemoryAllocation ? FT_ERR_OOM : FT_ERR_CUDA);           \
        }                                                                                      \
    } while (0)
    INIT_CUDA(cudaGetDevice(&c->device));
    INIT_CUDA(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device));
    if (fmt == FT_FMT_FP8 && (size_t)T_max * k * ((H + c->num_sms - 1) / c->num_sms) * 4 > 227 * 1024)
        return fail(FT_ERR_ARG);  // the down kernel keeps [assignment, rows] in shared memory
    if (fmt == FT_FMT_NVFP4 || fmt == FT_FMT_MXFP4)
        for (int t = 1; t <= T_max; ++t)  // the FP4 decode kernel needs a shared-memory plan for every T
            if (!expert_ffn_fp4_fits(H, F, t, k, fmt, c->num_sms)) return fail(FT_ERR_ARG);
    if (fmt == FT_FMT_BF16)
        for (int t = 1; t <= T_max; ++t)  // the x staging format switches with T: check every T
            if (!expert_ffn_fits(H, F, t, k, c->num_sms)) return fail(FT_ERR_ARG);
    // Device address of the host pool: the mapping of page-locked memory, or
    // the host address itself where the GPU reads pageable memory directly.
    void* dptr = nullptr;
    if (cudaHostGetDevicePointer(&dptr, const_cast<void*>(host_pool), 0) != cudaSuccess) {
        cudaGetLastError();
        int pageable = 0;
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccessUsesHostPageTables, c->device);
        if (!pageable) return fail(FT_ERR_ARG);
        dptr = const_cast<void*>(host_pool);
    }
    c->host_pool_dev = (const uint8_t*)dptr;
    if ((uintptr_t)dptr % 16) return fail(FT_ERR_ARG);

    INIT_CUDA(cudaMalloc(&c->slot_pool, (size_t)S * c->rb));
    INIT_CUDA(cudaMalloc(&c->slot_for_id, (size_t)L * E * 4));
    INIT_CUDA(cudaMalloc(&c->id_for_slot, (size_t)S * 4));
    INIT_CUDA(cudaMalloc(&c->stamps, (size_t)S * 4));
    INIT_CUDA(cudaMemset(c->slot_for_id, 0xff, (size_t)L * E * 4));
    INIT_CUDA(cudaMemset(c->id_for_slot, 0xff, (size_t)S * 4));
    INIT_CUDA(cudaMemset(c->stamps, 0, (size_t)S * 4));

    const size_t TK = (size_t)T_max * k;
    size_t off = 0;
    auto carve = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_clock = carve(4), o_ids = carve(TK * 4), o_gates = carve(TK * 4), o_slots = carve(TK * 4),
                 o_pos = carve(TK * 4), o_astok = carve(TK * 4), o_asg = carve(TK * 4),
                 o_wls = carve((size_t)E * 4), o_wlo = carve((size_t)(E + 1) * 4), o_wlf = carve((size_t)E * 4), o_wlfill = carve((size_t)E * 4),
                 o_ready = carve((size_t)E * 4), o_wdc = carve((size_t)E * 4),
                 o_fs = carve((size_t)E * 4),
                 o_ff = carve((size_t)E * 4), o_F = carve((size_t)E * 4), o_C = carve((size_t)E * 4),
                 o_v = carve((size_t)E * 4), o_info = carve(INFO_WORDS * 4), o_cnt = carve(CNT_WORDS * 8),
                 o_err = carve(4), o_gbar = carve(16);
    INIT_CUDA(cudaMalloc(&c->arena, off));
    INIT_CUDA(cudaMemset(c->arena, 0, off));
    uint8_t* a = (uint8_t*)c->arena;
    c->clock = (unsigned*)(a + o_clock);
    c->ids = (int*)(a + o_ids);
    c->gates = (float*)(a + o_gates);
    c->slots_topk = (int*)(a + o_slots);
    c->pos = (int*)(a + o_pos);
    c->as_tok = (int*)(a + o_astok);
    c->as_gate = (float*)(a + o_asg);
    c->wl_slot = (int*)(a + o_wls);
    c->wl_off = (int*)(a + o_wlo);
    c->wl_fid = (int*)(a + o_wlf);
    c->wl_fill = (int*)(a + o_wlfill);
    c->ready = (unsigned*)(a + o_ready);
    c->wdc = (unsigned*)(a + o_wdc);
    c->fill_slot = (int*)(a + o_fs);
    c->fill_fid = (int*)(a + o_ff);
    c->Fl = (int*)(a + o_F);
    c->Cl = (int*)(a + o_C);
    c->victims = (int*)(a + o_v);
    c->info = (int*)(a + o_info);
    c->counters = (unsigned long long*)(a + o_cnt);
    c->err = (unsigned*)(a + o_err);
    c->gbar = (unsigned*)(a + o_gbar);
    INIT_CUDA(cudaMalloc(&c->hbuf, TK * F * 4));
    if (nvfp4_global) {
        INIT_CUDA(cudaMalloc(&c->nvfp4_global, (size_t)L * E * 4));
        INIT_CUDA(cudaMemcpy(c->nvfp4_global, nvfp4_global, (size_t)L * E * 4, cudaMemcpyHostToDevice));
    } else if (fmt == FT_FMT_MXFP4) {
        // MXFP4 records carry no global: the shared FP4 kernels read 1.0
        std::vector<float> ones((size_t)L * E, 1.0f);
        INIT_CUDA(cudaMalloc(&c->nvfp4_global, (size_t)L * E * 4));
        INIT_CUDA(cudaMemcpy(c->nvfp4_global, ones.data(), (size_t)L * E * 4, cudaMemcpyHostToDevice));
    }
    if (fmt == FT_FMT_NVFP4 || fmt == FT_FMT_MXFP4) {
        INIT_CUDA(cudaMalloc(&c->x16, (size_t)T_max * H * 2));
        INIT_CUDA(cudaMalloc(&c->xsc, (size_t)T_max * 4));
    }
    if (T_prefill_max > 0) {
        st = prefill_alloc(c->pf, T_prefill_max, k, H, F, E, fmt);
        if (st != FT_OK) return fail(st);
    }
    c->pf.E = E;
    INIT_CUDA(cudaDeviceSynchronize());
#undef INIT_CUDA
    *out = c;
    return FT_OK;
}

ft_status ft_route_ctl(ft_ctx* c, int32_t layer, int32_t T, const float* logits, const int32_t* topk_ids,
                       const float* topk_w, double B_P, double B_H) {
    if (!c || layer < 0 || layer >= c->L || T < 1 || T > c->T_max) return FT_ERR_ARG;
    if (!(B_P > 0.0) || !(B_H > 0.0)) return FT_ERR_ARG;
    if ((logits != nullptr) == (topk_ids != nullptr || topk_w != nullptr)) return FT_ERR_ARG;
    if (!logits && (!topk_ids || !topk_w)) return FT_ERR_ARG;
    if (c->pf.open) return FT_ERR_STATE;
    FT_CUDA(flush_fill(c));
    CtlParams p{};
    p.layer = layer; p.T = T; p.E = c->E; p.k = c->k; p.L = c->L; p.S = c->S;
    p.logits = logits; p.topk_ids = topk_ids; p.topk_w = topk_w;
    p.B_P = B_P; p.B_H = B_H;
    // q0 per miss count, evaluated here with the same fp64 expression the
    // device uses (a product, then a quotient, both rounded to nearest, then
    // round half away from zero): the kernel indexes it instead of running a
    // slow fp64 divide on the critical path
    p.q0_n = 0;
    if (c->E < (int)(sizeof(p.q0tab) / sizeof(p.q0tab[0]))) {
        for (int m = 0; m <= c->E; ++m) {
            const double x = ((double)m * B_P) / B_H;
            const double r = std::round(x);
            p.q0tab[m] = r > 1.0e9 ? 1000000000 : (int)r;
        }
        p.q0_n = c->E + 1;
    }
    p.slot_for_id = c->slot_for_id; p.id_for_slot = c->id_for_slot; p.stamps = c->stamps; p.clock = c->clock;
    p.out_ids = c->ids; p.out_gates = c->gates; p.out_slots = c->slots_topk; p.out_pos = c->pos;
    p.wl_slot = c->wl_slot; p.wl_off = c->wl_off; p.wl_fid = c->wl_fid; p.wl_fill = c->wl_fill; p.ready = c->ready;
    p.as_tok = c->as_tok; p.as_gate = c->as_gate;
    p.fill_slot = c->fill_slot; p.fill_fid = c->fill_fid;
    p.out_F = c->Fl; p.out_C = c->Cl; p.out_victims = c->victims;
    p.info = c->info; p.counters = c->counters; p.err = c->err;
    {
        ProfScope ps(c->prof, FT_K_ROUTE_CTL, c->cs);
        FT_CUDA(launch_route_ctl(p, c->cs));
    }
    c->fill_pending = true;  // performed by the next ft_moe_forward, or flushed
    c->last_T = T;
    c->have_ctl = true;
    return FT_OK;
}

ft_status ft_moe_forward(ft_ctx* c, const void* x, const float* partial_C, float* y) {
    if (!c || !x || !y) return FT_ERR_ARG;
    if (!c->have_ctl) return FT_ERR_STATE;
    if ((const void*)y == x || (const void*)y == (const void*)partial_C) return FT_ERR_ARG;
    ExpertParams p{};
    p.slot_pool = c->slot_pool; p.rb = c->rb; p.H = c->H; p.F = c->F; p.T = c->last_T; p.k = c->k;
    p.x = (const __nv_bfloat16*)x; p.partial_C = partial_C; p.y = y;
    p.info = c->info; p.wl_slot = c->wl_slot; p.wl_off = c->wl_off; p.as_tok = c->as_tok;
    p.as_gate = c->as_gate; p.out_pos = c->pos; p.hbuf = c->hbuf; p.err = c->err; p.gbar = c->gbar;
    p.wl_fid = c->wl_fid; p.gscale = c->nvfp4_global; p.x16 = c->x16; p.xsc = c->xsc;
    p.wait_ns = c->wait_ns;
    p.do_fill = c->fill_pending ? 1 : 0;
    p.host_pool = (const uint4*)c->host_pool_dev;
    p.fill_slot = c->fill_slot;
    p.fill_fid = c->fill_fid;
    p.wl_fill = c->wl_fill;
    p.ready = c->ready;
    p.wdc = c->wdc;
    c->fill_pending = false;
    {
        ProfScope ps(c->prof, FT_K_EXPERT, c->cs);
        if (c->fmt == FT_FMT_NVFP4 || c->fmt == FT_FMT_MXFP4)
            FT_CUDA(launch_expert_ffn_fp4(p, c->fmt, c->num_sms, c->cs));
        else if (c->fmt == FT_FMT_FP8)
            FT_CUDA(launch_expert_ffn_fp8(p, c->num_sms, c->cs));
        else
            FT_CUDA(launch_expert_ffn(p, c->num_sms, c->cs));
    }
    return FT_OK;
}

// -------------------------------------------------------------------- resize

ft_status ft_cache_resize(ft_ctx* c, int32_t S_new) {
    if (!c || S_new < 1) return FT_ERR_ARG;
    if (route_ctl_smem_bytes(c->T_max, c->k, c->E, S_new) > kCtlSmemMax) return FT_ERR_ARG;
    if (c->pf.open) return FT_ERR_STATE;
    FT_CUDA(flush_fill(c));
    FT_CUDA(cudaStreamSynchronize(c->cs));
    if (c->ts) FT_CUDA(cudaStreamSynchronize(c->ts));
    const int S = c->S, LE = c->L * c->E;
    std::vector<int> sfi(LE), ifs(S);
    std::vector<unsigned> stamp(S);
    FT_CUDA(cudaMemcpy(sfi.data(), c->slot_for_id, (size_t)LE * 4, cudaMemcpyDeviceToHost));
    FT_CUDA(cudaMemcpy(ifs.data(), c->id_for_slot, (size_t)S * 4, cudaMemcpyDeviceToHost));
    FT_CUDA(cudaMemcpy(stamp.data(), c->stamps, (size_t)S * 4, cudaMemcpyDeviceToHost));

    // plan: (old slot -> new slot) moves of the kept records
    std::vector<std::pair<int, int>> moves;
    std::vector<int> nifs(S_new, -1);
    std::vector<unsigned> nstamp(S_new, 0u);
    std::vector<int> nsfi = sfi;
    if (S_new >= S) {
        for (int s = 0; s < S; ++s) {
            nifs[s] = ifs[s];
            nstamp[s] = stamp[s];
            if (ifs[s] >= 0) moves.emplace_back(s, s);
        }
    } else {
        std::vector<int> occ;
        for (int s = 0; s < S; ++s)
            if (ifs[s] >= 0) occ.push_back(s);
        std::sort(occ.begin(), occ.end(), [&](int a, int b) {
            return stamp[a] != stamp[b] ? stamp[a] < stamp[b] : a < b;
        });
        const size_t drop = occ.size() > (size_t)S_new ? occ.size() - S_new : 0;
        for (size_t i = 0; i < drop; ++i) nsfi[ifs[occ[i]]] = -1;
        std::vector<int> keep(occ.begin() + drop, occ.end());
        std::sort(keep.begin(), keep.end());
        for (size_t i = 0; i < keep.size(); ++i) {
            const int s = keep[i];
            nifs[i] = ifs[s];
            nstamp[i] = stamp[s];
            nsfi[ifs[s]] = (int)i;
            moves.emplace_back(s, (int)i);
        }
    }
    uint8_t* npool = nullptr;
    int* nifs_d = nullptr;
    unsigned* nstamp_d = nullptr;
    auto undo = [&](ft_status s) {
        cudaFree(npool);
        cudaFree(nifs_d);
        cudaFree(nstamp_d);
        cudaGetLastError();
        return s;
    };
    if (cudaMalloc(&npool, (size_t)S_new * c->rb) != cudaSuccess) return undo(FT_ERR_OOM);
    if (cudaMalloc(&nifs_d, (size_t)S_new * 4) != cudaSuccess) return undo(FT_ERR_OOM);
    if (cudaMalloc(&nstamp_d, (size_t)S_new * 4) != cudaSuccess) return undo(FT_ERR_OOM);
    for (auto& mv : moves) {
        if (cudaMemcpyAsync(npool + (size_t)mv.second * c->rb, c->slot_pool + (size_t)mv.first * c->rb, c->rb,
                            cudaMemcpyDeviceToDevice, c->cs) != cudaSuccess)
            return undo(FT_ERR_CUDA);
    }
    if (cudaMemcpyAsync(nifs_d, nifs.data(), (size_t)S_new * 4, cudaMemcpyHostToDevice, c->cs) != cudaSuccess ||
        cudaMemcpyAsync(nstamp_d, nstamp.data(), (size_t)S_new * 4, cudaMemcpyHostToDevice, c->cs) != cudaSuccess ||
        cudaStreamSynchronize(c->cs) != cudaSuccess)
        return undo(FT_ERR_CUDA);
    // commit: from here on the new cache replaces the old one
    if (cudaMemcpy(c->slot_for_id, nsfi.data(), (size_t)LE * 4, cudaMemcpyHostToDevice) != cudaSuccess)
        return undo(FT_ERR_CUDA);
    cudaFree(c->slot_pool);
    cudaFree(c->id_for_slot);
    cudaFree(c->stamps);
    c->slot_pool = npool;
    c->id_for_slot = nifs_d;
    c->stamps = nstamp_d;
    c->S = S_new;
    c->have_ctl = false;
    return FT_OK;
}

// ------------------------------------------------------------ observability

ft_status ft_get_ctl_state(ft_ctx* c, int32_t* slot_for_id, int32_t* id_for_slot, uint32_t* stamps,
                           uint32_t* clock) {
    if (!c) return FT_ERR_ARG;
    FT_CUDA(flush_fill(c));
    FT_CUDA(cudaStreamSynchronize(c->cs));
    if (slot_for_id) FT_CUDA(cudaMemcpy(slot_for_id, c->slot_for_id, (size_t)c->L * c->E * 4, cudaMemcpyDeviceToHost));
    if (id_for_slot) FT_CUDA(cudaMemcpy(id_for_slot, c->id_for_slot, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
    if (stamps) FT_CUDA(cudaMemcpy(stamps, c->stamps, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
    if (clock) FT_CUDA(cudaMemcpy(clock, c->clock, 4, cudaMemcpyDeviceToHost));
    return FT_OK;
}

ft_status ft_set_ctl_state(ft_ctx* c, const int32_t* slot_for_id, const int32_t* id_for_slot,
                           const uint32_t* stamps, uint32_t clock) {
    if (!c || !slot_for_id || !id_for_slot || !stamps) return FT_ERR_ARG;
    if (c->pf.open) return FT_ERR_STATE;
    const int LE = c->L * c->E, S = c->S;
    for (int s = 0; s < S; ++s) {
        const int o = id_for_slot[s];
        if (o < -1 || o >= LE) return FT_ERR_ARG;
        if (o >= 0 && slot_for_id[o] != s) return FT_ERR_ARG;
        if (stamps[s] > clock) return FT_ERR_ARG;
    }
    for (int f = 0; f < LE; ++f) {
        const int s = slot_for_id[f];
        if (s < -1 || s >= S) return FT_ERR_ARG;
        if (s >= 0 && id_for_slot[s] != f) return FT_ERR_ARG;
    }
    FT_CUDA(flush_fill(c));
    FT_CUDA(cudaStreamSynchronize(c->cs));
    FT_CUDA(cudaMemcpy(c->slot_for_id, slot_for_id, (size_t)LE * 4, cudaMemcpyHostToDevice));
    FT_CUDA(cudaMemcpy(c->id_for_slot, id_for_slot, (size_t)S * 4, cudaMemcpyHostToDevice));
    FT_CUDA(cudaMemcpy(c->stamps, stamps, (size_t)S * 4, cudaMemcpyHostToDevice));
    FT_CUDA(cudaMemcpy(c->clock, &clock, 4, cudaMemcpyHostToDevice));
    c->have_ctl = false;
    return FT_OK;
}

ft_status ft_get_last_ctl(ft_ctx* c, ft_ctl_info* info, int32_t* F, int32_t* C, int32_t* victims,
                          int32_t* topk_ids, float* gates, int32_t* slots_topk) {
    if (!c) return FT_ERR_ARG;
    if (!c->have_ctl) return FT_ERR_STATE;
    FT_CUDA(cudaStreamSynchronize(c->cs));
    int I[INFO_WORDS];
    FT_CUDA(cudaMemcpy(I, c->info, sizeof(I), cudaMemcpyDeviceToHost));
    if (info) {
        info->layer = I[INFO_LAYER]; info->T = I[INFO_T]; info->u = I[INFO_U]; info->h = I[INFO_H];
        info->m = I[INFO_M]; info->q0 = I[INFO_Q0]; info->q1 = I[INFO_Q1]; info->q = I[INFO_Q];
        info->nC = I[INFO_NC]; info->u_gpu = I[INFO_UGPU]; info->n_assign = I[INFO_NASSIGN];
        info->clock = (uint32_t)I[INFO_CLOCK];
    }
    const size_t TK = (size_t)c->last_T * c->k;
    if (F && I[INFO_Q] > 0) FT_CUDA(cudaMemcpy(F, c->Fl, (size_t)I[INFO_Q] * 4, cudaMemcpyDeviceToHost));
    if (C && I[INFO_NC] > 0) FT_CUDA(cudaMemcpy(C, c->Cl, (size_t)I[INFO_NC] * 4, cudaMemcpyDeviceToHost));
    if (victims && I[INFO_Q] > 0) FT_CUDA(cudaMemcpy(victims, c->victims, (size_t)I[INFO_Q] * 4, cudaMemcpyDeviceToHost));
    if (topk_ids) FT_CUDA(cudaMemcpy(topk_ids, c->ids, TK * 4, cudaMemcpyDeviceToHost));
    if (gates) FT_CUDA(cudaMemcpy(gates, c->gates, TK * 4, cudaMemcpyDeviceToHost));
    if (slots_topk) FT_CUDA(cudaMemcpy(slots_topk, c->slots_topk, TK * 4, cudaMemcpyDeviceToHost));
    return FT_OK;
}

ft_status ft_read_slot(ft_ctx* c, int32_t slot, void* host_dst) {
    if (!c || !host_dst || slot < 0 || slot >= c->S) return FT_ERR_ARG;
    FT_CUDA(flush_fill(c));
    FT_CUDA(cudaStreamSynchronize(c->cs));
    if (c->ts) FT_CUDA(cudaStreamSynchronize(c->ts));
    FT_CUDA(cudaMemcpy(host_dst, c->slot_pool + (size_t)slot * c->rb, c->rb, cudaMemcpyDeviceToHost));
    return FT_OK;
}

ft_status ft_get_counters(ft_ctx* c, ft_counters* out) {
    if (!c || !out) return FT_ERR_ARG;
    FT_CUDA(cudaStreamSynchronize(c->cs));
    unsigned long long v[CNT_WORDS];
    FT_CUDA(cudaMemcpy(v, c->counters, sizeof(v), cudaMemcpyDeviceToHost));
    out->calls = v[CNT_CALLS]; out->unique = v[CNT_UNIQUE]; out->hits = v[CNT_HITS];
    out->misses = v[CNT_MISSES]; out->fills = v[CNT_FILLS]; out->cpu = v[CNT_CPU];
    out->assign = v[CNT_ASSIGN];
    return FT_OK;
}

ft_status ft_profile_enable(ft_ctx* c, int32_t enable) {
    if (!c) return FT_ERR_ARG;
    FT_CUDA(cudaStreamSynchronize(c->cs));
    if (c->ts) FT_CUDA(cudaStreamSynchronize(c->ts));
    for (auto& r : c->prof.pending) {
        c->prof.pool.push_back(r.a);
        c->prof.pool.push_back(r.b);
    }
    c->prof.pending.clear();
    for (int i = 0; i < FT_K_COUNT; ++i) {
        c->prof.ms[i] = 0.0;
        c->prof.n[i] = 0;
    }
    c->prof.on = enable != 0;
    c->prof.paused = false;
    return FT_OK;
}

ft_status ft_profile_pause(ft_ctx* c, int32_t paused) {
    if (!c) return FT_ERR_ARG;
    c->prof.paused = paused != 0;
    return FT_OK;
}

ft_status ft_profile_read(ft_ctx* c, ft_profile* out) {
    if (!c || !out) return FT_ERR_ARG;
    FT_CUDA(cudaStreamSynchronize(c->cs));
    if (c->ts) FT_CUDA(cudaStreamSynchronize(c->ts));
    for (auto& r : c->prof.pending) {
        float ms = 0.f;
        FT_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
        c->prof.ms[r.kid] += ms;
        c->prof.n[r.kid] += 1;
        c->prof.pool.push_back(r.a);
        c->prof.pool.push_back(r.b);
    }
    c->prof.pending.clear();
    for (int i = 0; i < FT_K_COUNT; ++i) {
        out->ms[i] = c->prof.ms[i];
        out->launches[i] = c->prof.n[i];
    }
    return FT_OK;
}

const char* ft_kernel_name(int32_t id) {
    static const char* names[FT_K_COUNT] = {"route_ctl", "fill", "expert_ffn", nullptr, "pf_route",
                                            "pf_permute_gather", "pf_gemm1_swiglu", "pf_gemm2", "pf_combine", "pf_h2d", "pf_dequant"};
    return (id >= 0 && id < FT_K_COUNT) ? names[id] : nullptr;
}

int32_t ft_num_slots(const ft_ctx* c) { return c ? c->S : 0; }

ft_status ft_get_status(ft_ctx* c) {
    if (!c) return FT_ERR_ARG;
    if (flush_fill(c) != cudaSuccess) return FT_ERR_CUDA;
    cudaError_t e1 = cudaStreamSynchronize(c->cs);
    cudaError_t e2 = c->ts ? cudaStreamSynchronize(c->ts) : cudaSuccess;
    if (e1 != cudaSuccess || e2 != cudaSuccess) return FT_ERR_CUDA;
    unsigned e = 0;
    if (cudaMemcpy(&e, c->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return FT_ERR_CUDA;
    if (e) {
        const unsigned z = 0;
        if (cudaMemcpy(c->err, &z, 4, cudaMemcpyHostToDevice) != cudaSuccess) return FT_ERR_CUDA;
    }
    if (e & FT_DEVERR_TIMEOUT) {
        // A wait that gave up may have left a fill record incomplete: every
        // slot is evicted, and the host pool refills the cache on demand.
        if (cudaMemset(c->slot_for_id, 0xff, (size_t)c->L * c->E * 4) != cudaSuccess ||
            cudaMemset(c->id_for_slot, 0xff, (size_t)c->S * 4) != cudaSuccess ||
            cudaMemset(c->stamps, 0, (size_t)c->S * 4) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return FT_ERR_CUDA;
        c->have_ctl = false;
        return FT_ERR_TIMEOUT;
    }
    if (e & FT_DEVERR_ARG) return FT_ERR_DEVICE;
    return FT_OK;
}

ft_status ft_set_wait_limit(ft_ctx* c, uint64_t ns) {
    if (!c || (ns != 0 && (ns < 1000 || ns > FT_WAIT_LIMIT_NS))) return FT_ERR_ARG;
    c->wait_ns = ns ? ns : FT_WAIT_LIMIT_NS;
    return FT_OK;
}

void ft_destroy(ft_ctx* c) {
    if (!c) return;
    cudaStreamSynchronize(c->cs);
    if (c->ts) cudaStreamSynchronize(c->ts);
    free_ctx(c);
}

// ------------------------------------------------------------------ prefill

ft_status ft_prefill_begin(ft_ctx* c, int32_t layer) {
    if (!c || layer < 0 || layer >= c->L) return FT_ERR_ARG;
    if (c->T_prefill_max <= 0 || c->pf.open) return FT_ERR_STATE;
    if (c->S < 2 * c->E) return FT_ERR_CAPACITY;
    FT_CUDA(flush_fill(c));
    if (c->pf.maps_pool != c->slot_pool) {
        const ft_status st = prefill_set_pool(c->pf, c->slot_pool, c->rb);
        if (st != FT_OK) return st;
    }
    PrefillState& pf = c->pf;
    cudaStream_t ts = c->ts ? c->ts : c->cs;
    const size_t layer_bytes = (size_t)c->E * c->rb;
    // buffer 0: clear its owners after earlier decode work, then the begin
    // fence orders the copy after everything enqueued so far on compute
    FT_CUDA(launch_pf_invalidate(0, c->E, c->slot_for_id, c->id_for_slot, c->stamps, c->cs));
    FT_CUDA(cudaEventRecord(pf.fence, c->cs));
    FT_CUDA(cudaStreamWaitEvent(ts, pf.fence, 0));
    {
        ProfScope ps(c->prof, FT_K_PF_H2D, ts);
        FT_CUDA(cudaMemcpyAsync(c->slot_pool, static_cast<const uint8_t*>(c->host_pool) + (size_t)layer * layer_bytes,
                                layer_bytes, cudaMemcpyHostToDevice, ts));
    }
    FT_CUDA(cudaEventRecord(pf.loaded[0], ts));
    pf.open = true;
    pf.cur = 0;
    pf.buf_layer[0] = layer;
    pf.buf_layer[1] = -1;
    c->have_ctl = false;
    return FT_OK;
}

ft_status ft_prefill_layer(ft_ctx* c, int32_t buffer, int32_t layer, int32_t next_layer, int32_t T, const void* x,
                           const float* logits, float* y) {
    if (!c || !x || !logits || !y) return FT_ERR_ARG;
    PrefillState& pf = c->pf;
    if (!pf.open) return FT_ERR_STATE;
    if (buffer != pf.cur || layer != pf.buf_layer[buffer]) return FT_ERR_STATE;
    if (T < 1 || T > c->T_prefill_max || next_layer < -1 || next_layer >= c->L) return FT_ERR_ARG;
    cudaStream_t cs = c->cs, ts = c->ts ? c->ts : c->cs;
    const int nb = buffer ^ 1;
    const size_t layer_bytes = (size_t)c->E * c->rb;
    if (next_layer >= 0) {
        // the other buffer is released once the previous layer's GEMMs (earlier
        // on compute) are done; its owners are cleared before it is overwritten
        FT_CUDA(launch_pf_invalidate(nb * c->E, c->E, c->slot_for_id, c->id_for_slot, c->stamps, cs));
        FT_CUDA(cudaEventRecord(pf.released[nb], cs));
        FT_CUDA(cudaStreamWaitEvent(ts, pf.released[nb], 0));
        {
            ProfScope ps(c->prof, FT_K_PF_H2D, ts);
            FT_CUDA(cudaMemcpyAsync(c->slot_pool + (size_t)nb * layer_bytes,
                                    static_cast<const uint8_t*>(c->host_pool) + (size_t)next_layer * layer_bytes,
                                    layer_bytes, cudaMemcpyHostToDevice, ts));
        }
        FT_CUDA(cudaEventRecord(pf.loaded[nb], ts));
        pf.buf_layer[nb] = next_layer;
    }
    FT_CUDA(cudaStreamWaitEvent(cs, pf.loaded[buffer], 0));
    const float* escale = nullptr;
    if (c->fmt == FT_FMT_NVFP4 || c->fmt == FT_FMT_MXFP4 || c->fmt == FT_FMT_FP8) {
        ProfScope ps(c->prof, FT_K_PF_DEQUANT, cs);
        FT_CUDA(launch_pf_dequant(pf, c->slot_pool + (size_t)buffer * layer_bytes, cs));
        if (c->fmt == FT_FMT_NVFP4) escale = c->nvfp4_global + (size_t)layer * c->E;
    }
    {
        ProfScope ps(c->prof, FT_K_PF_ROUTE, cs);
        FT_CUDA(launch_pf_route(pf, logits, T, c->err, cs));
    }
    {
        ProfScope ps(c->prof, FT_K_PF_PERMUTE, cs);
        FT_CUDA(launch_pf_permute(pf, T, cs));
        FT_CUDA(launch_pf_gather(pf, x, T, cs));
    }
    {
        ProfScope ps(c->prof, FT_K_PF_GEMM1, cs);
        FT_CUDA(launch_pf_gemm1(pf, buffer, escale, c->num_sms, c->err, cs));
    }
    {
        ProfScope ps(c->prof, FT_K_PF_GEMM2, cs);
        FT_CUDA(launch_pf_gemm2(pf, buffer, escale, c->num_sms, c->err, cs));
    }
    {
        ProfScope ps(c->prof, FT_K_PF_COMBINE, cs);
        FT_CUDA(launch_pf_combine(pf, T, y, cs));
    }
    if (next_layer < 0) {
        pf.open = false;
        pf.buf_layer[0] = pf.buf_layer[1] = -1;
        pf.cur = 0;
    } else {
        pf.cur = nb;
    }
    return FT_OK;
}


ft_status ft_measure_link(ft_ctx* c, int32_t n_records, int32_t reps, double* gbps) {
    if (!c || !gbps || n_records < 1 || (long long)n_records > (long long)c->L * c->E || reps < 1 || reps > 1000)
        return FT_ERR_ARG;
    if (c->pf.open) return FT_ERR_STATE;
    FT_CUDA(flush_fill(c));
    FT_CUDA(cudaStreamSynchronize(c->cs));
    const size_t rec = c->rb, lists = ((size_t)(INFO_WORDS + 2 * n_records) * 4 + 255) & ~(size_t)255;
    unsigned char* buf = nullptr;
    if (cudaMalloc(&buf, lists + (size_t)n_records * rec) != cudaSuccess) {
        cudaGetLastError();
        return FT_ERR_OOM;
    }
    std::vector<int> h(INFO_WORDS + 2 * (size_t)n_records, 0);
    h[INFO_Q] = n_records;
    const long long nid = (long long)c->L * c->E;
    for (int i = 0; i < n_records; ++i) {
        h[INFO_WORDS + i] = i;                                                // destination record i
        h[INFO_WORDS + n_records + i] = (int)((long long)i * nid / n_records);  // flat id, spread over the pool
    }
    ft_status st = FT_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    float best = -1.f;
    if (cudaMemcpy(buf, h.data(), h.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        st = FT_ERR_CUDA;
    } else {
        FillParams fp{};
        fp.host_pool = (const uint4*)c->host_pool_dev;
        fp.slot_pool = (uint4*)(buf + lists);
        fp.rec16 = rec / 16;
        fp.info = reinterpret_cast<const int*>(buf);
        fp.fill_slot = reinterpret_cast<const int*>(buf) + INFO_WORDS;
        fp.fill_fid = reinterpret_cast<const int*>(buf) + INFO_WORDS + n_records;
        for (int r = 0; r < reps && st == FT_OK; ++r) {
            float ms = 0.f;
            if (cudaEventRecord(e0, c->cs) != cudaSuccess || launch_fill(fp, 2 * c->num_sms, c->cs) != cudaSuccess ||
                cudaEventRecord(e1, c->cs) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
                st = FT_ERR_CUDA;
            else if (best < 0.f || ms < best)
                best = ms;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(buf);
    if (st != FT_OK) return st;
    *gbps = best > 0.f ? (double)n_records * (double)rec / (best * 1e-3) / 1e9 : 0.0;
    return FT_OK;
}

}  // extern "C"
