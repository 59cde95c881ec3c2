// ft_expert_ffn_noalloc: the decode expert FFN for callers that cannot
// allocate device memory.
//
// Some callers of this library may not call cudaMalloc once they are
// running: serving engines that carve all device memory into their own pools
// at start-up and forbid later allocations, and latency-critical paths where
// the implicit device synchronisation of cudaMalloc / cudaFree is not
// acceptable.  A context (ft_layer_init) allocates its slot pool, maps and
// scratch, so those callers need a context-free entry point.  This one runs
// the same expert kernel as ft_moe_forward, on records the caller already
// holds in device memory, and keeps its scratch (the SwiGLU activations h,
// the worklist, the completion counters and an error word) in one file-scope
// device array of fixed size.
//
// That array exists once per device that loads the library and stays
// allocated until the process exits.  Every call shares it and finds the
// previous call's contents there: the preparation kernel rewrites every
// field the expert kernel reads, and the completion counters return to their
// resting value (zero) after each call.  The error word is sticky: problems
// found by any call (an out-of-range record index, a bounded wait that gave
// up) stay latched until ft_noalloc_status reads and clears them.  Calls
// that overlap on the GPU (different streams, or concurrent host threads)
// race on the array and must not be issued.
#include "ft_common.cuh"
#include "../../include/ft.h"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FT_NOALLOC_SCRATCH_BYTES];

constexpr int PREP_THREADS = 512;
constexpr int MAX_ROUTES = 1024;  // T*k
// Byte offsets inside the scratch array.
constexpr size_t OFF_INFO = 0;       // int[INFO_WORDS]
constexpr size_t OFF_GBAR = 128;     // unsigned[4]: completion words, zero at load, self-resetting
constexpr size_t OFF_ERR = 192;      // unsigned
constexpr size_t OFF_META = 256;     // worklist arrays, MAX_ROUTES entries each
constexpr size_t OFF_DONE = 32768;   // unsigned[MAX_ROUTES]: h features written per entry
constexpr size_t OFF_H = 65536;      // fp32 h [T*k, F]
static_assert(OFF_META + (5 * MAX_ROUTES + 1) * 4 <= OFF_DONE, "worklist overlaps the counters");
static_assert(OFF_DONE + MAX_ROUTES * 4 <= OFF_H, "counters overlap h");

// Worklist of the expert kernel from per-route record indices: entries are
// the distinct records in ascending index, each with its routes in (t, j)
// order.  One CTA; O((T*k)^2 / threads) work for at most 1024 routes.
__global__ void __launch_bounds__(PREP_THREADS) noalloc_prep_kernel(const int* __restrict__ route_records,
                                                                    const float* __restrict__ gates, int T, int k,
                                                                    int n_records, unsigned char* scratch) {
    __shared__ int s_rec[MAX_ROUTES];
    __shared__ float s_g[MAX_ROUTES];
    __shared__ unsigned char s_lead[MAX_ROUTES];
    __shared__ int s_ug, s_na, s_bad;
    const int TK = T * k, tid = threadIdx.x;
    int* info = reinterpret_cast<int*>(scratch + OFF_INFO);
    int* wl_slot = reinterpret_cast<int*>(scratch + OFF_META);
    int* wl_off = wl_slot + MAX_ROUTES;
    int* as_tok = wl_off + MAX_ROUTES + 1;
    float* as_gate = reinterpret_cast<float*>(as_tok + MAX_ROUTES);
    int* out_pos = reinterpret_cast<int*>(as_gate + MAX_ROUTES);
    unsigned* done = reinterpret_cast<unsigned*>(scratch + OFF_DONE);
    for (int i = tid; i < MAX_ROUTES; i += PREP_THREADS) done[i] = 0u;
    if (tid == 0) {
        s_ug = 0;
        s_na = 0;
        s_bad = 0;
    }
    __syncthreads();
    for (int a = tid; a < TK; a += PREP_THREADS) {
        const int r = route_records[a];
        if (r < -1 || r >= n_records) s_bad = 1;
        s_rec[a] = r;
        s_g[a] = gates[a];
    }
    __syncthreads();
    // an index outside [-1, n_records) latches the error and the call routes
    // nothing to the GPU: y = partial_C
    if (s_bad) {
        for (int a = tid; a < TK; a += PREP_THREADS) s_rec[a] = -1;
        if (tid == 0) atomicOr(reinterpret_cast<unsigned*>(scratch + OFF_ERR), FT_DEVERR_ARG);
    }
    __syncthreads();
    for (int a = tid; a < TK; a += PREP_THREADS) {
        const int r = s_rec[a];
        bool lead = r >= 0;
        for (int a2 = 0; a2 < a && lead; ++a2) lead = s_rec[a2] != r;
        s_lead[a] = lead ? 1 : 0;
    }
    __syncthreads();
    for (int a = tid; a < TK; a += PREP_THREADS) {
        const int r = s_rec[a];
        if (r < 0) {
            out_pos[a] = -1;
            continue;
        }
        int ent = 0, off = 0, rank = 0;
        for (int a2 = 0; a2 < TK; ++a2) {
            const int r2 = s_rec[a2];
            if (r2 >= 0 && r2 < r) {
                ++off;
                ent += s_lead[a2];
            }
            if (a2 < a && r2 == r) ++rank;
        }
        const int pos = off + rank;
        as_tok[pos] = a / k;
        as_gate[pos] = s_g[a];
        out_pos[a] = pos;
        if (s_lead[a]) {
            wl_slot[ent] = r;
            wl_off[ent] = off;
            atomicAdd(&s_ug, 1);
        }
        atomicAdd(&s_na, 1);
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < INFO_WORDS; ++i) info[i] = 0;
        info[INFO_T] = T;
        info[INFO_UGPU] = s_ug;
        info[INFO_NASSIGN] = s_na;
        info[INFO_VALID] = 1;
        wl_off[s_ug] = s_na;
    }
}

struct DeviceSetup {
    unsigned char* scratch = nullptr;
    int num_sms = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[64];

// Set-up, once per device, with that device current: the device address of
// the scratch array (in host code the array's name is only a stand-in) and
// the SM count.  Returns false on a CUDA error.
bool device_setup(DeviceSetup& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_setup[dev].scratch) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        g_setup[dev].scratch = static_cast<unsigned char*>(ptr);
        g_setup[dev].num_sms = sms;
    }
    out = g_setup[dev];
    return true;
}

}  // namespace

extern "C" ft_status ft_expert_ffn_noalloc(const void* records, int32_t n_records, const int32_t* route_records,
                                           const float* gates, const void* x, const float* partial_C, float* y,
                                           int32_t T, int32_t k, int32_t H, int32_t F, void* stream) {
    if (!records || !route_records || !gates || !x || !y || n_records < 1 || T < 1 || k < 1 || k > 16 ||
        T * k > MAX_ROUTES || H < 64 || H % 64 || F < 64 || F % 64 || (size_t)T * H * 2 > 65536)
        return FT_ERR_ARG;
    if ((const void*)y == x || (const void*)y == (const void*)partial_C || (uintptr_t)records % 16)
        return FT_ERR_ARG;
    if (OFF_H + (size_t)T * k * F * 4 > FT_NOALLOC_SCRATCH_BYTES) return FT_ERR_ARG;

    DeviceSetup ds;
    if (!device_setup(ds)) return FT_ERR_CUDA;
    if (!expert_ffn_fits(H, F, T, k, ds.num_sms)) return FT_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    noalloc_prep_kernel<<<1, PREP_THREADS, 0, s>>>(route_records, gates, T, k, n_records, ds.scratch);
    if (cudaGetLastError() != cudaSuccess) return FT_ERR_CUDA;

    unsigned char* sc = ds.scratch;
    int* wl_slot = reinterpret_cast<int*>(sc + OFF_META);
    int* wl_off = wl_slot + MAX_ROUTES;
    int* as_tok = wl_off + MAX_ROUTES + 1;
    float* as_gate = reinterpret_cast<float*>(as_tok + MAX_ROUTES);
    int* out_pos = reinterpret_cast<int*>(as_gate + MAX_ROUTES);
    ExpertParams p{};
    p.slot_pool = static_cast<const uint8_t*>(records);
    p.rb = ft_record_bytes(H, F, FT_FMT_BF16);
    p.H = H; p.F = F; p.T = T; p.k = k;
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.partial_C = partial_C;
    p.y = y;
    p.info = reinterpret_cast<const int*>(sc + OFF_INFO);
    p.wl_slot = wl_slot;
    p.wl_off = wl_off;
    p.as_tok = as_tok;
    p.as_gate = as_gate;
    p.out_pos = out_pos;
    p.hbuf = reinterpret_cast<float*>(sc + OFF_H);
    p.err = reinterpret_cast<unsigned*>(sc + OFF_ERR);
    p.gbar = reinterpret_cast<unsigned*>(sc + OFF_GBAR);
    p.ready = reinterpret_cast<unsigned*>(sc + OFF_DONE);
    return launch_expert_ffn(p, ds.num_sms, s) == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

extern "C" ft_status ft_noalloc_status(void* stream) {
    DeviceSetup ds;
    if (!device_setup(ds)) return FT_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FT_ERR_CUDA;
    unsigned* err = reinterpret_cast<unsigned*>(ds.scratch + OFF_ERR);
    unsigned e = 0;
    if (cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return FT_ERR_CUDA;
    if (e) {
        const unsigned z = 0;
        if (cudaMemcpy(err, &z, 4, cudaMemcpyHostToDevice) != cudaSuccess) return FT_ERR_CUDA;
    }
    if (e & FT_DEVERR_TIMEOUT) return FT_ERR_TIMEOUT;
    if (e & FT_DEVERR_ARG) return FT_ERR_DEVICE;
    return FT_OK;
}
