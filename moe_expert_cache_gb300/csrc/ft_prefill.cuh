// Prefill state of a context: the double-buffer events, the tensor maps of
// the grouped GEMMs and the scratch of the prefill path.  Internal to libft.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ft.h"

struct PrefillState {
    bool open = false;
    int T_max = 0;
    int E = 0, k = 0, H = 0, F = 0;
    int cur = 0;                   // buffer holding the layer to compute next
    int buf_layer[2] = {-1, -1};   // layer held (or being streamed) by each buffer
    cudaEvent_t loaded[2] = {nullptr, nullptr};
    cudaEvent_t released[2] = {nullptr, nullptr};
    cudaEvent_t fence = nullptr;
    // scratch (sized for T_max)
    void* xperm = nullptr;    // bf16 [T*k, H]  tokens gathered in expert order
    void* hperm = nullptr;    // bf16 [T*k, F]  SwiGLU activations in expert order
    __half* outp = nullptr;   // f16 [T*k, H]  gate * expert output per row (summed in fp32 by the combine)
    int* ids = nullptr;       // [T*k]
    float* gates = nullptr;   // [T*k]
    int* perm_tok = nullptr;  // [T*k] token of each expert-ordered row
    int* pos = nullptr;       // [T*k] expert-ordered row of route (t, j)
    float* row_gate = nullptr;// [T*k] gate of each expert-ordered row
    int* counts = nullptr;    // [E]
    int* offsets = nullptr;   // [E+1]
    int fmt = 0;              // record format of the slot pool
    size_t rb = 0;            // record bytes in the slot pool
    void* staging = nullptr;  // NVFP4: the layer's E records expanded to bf16 (e2m1 * e4m3, exact)
    // tensor maps: A operands are fixed scratch; B operands follow the slot pool
    CUtensorMap mapA1, mapA2;       // X_perm [T_max*k, H], h [T_max*k, F]
    CUtensorMap mapB1[2], mapB2[2]; // W_gu, W_d of the E records of buffer b
    const void* maps_pool = nullptr; // slot pool the B maps were encoded for
};

ft_status prefill_alloc(PrefillState& pf, int T_max, int k, int H, int F, int E, int fmt);
void prefill_free(PrefillState& pf);
// (Re)encode the B tensor maps for a slot pool (after init or a resize).
ft_status prefill_set_pool(PrefillState& pf, const uint8_t* slot_pool, size_t record_bytes);

// Launchers of the prefill kernels (all on stream s).
cudaError_t launch_pf_invalidate(int s0, int n, int* slot_for_id, int* id_for_slot, unsigned* stamps,
                                 cudaStream_t s);
cudaError_t launch_pf_route(PrefillState& pf, const float* logits, int T, unsigned* err, cudaStream_t s);
cudaError_t launch_pf_permute(PrefillState& pf, int T, cudaStream_t s);
cudaError_t launch_pf_gather(PrefillState& pf, const void* x, int T, cudaStream_t s);
cudaError_t launch_pf_dequant(PrefillState& pf, const uint8_t* layer_records, cudaStream_t s);
// expert_scale: per-expert fp32 factor of this layer's weights (NVFP4 global), or null
cudaError_t launch_pf_gemm1(PrefillState& pf, int buffer, const float* expert_scale, int num_sms, unsigned* err,
                            cudaStream_t s);
cudaError_t launch_pf_gemm2(PrefillState& pf, int buffer, const float* expert_scale, int num_sms, unsigned* err,
                            cudaStream_t s);
cudaError_t launch_pf_combine(PrefillState& pf, int T, float* y, cudaStream_t s);
