// Prefill state of a context: the double-buffer events and the scratch of
// the grouped-GEMM path.  Internal to libft.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ft.h"

struct PrefillState {
    bool open = false;
    int T_max = 0;
    int E = 0, k = 0, H = 0, F = 0;
    int buf_layer[2] = {-1, -1};   // layer held (or being streamed) by each buffer
    cudaEvent_t loaded[2] = {nullptr, nullptr};
    cudaEvent_t released[2] = {nullptr, nullptr};
    cudaEvent_t fence = nullptr;
    // scratch (sized for T_max)
    void* xperm = nullptr;    // bf16 [T*k, H]  tokens gathered in expert order
    void* hperm = nullptr;    // bf16 [T*k, F]  SwiGLU activations in expert order
    float* outp = nullptr;    // fp32 [T*k, H]  per-assignment expert outputs
    int* ids = nullptr;       // [T*k]
    float* gates = nullptr;   // [T*k]
    int* perm_tok = nullptr;  // [T*k] token of each expert-ordered assignment
    int* pos = nullptr;       // [T*k] expert-ordered position of assignment (t, j)
    int* counts = nullptr;    // [E]
    int* offsets = nullptr;   // [E+1]
    int* tiles = nullptr;     // tile schedule
};

ft_status prefill_alloc(PrefillState& pf, int T_max, int k, int H, int F, int E);
void prefill_free(PrefillState& pf);
