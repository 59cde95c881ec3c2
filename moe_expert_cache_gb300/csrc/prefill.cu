// Prefill path of the expert cache (full-layer double buffer + grouped GEMM).
#include "ft_common.cuh"
#include "ft_prefill.cuh"

ft_status prefill_alloc(PrefillState& pf, int T_max, int k, int H, int F, int E) {
    pf.T_max = T_max;
    pf.E = E; pf.k = k; pf.H = H; pf.F = F;
    const size_t TK = (size_t)T_max * k;
    if (cudaMalloc(&pf.xperm, TK * H * 2) != cudaSuccess || cudaMalloc(&pf.hperm, TK * F * 2) != cudaSuccess ||
        cudaMalloc(&pf.outp, TK * H * 4) != cudaSuccess || cudaMalloc(&pf.ids, TK * 4) != cudaSuccess ||
        cudaMalloc(&pf.gates, TK * 4) != cudaSuccess || cudaMalloc(&pf.perm_tok, TK * 4) != cudaSuccess ||
        cudaMalloc(&pf.pos, TK * 4) != cudaSuccess || cudaMalloc(&pf.counts, (size_t)E * 4) != cudaSuccess ||
        cudaMalloc(&pf.offsets, (size_t)(E + 1) * 4) != cudaSuccess) {
        cudaGetLastError();
        return FT_ERR_OOM;
    }
    for (int b = 0; b < 2; ++b) {
        if (cudaEventCreateWithFlags(&pf.loaded[b], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&pf.released[b], cudaEventDisableTiming) != cudaSuccess)
            return FT_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&pf.fence, cudaEventDisableTiming) != cudaSuccess) return FT_ERR_CUDA;
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
    cudaFree(pf.counts);
    cudaFree(pf.offsets);
    cudaFree(pf.tiles);
    for (int b = 0; b < 2; ++b) {
        if (pf.loaded[b]) cudaEventDestroy(pf.loaded[b]);
        if (pf.released[b]) cudaEventDestroy(pf.released[b]);
    }
    if (pf.fence) cudaEventDestroy(pf.fence);
    pf = PrefillState();
}
