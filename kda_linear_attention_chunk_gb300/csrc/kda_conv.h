// kda_conv.h -- launch interface of the short-conv prologue kernels
// (kda_conv.cu) for the C ABI (kda_api.cu).  Not installed; the public
// interface is include/kda.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// causal depthwise conv over each sequence's rows (4 taps: 3 carried in the
// window, the current row), optional SiLU, L2 norm of each head's q and k
struct ConvArgs {
    const void *x[3];               // q, k, v projections [T][H][128] bf16
    void *y[3];                     // q, k, v out [T][H][128] bf16
    const float *weight;            // [3][H*128][4] fp32
    const int32_t *cu_seqlens;      // [N+1]
    const int32_t *conv_slots;      // [N] or nullptr (entry n)
    void *conv_pool;                // [num_slots][3 taps][3][H*128] bf16
    int N, T, H, num_slots;
    int activation;                 // 0 none, 1 SiLU
    float eps;
    cudaStream_t stream;
    int *err_word;
};

cudaError_t launch_kda_conv_bf16_d128(const ConvArgs &a);

}  // namespace kda
