// kda_decode.h -- launch interface of the decode kernel (kda_decode.cu) for the
// C ABI (kda_api.cu).  Not installed; the public interface is include/kda.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// one recurrence step per sequence (decode), bf16, d = 128
struct DecodeArgs {
    const void *q, *k, *v;          // [N][H][128] bf16
    const float *g, *beta;          // [N][H][128], [N][H]
    const int32_t *state_slots;     // [N] or nullptr (entry n)
    float *state_pool;              // [num_slots][H][128][128]
    void *out;                      // [N][H][128] bf16
    int N, H, num_slots;
    cudaStream_t stream;
    int *err_word;
};

cudaError_t launch_kda_decode_bf16_d128(const DecodeArgs &a);

// the decode step with the short conv fused in front of it, bf16, d = 128
struct DecodeConvArgs {
    const void *xq, *xk, *xv;       // [N][H][128] bf16 projections
    const float *conv_weight;       // [3][H*128][4]
    const int32_t *conv_slots;      // [N] or nullptr (entry n)
    void *conv_pool;                // [conv_num_slots][3][3][H*128] bf16
    const float *g, *beta;          // [N][H][128], [N][H]
    const int32_t *state_slots;     // [N] or nullptr (entry n)
    float *state_pool;              // [num_slots][H][128][128]
    void *out;                      // [N][H][128] bf16
    int N, H, num_slots, conv_num_slots, activation;
    float eps;
    cudaStream_t stream;
    int *err_word;
};

cudaError_t launch_kda_decode_conv_bf16_d128(const DecodeConvArgs &a);

// commit of a speculative round: the first accepted[n] tokens of each window
struct FoldArgs {
    const void *k, *v;              // [N][W][H][128] bf16
    const float *g, *beta;          // [N][W][H][128], [N][W][H]
    const int32_t *accepted;        // [N]
    const int32_t *state_slots;     // [N] or nullptr (entry n)
    float *state_pool;              // [num_slots][H][128][128]
    int N, W, H, num_slots;
    int num_sms;                    // persistent grid: 4 CTAs per SM
    cudaStream_t stream;
    int *err_word;
};

cudaError_t launch_kda_fold_bf16_d128(const FoldArgs &a);

}  // namespace kda
