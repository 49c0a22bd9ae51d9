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

}  // namespace kda
