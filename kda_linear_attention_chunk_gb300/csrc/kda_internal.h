// kda_internal.h -- launch interface between the C ABI (kda_api.cu) and the
// kernels.  Not installed; the public interface is include/kda.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

struct KdaArgs {
    const void *q, *k, *v;          // [T][H][dk|dv], bf16 or fp32
    const float *g, *beta;          // [T][H][dk], [T][H]
    const int32_t *cu_seqlens;      // [N+1]
    const float *initial_state;     // [N][H][dv][dk] or nullptr
    void *out;                      // [T][H][dv], bf16 or fp32
    float *final_state;             // [N][H][dv][dk] or nullptr
    int N, T, H, dk, dv;
    cudaStream_t stream;
    int *err_word;                  // device address of the sticky error word
    unsigned int *sched;            // 2 words of device scratch for the dynamic unit deal (reset by the kernel), or nullptr
    int num_sms;                    // SM count of the current device
};

cudaError_t launch_kda_simt_f32_d64(const KdaArgs &a);
cudaError_t launch_kda_simt_bf16_d128(const KdaArgs &a);
cudaError_t launch_kda_tc_bf16_d128(const KdaArgs &a);

}  // namespace kda
