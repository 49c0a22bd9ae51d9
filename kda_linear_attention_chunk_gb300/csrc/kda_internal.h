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
    // optional: a length-sorted unit order prepared in device memory (any N);
    // when set, the tensor-core kernel reads its sequence table from here
    const int *g_order = nullptr;   // [N] sequence indices, longest first
    const int2 *g_rows = nullptr;   // [N] clamped {bos, eos}
    const int *g_units_nonempty = nullptr;   // nonempty sequences x H
    // optional: states addressed through a slot table (tensor-core kernel);
    // initial_state == final_state is then the pool [num_slots][H][dv][dk]
    const int32_t *state_slots = nullptr;    // [N], -1 = padded sequence
    int num_slots = 0;
    // optional: the short-conv prologue fused into the tensor-core kernel; q, k,
    // v above are then the raw projections x_q, x_k, x_v
    const float *conv_w = nullptr;           // [3][H*128][4]
    uint16_t *conv_pool = nullptr;           // [entries][3][3][H*128] bf16 windows, updated in place
    int conv_act = 0;                        // 0 identity, 1 SiLU
    float conv_eps = 0.f;
    // optional: split mode (tensor-core kernel, no conv): the chunk ring and its
    // flags, tc_split_bytes(N * H) bytes of device memory, the flags (the
    // tail tc_split_flag_bytes(N * H) bytes) zeroed on the stream before the launch
    uint8_t *split_ring = nullptr;
    bool split_half = false;   // split mode with two chain CTAs per unit (tc_split_half_possible)
};

// CUDA-core kernel, any dk, dv in {64, 128}, bf16 (f32 = false) or fp32
// q/k/v/out, no limit on the decay range (kda_simt.cu)
cudaError_t launch_kda_simt(const KdaArgs &a, bool f32);
// tensor-core kernel, bf16, dk = dv = 128 (kda_tc.cu)
cudaError_t launch_kda_tc_bf16_d128(const KdaArgs &a);
int tc_max_sorted_seqs();   // largest N the tensor-core kernel sorts by itself
// split mode: whether a call of `units` (sequence, head) pairs and N sequences
// can run split on a device of num_sms SMs, and the device memory it needs
bool tc_split_possible(int units, int N, int num_sms);
bool tc_split_half_possible(int units, int N, int num_sms);
size_t tc_split_bytes(int units);
size_t tc_split_flag_bytes(int units);

// kda_api.cu: the checks of kda_chunk_prefill, and the current device's
// error-word address and SM count (also checks the device)
int validate_bf16_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const int32_t *cu, const float *s0, const void *out, const float *s1, int N, int T, int H,
                       int dk, int dv);
int error_word_address(int **out);

}  // namespace kda
