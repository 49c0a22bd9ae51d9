// kda_common.cuh -- small device helpers shared by the KDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kda {

constexpr int kChunk = 64;  // rows per chunk (the 64-token chunk of the method)

// Sticky device error word (bit flags), read by kda_device_error().
enum : int {
    kErrWaitTimeout = 1,   // a bounded mbarrier wait ran out
    kErrBadSeqlens = 2,    // cu_seqlens violated its contract (indices clamped)
    kErrLayout = 4,        // shared-memory carve-up did not fit (never expected)
    kErrBadSlot = 8,       // a state slot id outside [-1, num_slots) (that sequence skipped)
    kErrBadAccepted = 16,  // an accepted count of the fold outside [0, W] (clamped)
    kErrDecayRange = 32,   // a chunk's decay factors left the fp16 operand range (tensor-core kernel)
};

__device__ __forceinline__ float load_in(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Clamp a cu_seqlens entry into [0, T]; flags a contract violation.
__device__ __forceinline__ int clamp_row(int x, int T, int *err)
{
    if (x < 0 || x > T) {
        if (err) atomicOr(err, kErrBadSeqlens);
        return x < 0 ? 0 : T;
    }
    return x;
}

}  // namespace kda
