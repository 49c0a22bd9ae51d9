// kda_noalloc.cu -- kda_chunk_prefill_noalloc: the tensor-core prefill for
// packed batches of up to KDA_NOALLOC_MAX_SEQS sequences, with every byte of
// working memory it needs held by the library itself.
//
// Who needs it: callers that cannot allocate device memory per call -- code
// running inside a serving runtime whose device memory is planned in full when
// a model is loaded (every buffer comes from a fixed pool or manifest, and the
// runtime's own allocator is closed to kernels' helpers), or library code that
// is handed only the tensors of one layer.  With many short sequences the
// prefill must sort the sequences by length and deal their (sequence, head)
// units to the SMs from a shared counter; that bookkeeping needs a small table
// in device memory.  Here it lives in a file-scope static device array
// (g_kda_noalloc_scratch, about 196 KB), which every GPU that loads the library
// holds until the process exits, so the call itself allocates nothing: no
// cudaMalloc, no cudaFree, no allocator of any library.
//
// The caller passes inputs and outputs exactly as to kda_chunk_prefill.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace {

constexpr int kMaxSeqs = KDA_NOALLOC_MAX_SEQS;
constexpr int kMaxDevices = 64;
constexpr int kThreads = 256;

// Layout (32-bit words): [0] claim counter and [1] finished-CTA count of the
// unit deal, [2] nonempty sequences x H, [3] unused, then the clamped row
// ranges {bos, eos} of every sequence, then the length-sorted sequence order.
constexpr int kWordsHead = 4;
constexpr int kWords = kWordsHead + 2 * kMaxSeqs + kMaxSeqs;
static __device__ __align__(256) int g_kda_noalloc_scratch[kWords];

// Written under g_na_mutex and published by the release store of `ready`, so
// that host threads racing on a device's first call see complete fields.
struct NoAllocDev {
    std::atomic<int> ready{0};   // 1 once the scratch address, SM count and error word are known
    int num_sms = 0;
    int *scratch = nullptr;      // device address of g_kda_noalloc_scratch
    int *err = nullptr;          // device address of the library's error word
};
NoAllocDev g_na[kMaxDevices];
std::mutex g_na_mutex;

// rows and lengths: one thread per sequence
__global__ void noalloc_rows(const int32_t *cu, int N, int T, int H, int *err, int *scratch)
{
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const int b = kda::clamp_row(cu[n], T, err);
    int e = kda::clamp_row(cu[n + 1], T, err);
    if (e < b) e = b;
    reinterpret_cast<int2 *>(scratch + kWordsHead)[n] = make_int2(b, e);
    if (e > b) atomicAdd(scratch + 2, H);
}

// length-sorted order (longest first, ties by index): each thread ranks one
// sequence against all others, reading the lengths through shared memory tiles
__global__ void noalloc_order(int N, int *scratch)
{
    __shared__ int len[kThreads];
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int2 *rows = reinterpret_cast<const int2 *>(scratch + kWordsHead);
    const int my = n < N ? rows[n].y - rows[n].x : 0;
    int rank = 0;
    for (int base = 0; base < N; base += kThreads) {
        const int m = base + threadIdx.x;
        len[threadIdx.x] = m < N ? rows[m].y - rows[m].x : -1;
        __syncthreads();
        const int cnt = min(kThreads, N - base);
        for (int i = 0; i < cnt; i++) {
            const int lm = len[i];
            rank += (lm > my) || (lm == my && base + i < n);
        }
        __syncthreads();
    }
    if (n < N) (scratch + kWordsHead + 2 * kMaxSeqs)[rank] = n;
}

// once per device, with that device current: the scratch array's device
// address (its name in host code is only a host-side stand-in), the SM count
// and the error word's address
int noalloc_setup(NoAllocDev **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    NoAllocDev &d = g_na[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_na_mutex);
        if (d.ready.load(std::memory_order_relaxed)) {
            *out = &d;
            return KDA_OK;
        }
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_DEVICE;
        }
        if (major != 10 || minor != 3) return KDA_ERR_DEVICE;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_kda_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        int *err = nullptr;
        const int st = kda::error_word_address(&err);
        if (st != KDA_OK) return st;
        d.scratch = static_cast<int *>(ptr);
        d.err = err;
        d.num_sms = sms;
        d.ready.store(1, std::memory_order_release);
    }
    *out = &d;
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_prefill_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                                         const float *beta, const int32_t *cu_seqlens, const float *initial_state,
                                         uint16_t *out, float *final_state, int N, int T, int H, int dk, int dv,
                                         void *stream)
{
    // the checks of kda_chunk_prefill first, so that a bad pointer or size gets
    // the same status as there; then the size of the library-held table
    int st = kda::validate_bf16_args(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H, dk,
                                     dv);
    if (st != KDA_OK) return st;
    if (N > kMaxSeqs) return KDA_ERR_NOALLOC_LIMIT;
    NoAllocDev *d = nullptr;
    if ((st = noalloc_setup(&d)) != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::KdaArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu_seqlens = cu_seqlens;
    a.initial_state = initial_state; a.out = out; a.final_state = final_state;
    a.N = N; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    a.stream = s;
    a.err_word = d->err;
    a.num_sms = d->num_sms;
    // other head sizes run on the CUDA-core kernel, one CTA per (sequence,
    // head): it needs no table
    if (dk != 128 || dv != 128) return kda::launch_kda_simt(a, false) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    // the deal counters and the nonempty count must start at zero on every call
    if (cudaMemsetAsync(d->scratch, 0, kWordsHead * sizeof(int), s) != cudaSuccess) return KDA_ERR_CUDA;
    const int blocks = (N + kThreads - 1) / kThreads;
    noalloc_rows<<<blocks, kThreads, 0, s>>>(cu_seqlens, N, T, H, d->err, d->scratch);
    noalloc_order<<<blocks, kThreads, 0, s>>>(N, d->scratch);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    a.sched = reinterpret_cast<unsigned int *>(d->scratch);
    a.g_order = d->scratch + kWordsHead + 2 * kMaxSeqs;
    a.g_rows = reinterpret_cast<const int2 *>(d->scratch + kWordsHead);
    a.g_units_nonempty = d->scratch + 2;
    return kda::launch_kda_tc_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
