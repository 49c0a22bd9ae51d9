// kda_api.cu -- the C ABI declared in include/kda.h: argument validation,
// device checks and kernel dispatch.  Validation is synchronous and happens
// before any CUDA call, so a rejected call touches no device state.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "kda.h"
#include "kda_conv.h"
#include "kda_decode.h"
#include "kda_internal.h"

namespace {

__device__ int g_kda_error_word = 0;

// Scratch of the dynamic unit deal: per slot a claim counter and a count of
// finished CTAs; the last CTA of a launch returns its slot to zero.  Calls take
// slots round-robin, so launches in flight at the same time (on different
// streams) use different slots unless more than kSchedSlots are in flight.
constexpr int kSchedSlots = 256;
static __device__ __align__(256) unsigned int g_kda_sched[kSchedSlots][2];
std::atomic<unsigned> g_sched_next{0};

constexpr int kMaxDevices = 64;

// Per-device facts looked up on the first call with that device current.  The
// fields are written under g_dev_mutex and published by the release store of
// `checked`; a caller that sees `checked` != 0 through an acquire load also
// sees the fields (host threads may race on a device's first call).
struct DevInfo {
    std::atomic<int> checked{0};   // 0 unknown, 1 ok, -1 unsupported
    int num_sms = 0;
    int *err = nullptr;
    unsigned int *sched = nullptr;
    cudaMemPool_t pool = nullptr;  // the library's own stream-ordered pool (split mode's ring); null: none
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

Range range_of(const void *p, size_t bytes)
{
    uintptr_t lo = (uintptr_t)p;
    return {lo, lo + (p ? bytes : 0)};
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Fills in d for device dev (called once, under g_dev_mutex).  A failed
// query leaves d unknown, so that a later call asks again.
int init_device(DevInfo &d, int dev)
{
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    void *err = nullptr, *sched = nullptr;
    if (cudaGetSymbolAddress(&err, g_kda_error_word) != cudaSuccess ||
        cudaGetSymbolAddress(&sched, g_kda_sched) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    d.num_sms = sms;
    d.err = (int *)err;
    d.sched = (unsigned int *)sched;
    // a pool of the library's own, which keeps what it has reserved (a few MB
    // per call in split mode), so that calls after the first allocate nothing
    // from the driver; without it split mode is off
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
        uint64_t keep = ~uint64_t(0);
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) == cudaSuccess) {
            d.pool = pool;
        } else {
            cudaMemPoolDestroy(pool);
        }
    }
    cudaGetLastError();
    d.checked.store((major == 10 && minor == 3) ? 1 : -1, std::memory_order_release);
    return KDA_OK;
}

int device_info(DevInfo **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    DevInfo &d = g_dev[dev];
    if (d.checked.load(std::memory_order_acquire) == 0) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (d.checked.load(std::memory_order_relaxed) == 0) {
            const int st = init_device(d, dev);
            if (st != KDA_OK) return st;
        }
    }
    if (d.checked.load(std::memory_order_acquire) != 1) return KDA_ERR_DEVICE;
    *out = &d;
    return KDA_OK;
}

// Validation shared by the entry points.  elem = bytes per q/k/v/out element;
// the state tensors hold state_n entries of [H][dv][dk] (N unless the states
// are addressed through the slot table `slots`, an [N] int32 input).
int validate(const void *q, const void *k, const void *v, const float *g, const float *beta,
             const int32_t *cu, const float *s0, const void *out, const float *s1,
             int N, int T, int H, int dk, int dv, size_t elem,
             const int32_t *slots = nullptr, int state_n = -1)
{
    if (state_n < 0) state_n = N;
    if (!cu) return KDA_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (N < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return KDA_ERR_SHAPE;
    const size_t rows = (size_t)T * (size_t)H;
    if ((size_t)N * (size_t)H > 0x7fffffffu || rows * (size_t)(dk > dv ? dk : dv) * 4 >= ((size_t)1 << 40) ||
        (size_t)state_n * (size_t)H > 0x7fffffffu)
        return KDA_ERR_SHAPE;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return KDA_ERR_UNSUPPORTED;
    const void *aligned_ptrs[] = {q, k, v, g, out, s0, s1};
    for (const void *p : aligned_ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    if (((uintptr_t)beta & 3u) || ((uintptr_t)cu & 3u) || ((uintptr_t)slots & 3u)) return KDA_ERR_ALIGN;

    const size_t state_bytes = (size_t)state_n * H * dv * dk * sizeof(float);
    const Range in[] = {range_of(q, rows * dk * elem), range_of(k, rows * dk * elem),
                        range_of(v, rows * dv * elem), range_of(g, rows * dk * sizeof(float)),
                        range_of(beta, rows * sizeof(float)),
                        range_of(cu, (size_t)(N + 1) * sizeof(int32_t)),
                        range_of(slots, (size_t)N * sizeof(int32_t)),
                        range_of(s0, state_bytes)};
    constexpr int kStateIn = 7;   // in[kStateIn] is the initial state
    const Range ro = range_of(out, rows * dv * elem);
    const Range rs = range_of(s1, state_bytes);
    for (const Range &r : in)
        if (overlap(ro, r)) return KDA_ERR_ALIAS;
    if (overlap(ro, rs)) return KDA_ERR_ALIAS;
    for (int i = 0; i < kStateIn; i++)
        if (overlap(rs, in[i])) return KDA_ERR_ALIAS;
    if (s0 && s1 && overlap(rs, in[kStateIn]) && (s0 != s1)) return KDA_ERR_ALIAS;
    return KDA_OK;
}

kda::KdaArgs make_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const int32_t *cu, const float *s0, void *out, float *s1, int N, int T, int H,
                       int dk, int dv, void *stream, const DevInfo *d)
{
    kda::KdaArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu_seqlens = cu;
    a.initial_state = s0; a.out = out; a.final_state = s1;
    a.N = N; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    a.stream = (cudaStream_t)stream;
    a.err_word = d->err;
    a.sched = d->sched + 2 * (g_sched_next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
    a.num_sms = d->num_sms;
    return a;
}

}  // namespace

namespace kda {

int validate_bf16_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const int32_t *cu, const float *s0, const void *out, const float *s1, int N, int T, int H,
                       int dk, int dv)
{
    return validate(q, k, v, g, beta, cu, s0, out, s1, N, T, H, dk, dv, sizeof(uint16_t));
}

int error_word_address(int **out)
{
    DevInfo *d = nullptr;
    const int st = device_info(&d);
    if (st == KDA_OK) *out = d->err;
    return st;
}

}  // namespace kda

extern "C" {

const char *kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_NULL: return "KDA_ERR_NULL: a required pointer is NULL";
    case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE: bad sizes (N >= 1, T >= 0, H >= 1) or size overflow";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: dk/dv/dtype combination or N not supported";
    case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN: tensor pointer not 16-byte aligned";
    case KDA_ERR_ALIAS: return "KDA_ERR_ALIAS: an output overlaps another argument";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call failed (see cudaGetLastError)";
    case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE: no CUDA device, or the device is not sm_103";
    case KDA_ERR_NOALLOC_LIMIT:
        return "KDA_ERR_NOALLOC_LIMIT: N is above KDA_NOALLOC_MAX_SEQS, the size of the library-held scratch";
    default: return "unknown kda_status";
    }
}

// Split mode (kda.h, kda_chunk_prefill): 0 off, 1 one chain CTA per unit,
// 2 two (half chains).  On for calls of few units and T >= 1024, unless the
// environment variable KDA_SPLIT says otherwise: "0" never, "1" whenever the
// call allows it, "full" / "half" whenever it allows it and in that form
// (half only where possible).  Half chains by default where the producers
// keep up with them: units at most a fifth of the SMs (measured 18-21 %
// faster at 8-24 units on 152 SMs; at 32 units the 88 producers set the pace
// and the two forms come within a few per cent of each other, either way
// from run to run).
int want_split(const kda::KdaArgs &a, const DevInfo *d)
{
    // (the producers pack a chunk index into 23 bits: far beyond any T that fits the device)
    const int units = a.N * a.H;
    if (!d->pool || a.T == 0 || a.T >= (1 << 29) || !kda::tc_split_possible(units, a.N, d->num_sms)) return 0;
    const bool half_ok = kda::tc_split_half_possible(units, a.N, d->num_sms);
    const char *env = getenv("KDA_SPLIT");
    if (env && env[0] == '0') return 0;
    if (env && strcmp(env, "full") == 0) return 1;
    if (env && strcmp(env, "half") == 0) return half_ok ? 2 : 1;
    const bool half = half_ok && 5 * units <= d->num_sms;
    if (env && env[0] == '1') return half ? 2 : 1;
    return a.T >= 1024 ? (half ? 2 : 1) : 0;
}

// the tensor-core kernel, split when that pays: the ring comes from the
// library's pool on the call's stream and goes back to it after the launch
cudaError_t launch_tc(kda::KdaArgs &a, const DevInfo *d)
{
    const int mode = want_split(a, d);
    if (!mode) return kda::launch_kda_tc_bf16_d128(a);
    const int units = a.N * a.H;
    const size_t bytes = kda::tc_split_bytes(units), flag_bytes = kda::tc_split_flag_bytes(units);
    void *ring = nullptr;
    if (cudaMallocFromPoolAsync(&ring, bytes, d->pool, a.stream) != cudaSuccess) {
        cudaGetLastError();
        return kda::launch_kda_tc_bf16_d128(a);
    }
    cudaError_t e = cudaMemsetAsync((uint8_t *)ring + bytes - flag_bytes, 0, flag_bytes, a.stream);
    if (e == cudaSuccess) {
        a.split_ring = (uint8_t *)ring;
        a.split_half = mode == 2;
        e = kda::launch_kda_tc_bf16_d128(a);
        a.split_ring = nullptr;
        a.split_half = false;
        if (e == cudaErrorCooperativeLaunchTooLarge) {   // the device cannot hold every CTA at once now
            cudaGetLastError();
            e = kda::launch_kda_tc_bf16_d128(a);
        }
    }
    const cudaError_t ef = cudaFreeAsync(ring, a.stream);
    return e != cudaSuccess ? e : ef;
}

int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                      const float *beta, const int32_t *cu_seqlens, const float *initial_state,
                      uint16_t *out, float *final_state, int N, int T, int H, int dk, int dv,
                      void *stream)
{
    int st = validate(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H, dk, dv,
                      sizeof(uint16_t));
    if (st != KDA_OK) return st;
    DevInfo *d = nullptr;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::KdaArgs a = make_args(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H,
                               dk, dv, stream, d);
    const cudaError_t e = (dk == 128 && dv == 128) ? launch_tc(a, d) : kda::launch_kda_simt(a, false);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill_fullrange(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                                const float *beta, const int32_t *cu_seqlens, const float *initial_state,
                                uint16_t *out, float *final_state, int N, int T, int H, int dk, int dv,
                                void *stream)
{
    int st = validate(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H, dk, dv,
                      sizeof(uint16_t));
    if (st != KDA_OK) return st;
    DevInfo *d = nullptr;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::KdaArgs a = make_args(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H,
                               dk, dv, stream, d);
    return kda::launch_kda_simt(a, false) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill_f32(const float *q, const float *k, const float *v, const float *g,
                          const float *beta, const int32_t *cu_seqlens, const float *initial_state,
                          float *out, float *final_state, int N, int T, int H, int dk, int dv,
                          void *stream)
{
    int st = validate(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H, dk, dv,
                      sizeof(float));
    if (st != KDA_OK) return st;
    DevInfo *d = nullptr;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::KdaArgs a = make_args(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, N, T, H,
                               dk, dv, stream, d);
    return kda::launch_kda_simt(a, true) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill_slots(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                            const float *beta, const int32_t *cu_seqlens, const int32_t *state_slots,
                            float *state_pool, int num_slots, uint16_t *out, int N, int T, int H, int dk,
                            int dv, void *stream)
{
    if (!state_slots || !state_pool) return KDA_ERR_NULL;
    if (num_slots < 1) return KDA_ERR_SHAPE;
    int st = validate(q, k, v, g, beta, cu_seqlens, state_pool, out, state_pool, N, T, H, dk, dv,
                      sizeof(uint16_t), state_slots, num_slots);
    if (st != KDA_OK) return st;
    DevInfo *d = nullptr;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::KdaArgs a = make_args(q, k, v, g, beta, cu_seqlens, state_pool, out, state_pool, N, T, H,
                               dk, dv, stream, d);
    a.state_slots = state_slots;
    a.num_slots = num_slots;
    const cudaError_t e = (dk == 128 && dv == 128) ? launch_tc(a, d) : kda::launch_kda_simt(a, false);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv, const float *conv_weight,
                           const float *g, const float *beta, const int32_t *cu_seqlens, const int32_t *slots,
                           uint16_t *conv_pool, int conv_num_slots, float *state_pool, int num_slots, uint16_t *out,
                           int N, int T, int H, int dk, int dv, int activation, float eps, void *stream)
{
    if (!cu_seqlens || !conv_weight || !conv_pool || !state_pool) return KDA_ERR_NULL;
    if (N < 1 || T < 0 || H < 1 || num_slots < 1 || conv_num_slots < 1) return KDA_ERR_SHAPE;
    if (!slots && (num_slots < N || conv_num_slots < N)) return KDA_ERR_SHAPE;
    if (activation != 0 && activation != 1) return KDA_ERR_SHAPE;
    if (!(eps >= 0.f && eps <= 3.0e38f)) return KDA_ERR_SHAPE;   // also rejects NaN
    if ((size_t)conv_num_slots * (size_t)H * 128 * 9 * 2 >= ((size_t)1 << 40)) return KDA_ERR_SHAPE;
    // the prefill's own checks, the state pool as both initial and final state
    int st = validate(xq, xk, xv, g, beta, cu_seqlens, state_pool, out, state_pool, N, T, H, dk, dv,
                      sizeof(uint16_t), slots, num_slots);
    if (st != KDA_OK) return st;
    if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(conv_weight) || !aligned16(conv_pool)) return KDA_ERR_ALIGN;
    const size_t rows = (size_t)T * H;
    const Range rw = range_of(conv_weight, (size_t)3 * H * 128 * 4 * sizeof(float));
    const Range rp = range_of(conv_pool, (size_t)conv_num_slots * 9 * H * 128 * 2);
    const Range others[] = {range_of(xq, rows * 256), range_of(xk, rows * 256), range_of(xv, rows * 256),
                            range_of(g, rows * 128 * sizeof(float)), range_of(beta, rows * sizeof(float)),
                            range_of(cu_seqlens, (size_t)(N + 1) * sizeof(int32_t)),
                            range_of(slots, (size_t)N * sizeof(int32_t)),
                            range_of(state_pool, (size_t)num_slots * H * 128 * 128 * sizeof(float)),
                            range_of(out, rows * 256)};
    for (const Range &r : others)
        if (overlap(rp, r) || overlap(rw, r)) return KDA_ERR_ALIAS;
    if (overlap(rp, rw)) return KDA_ERR_ALIAS;
    DevInfo *d = nullptr;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::KdaArgs a = make_args(xq, xk, xv, g, beta, cu_seqlens, state_pool, out, state_pool, N, T, H, dk, dv,
                               stream, d);
    a.state_slots = slots;
    // with a slot table an id must name an entry of both pools
    a.num_slots = slots ? (num_slots < conv_num_slots ? num_slots : conv_num_slots) : num_slots;
    a.conv_w = conv_weight;
    a.conv_pool = conv_pool;
    a.conv_act = activation;
    a.conv_eps = eps;
    return kda::launch_kda_tc_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g, const float *beta,
               const int32_t *state_slots, float *state_pool, int num_slots, uint16_t *out, int N, int H, int dk,
               int dv, void *stream)
{
    if (!q || !k || !v || !g || !beta || !state_pool || !out) return KDA_ERR_NULL;
    if (N < 1 || H < 1 || dk < 1 || dv < 1 || num_slots < 1) return KDA_ERR_SHAPE;
    if (!state_slots && num_slots < N) return KDA_ERR_SHAPE;
    if ((size_t)N * (size_t)H > 0x1fffffffu || (size_t)num_slots * (size_t)H > 0x7fffffffu) return KDA_ERR_SHAPE;
    if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
    const void *aligned_ptrs[] = {q, k, v, g, out, state_pool};
    for (const void *p : aligned_ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    if (((uintptr_t)beta & 3u) || ((uintptr_t)state_slots & 3u)) return KDA_ERR_ALIGN;
    const size_t rows = (size_t)N * H;
    const Range in[] = {range_of(q, rows * dk * 2), range_of(k, rows * dk * 2), range_of(v, rows * dv * 2),
                        range_of(g, rows * dk * sizeof(float)), range_of(beta, rows * sizeof(float)),
                        range_of(state_slots, (size_t)N * sizeof(int32_t))};
    const Range rp = range_of(state_pool, (size_t)num_slots * H * dv * dk * sizeof(float));
    const Range ro = range_of(out, rows * dv * 2);
    for (const Range &r : in)
        if (overlap(rp, r) || overlap(ro, r)) return KDA_ERR_ALIAS;
    if (overlap(ro, rp)) return KDA_ERR_ALIAS;
    DevInfo *d = nullptr;
    int st;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
    a.state_slots = state_slots; a.state_pool = state_pool; a.out = out;
    a.N = N; a.H = H; a.num_slots = num_slots;
    a.stream = (cudaStream_t)stream;
    a.err_word = d->err;
    return kda::launch_kda_decode_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv, const float *conv_weight,
                    const int32_t *conv_slots, uint16_t *conv_pool, int conv_num_slots, const float *g,
                    const float *beta, const int32_t *state_slots, float *state_pool, int num_slots, uint16_t *out,
                    int N, int H, int dk, int dv, int activation, float eps, void *stream)
{
    if (!xq || !xk || !xv || !conv_weight || !conv_pool || !g || !beta || !state_pool || !out) return KDA_ERR_NULL;
    if (N < 1 || H < 1 || dk < 1 || dv < 1 || num_slots < 1 || conv_num_slots < 1) return KDA_ERR_SHAPE;
    if ((!state_slots && num_slots < N) || (!conv_slots && conv_num_slots < N)) return KDA_ERR_SHAPE;
    if (activation != 0 && activation != 1) return KDA_ERR_SHAPE;
    if (!(eps >= 0.f && eps <= 3.0e38f)) return KDA_ERR_SHAPE;   // also rejects NaN
    if ((size_t)N * (size_t)H > 0x1fffffffu || (size_t)num_slots * (size_t)H > 0x7fffffffu ||
        (size_t)conv_num_slots * (size_t)H * 128 * 9 * 2 >= ((size_t)1 << 40))
        return KDA_ERR_SHAPE;
    if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
    const void *aligned_ptrs[] = {xq, xk, xv, conv_weight, conv_pool, g, out, state_pool};
    for (const void *p : aligned_ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    if (((uintptr_t)beta & 3u) || ((uintptr_t)state_slots & 3u) || ((uintptr_t)conv_slots & 3u))
        return KDA_ERR_ALIGN;
    const size_t rows = (size_t)N * H;
    const Range in[] = {range_of(xq, rows * 256), range_of(xk, rows * 256), range_of(xv, rows * 256),
                        range_of(conv_weight, (size_t)3 * H * 128 * 4 * sizeof(float)),
                        range_of(conv_slots, (size_t)N * sizeof(int32_t)),
                        range_of(g, rows * 128 * sizeof(float)), range_of(beta, rows * sizeof(float)),
                        range_of(state_slots, (size_t)N * sizeof(int32_t))};
    const Range rw[] = {range_of(conv_pool, (size_t)conv_num_slots * 9 * H * 128 * 2),
                        range_of(state_pool, (size_t)num_slots * H * 128 * 128 * sizeof(float)),
                        range_of(out, rows * 256)};
    for (int i = 0; i < 3; i++) {
        for (const Range &r : in)
            if (overlap(rw[i], r)) return KDA_ERR_ALIAS;
        for (int j = i + 1; j < 3; j++)
            if (overlap(rw[i], rw[j])) return KDA_ERR_ALIAS;
    }
    DevInfo *d = nullptr;
    int st;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::DecodeConvArgs a;
    a.xq = xq; a.xk = xk; a.xv = xv; a.conv_weight = conv_weight;
    a.conv_slots = conv_slots; a.conv_pool = conv_pool; a.conv_num_slots = conv_num_slots;
    a.g = g; a.beta = beta; a.state_slots = state_slots; a.state_pool = state_pool; a.num_slots = num_slots;
    a.out = out; a.N = N; a.H = H; a.activation = activation; a.eps = eps;
    a.stream = (cudaStream_t)stream;
    a.err_word = d->err;
    return kda::launch_kda_decode_conv_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_fold_commit(const uint16_t *k, const uint16_t *v, const float *g, const float *beta, const int32_t *accepted,
                    const int32_t *state_slots, float *state_pool, int num_slots, int N, int W, int H, int dk, int dv,
                    void *stream)
{
    if (!k || !v || !g || !beta || !accepted || !state_pool) return KDA_ERR_NULL;
    if (N < 1 || W < 1 || H < 1 || dk < 1 || dv < 1 || num_slots < 1) return KDA_ERR_SHAPE;
    if (!state_slots && num_slots < N) return KDA_ERR_SHAPE;
    const size_t rows = (size_t)N * W * H;
    if ((size_t)N * (size_t)H > 0x1fffffffu || (size_t)num_slots * (size_t)H > 0x7fffffffu ||
        rows * 128 * 4 >= ((size_t)1 << 40))
        return KDA_ERR_SHAPE;
    if (dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
    const void *aligned_ptrs[] = {k, v, g, state_pool};
    for (const void *p : aligned_ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    if (((uintptr_t)beta & 3u) || ((uintptr_t)accepted & 3u) || ((uintptr_t)state_slots & 3u)) return KDA_ERR_ALIGN;
    const Range in[] = {range_of(k, rows * dk * 2), range_of(v, rows * dv * 2),
                        range_of(g, rows * dk * sizeof(float)), range_of(beta, rows * sizeof(float)),
                        range_of(accepted, (size_t)N * sizeof(int32_t)),
                        range_of(state_slots, (size_t)N * sizeof(int32_t))};
    const Range rp = range_of(state_pool, (size_t)num_slots * H * dv * dk * sizeof(float));
    for (const Range &r : in)
        if (overlap(rp, r)) return KDA_ERR_ALIAS;
    DevInfo *d = nullptr;
    int st;
    if ((st = device_info(&d)) != KDA_OK) return st;
    kda::FoldArgs a;
    a.k = k; a.v = v; a.g = g; a.beta = beta; a.accepted = accepted;
    a.state_slots = state_slots; a.state_pool = state_pool;
    a.N = N; a.W = W; a.H = H; a.num_slots = num_slots;
    a.num_sms = d->num_sms;
    a.stream = (cudaStream_t)stream;
    a.err_word = d->err;
    return kda::launch_kda_fold_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_short_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv, const float *conv_weight,
                   const int32_t *cu_seqlens, const int32_t *conv_slots, uint16_t *conv_pool, int num_slots,
                   uint16_t *q_out, uint16_t *k_out, uint16_t *v_out, int N, int T, int H, int d,
                   int activation, float eps, void *stream)
{
    if (!cu_seqlens || !conv_weight || !conv_pool) return KDA_ERR_NULL;
    if (T > 0 && (!xq || !xk || !xv || !q_out || !k_out || !v_out)) return KDA_ERR_NULL;
    if (N < 1 || T < 0 || H < 1 || d < 1 || num_slots < 1) return KDA_ERR_SHAPE;
    if (!conv_slots && num_slots < N) return KDA_ERR_SHAPE;
    if (activation != 0 && activation != 1) return KDA_ERR_SHAPE;
    if (!(eps >= 0.f && eps <= 3.0e38f)) return KDA_ERR_SHAPE;   // also rejects NaN
    const size_t rows = (size_t)T * (size_t)H;
    if (rows * 128 * 2 >= ((size_t)1 << 40) || (size_t)N * (size_t)H > ((size_t)1 << 26) ||
        (size_t)num_slots * (size_t)H * 128 * 9 * 2 >= ((size_t)1 << 40))
        return KDA_ERR_SHAPE;
    if (d != 128) return KDA_ERR_UNSUPPORTED;
    const void *aligned_ptrs[] = {xq, xk, xv, q_out, k_out, v_out, conv_pool, conv_weight};
    for (const void *p : aligned_ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    if (((uintptr_t)cu_seqlens & 3u) || ((uintptr_t)conv_slots & 3u)) return KDA_ERR_ALIGN;
    const size_t xbytes = rows * 128 * 2;
    const Range in[] = {range_of(xq, xbytes), range_of(xk, xbytes), range_of(xv, xbytes),
                        range_of(conv_weight, (size_t)3 * H * 128 * 4 * sizeof(float)),
                        range_of(cu_seqlens, (size_t)(N + 1) * sizeof(int32_t)),
                        range_of(conv_slots, (size_t)N * sizeof(int32_t))};
    const Range rp = range_of(conv_pool, (size_t)num_slots * 9 * H * 128 * 2);
    const Range ro[] = {range_of(q_out, xbytes), range_of(k_out, xbytes), range_of(v_out, xbytes)};
    for (const Range &r : in) {
        if (overlap(rp, r)) return KDA_ERR_ALIAS;
        for (const Range &o : ro)
            if (overlap(o, r)) return KDA_ERR_ALIAS;
    }
    for (int i = 0; i < 3; i++) {
        if (overlap(ro[i], rp)) return KDA_ERR_ALIAS;
        for (int j = i + 1; j < 3; j++)
            if (overlap(ro[i], ro[j])) return KDA_ERR_ALIAS;
    }
    DevInfo *dv = nullptr;
    int st;
    if ((st = device_info(&dv)) != KDA_OK) return st;
    kda::ConvArgs a;
    a.x[0] = xq; a.x[1] = xk; a.x[2] = xv;
    a.y[0] = q_out; a.y[1] = k_out; a.y[2] = v_out;
    a.weight = conv_weight;
    a.cu_seqlens = cu_seqlens;
    a.conv_slots = conv_slots;
    a.conv_pool = conv_pool;
    a.N = N; a.T = T; a.H = H; a.num_slots = num_slots;
    a.activation = activation;
    a.eps = eps;
    a.stream = (cudaStream_t)stream;
    a.err_word = dv->err;
    return kda::launch_kda_conv_bf16_d128(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_device_error(int *word, int reset)
{
    if (!word) return KDA_ERR_NULL;
    if (cudaMemcpyFromSymbol(word, g_kda_error_word, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_kda_error_word, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"
