// kda_decode.cu -- one KDA recurrence step per sequence (decode), states in a
// slot-addressed pool, updated in place.
//
// For sequence n and head h, with S = pool[slot[n]][h] (stored as S^T, [v][k]):
//     S <- (I - beta k k^T) Diag(exp(g)) S + beta k v^T,   o = S^T q
// i.e. S'[v][c] = S[v][c] exp(g_c),  e_v = sum_c S'[v][c] k_c,
//      S[v][c]  = S'[v][c] + beta k_c (v_v - e_v),  o_v = sum_c S[v][c] q_c.
// (The Kimi-K3 decode runs this step over a rank's heads on states held in the
// engine's [slot][head][v][k] f32 pool, skipping padded rows, slot -1:
// kern-k3-pp-prefill README, "D inside SGLang".)
//
// The step moves 128 KB of state per (sequence, head) against 1.5 KB of
// inputs, so it is bound by HBM bandwidth: four CTAs (32 value rows each) stream
// one state through registers once.  Thread (v, e) owns value row v and the
// 16-byte pieces 8j + e (j = 0..3) of it, so the eight threads of a row read
// 128 contiguous bytes per load and a warp reads four full lines.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_decode.h"

namespace kda {
namespace {

constexpr int kDecThreads = 256;   // 32 value rows x 8 threads
constexpr int kDecRows = 32;       // value rows per CTA
constexpr float kDecLog2e = 1.4426950408889634f;

__device__ __forceinline__ float dec_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

struct DecodeParams {
    const uint16_t *q, *k, *v;   // [N][H][128] bf16
    const float *g, *beta;       // [N][H][128], [N][H]
    const int32_t *slots;        // [N] or nullptr (entry n)
    float *pool;                 // [num_slots][H][128][128]
    uint16_t *out;               // [N][H][128] bf16
    int N, H, num_slots;
    int *err;
};

// One token's update of this thread's 16 state entries (row vr, pieces 8j + e),
// with exp(g), k and q of the token staged in shared memory:
//   S' = S exp(g),  e = S' . k (over the row's eight threads),
//   S = S' + k beta (v - e),  returns S . q (over the row's eight threads).
// The decode step and the fold both run exactly this sequence of operations,
// so folding a tokens equals a decode steps bit for bit.
__device__ __forceinline__ float token_step(float4 (&s)[4], const float4 *sa, const float4 *sk, const float4 *sq,
                                            int qe, float vv, float beta)
{
    float ep[4];                      // four partial sums: short dependent chains
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float4 a = sa[8 * j + qe], kk = sk[8 * j + qe];
        s[j].x *= a.x; s[j].y *= a.y; s[j].z *= a.z; s[j].w *= a.w;
        ep[j] = s[j].x * kk.x; ep[j] = fmaf(s[j].y, kk.y, ep[j]);
        ep[j] = fmaf(s[j].z, kk.z, ep[j]); ep[j] = fmaf(s[j].w, kk.w, ep[j]);
    }
    float e = (ep[0] + ep[1]) + (ep[2] + ep[3]);
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    e += __shfl_xor_sync(0xffffffffu, e, 2);
    e += __shfl_xor_sync(0xffffffffu, e, 4);
    const float u = beta * (vv - e);
    float op[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float4 kk = sk[8 * j + qe];
        s[j].x = fmaf(kk.x, u, s[j].x); s[j].y = fmaf(kk.y, u, s[j].y);
        s[j].z = fmaf(kk.z, u, s[j].z); s[j].w = fmaf(kk.w, u, s[j].w);
        if (sq) {
            const float4 qq = sq[8 * j + qe];
            op[j] = s[j].x * qq.x; op[j] = fmaf(s[j].y, qq.y, op[j]);
            op[j] = fmaf(s[j].z, qq.z, op[j]); op[j] = fmaf(s[j].w, qq.w, op[j]);
        }
    }
    float o = 0.f;
    if (sq) {
        o = (op[0] + op[1]) + (op[2] + op[3]);
        o += __shfl_xor_sync(0xffffffffu, o, 1);
        o += __shfl_xor_sync(0xffffffffu, o, 2);
        o += __shfl_xor_sync(0xffffffffu, o, 4);
    }
    return o;
}

// The pool entry of sequence n, -1 to skip it (padding, or an id outside the
// pool, which is reported).
__device__ __forceinline__ int decode_slot(const int32_t *slots, int n, int num_slots, int *err)
{
    if (!slots) return n;
    const int slot = slots[n];
    if (slot < -1 || slot >= num_slots) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadSlot);
        return -1;
    }
    return slot;
}

__global__ void __launch_bounds__(kDecThreads, 5) kda_decode_kernel(DecodeParams p)
{
    __shared__ float4 sa[32], sk[32], sq[32];   // exp(g), k, q of this (sequence, head), 128 each
    const int rh = blockIdx.x >> 2, vq = blockIdx.x & 3;   // (sequence, head), quarter of the value rows
    const int n = rh / p.H, h = rh % p.H;
    const int slot = decode_slot(p.slots, n, p.num_slots, p.err);
    if (slot < 0) return;   // padded row: nothing is computed or written
    const size_t row = (size_t)n * p.H + h;
    const int tid = threadIdx.x;
    if (tid < 128) {
        reinterpret_cast<float *>(sa)[tid] = dec_ex2(p.g[row * 128 + tid] * kDecLog2e);
        reinterpret_cast<float *>(sk)[tid] = bf16_bits_to_float(p.k[row * 128 + tid]);
        reinterpret_cast<float *>(sq)[tid] = bf16_bits_to_float(p.q[row * 128 + tid]);
    }
    const int vr = kDecRows * vq + (tid >> 3), qe = tid & 7;
    const float vv = bf16_bits_to_float(p.v[row * 128 + vr]);
    const float beta = p.beta[row];
    float4 *st = reinterpret_cast<float4 *>(p.pool + (((size_t)slot * p.H + h) * 128 + vr) * 128);
    float4 s[4];
#pragma unroll
    for (int j = 0; j < 4; j++) s[j] = st[8 * j + qe];
    __syncthreads();
    const float o = token_step(s, sa, sk, sq, qe, vv, beta);
#pragma unroll
    for (int j = 0; j < 4; j++) st[8 * j + qe] = s[j];
    if (qe == 0) {
        const __nv_bfloat16 ob = __float2bfloat16_rn(o);
        p.out[row * 128 + vr] = *reinterpret_cast<const uint16_t *>(&ob);
    }
}

struct FoldParams {
    const uint16_t *k, *v;       // [N][W][H][128] bf16: each sequence's window of W tokens
    const float *g, *beta;       // [N][W][H][128], [N][W][H]
    const int32_t *accepted;     // [N]: fold the first accepted[n] tokens of the window
    const int32_t *slots;        // [N] or nullptr (entry n)
    float *pool;                 // [num_slots][H][128][128]
    int N, W, H, num_slots;
    int *err;
};

// Commit of a speculative round: the state takes the first accepted[n] tokens
// of sequence n's window, one token_step each.  The state stays in registers;
// the tokens' exp(g), k, v and beta are staged in shared memory up to
// kFoldBatch tokens at a time, all loads of a batch in flight together, so the
// steps themselves wait on no memory.
constexpr int kFoldBatch = 16;

__global__ void __launch_bounds__(kDecThreads, 5) kda_fold_kernel(FoldParams p)
{
    __shared__ float4 sa[kFoldBatch][32], sk[kFoldBatch][32];
    __shared__ float sv[kFoldBatch][128], sb[kFoldBatch];
    const int rh = blockIdx.x >> 2, vq = blockIdx.x & 3;
    const int n = rh / p.H, h = rh % p.H;
    const int slot = decode_slot(p.slots, n, p.num_slots, p.err);
    if (slot < 0) return;
    int acc = p.accepted[n];
    if (acc < 0 || acc > p.W) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrBadAccepted);
        acc = acc < 0 ? 0 : p.W;
    }
    if (acc == 0) return;   // nothing accepted: the state stays as it is
    const int tid = threadIdx.x;
    const int vr = kDecRows * vq + (tid >> 3), qe = tid & 7;
    float4 *st = reinterpret_cast<float4 *>(p.pool + (((size_t)slot * p.H + h) * 128 + vr) * 128);
    float4 s[4];
#pragma unroll
    for (int j = 0; j < 4; j++) s[j] = st[8 * j + qe];
    for (int t0 = 0; t0 < acc; t0 += kFoldBatch) {
        const int nt = min(kFoldBatch, acc - t0);
        if (t0 > 0) __syncthreads();           // the previous batch is no longer read
        for (int i = tid; i < nt * 128; i += kDecThreads) {
            const int t = i >> 7, c = i & 127;
            const size_t row = ((size_t)n * p.W + t0 + t) * p.H + h;
            reinterpret_cast<float *>(sa[t])[c] = dec_ex2(p.g[row * 128 + c] * kDecLog2e);
            reinterpret_cast<float *>(sk[t])[c] = bf16_bits_to_float(p.k[row * 128 + c]);
            sv[t][c] = bf16_bits_to_float(p.v[row * 128 + c]);
            if (c == 0) sb[t] = p.beta[row];
        }
        __syncthreads();
        for (int t = 0; t < nt; t++) token_step(s, sa[t], sk[t], nullptr, qe, sv[t][vr], sb[t]);
    }
#pragma unroll
    for (int j = 0; j < 4; j++) st[8 * j + qe] = s[j];
}

}  // namespace

cudaError_t launch_kda_decode_bf16_d128(const DecodeArgs &a)
{
    if (a.N == 0) return cudaSuccess;
    DecodeParams p;
    p.q = (const uint16_t *)a.q; p.k = (const uint16_t *)a.k; p.v = (const uint16_t *)a.v;
    p.g = a.g; p.beta = a.beta; p.slots = a.state_slots; p.pool = a.state_pool;
    p.out = (uint16_t *)a.out;
    p.N = a.N; p.H = a.H; p.num_slots = a.num_slots;
    p.err = a.err_word;
    kda_decode_kernel<<<(128 / kDecRows) * a.N * a.H, kDecThreads, 0, a.stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_kda_fold_bf16_d128(const FoldArgs &a)
{
    FoldParams p;
    p.k = (const uint16_t *)a.k; p.v = (const uint16_t *)a.v;
    p.g = a.g; p.beta = a.beta; p.accepted = a.accepted; p.slots = a.state_slots; p.pool = a.state_pool;
    p.N = a.N; p.W = a.W; p.H = a.H; p.num_slots = a.num_slots;
    p.err = a.err_word;
    kda_fold_kernel<<<(128 / kDecRows) * a.N * a.H, kDecThreads, 0, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
