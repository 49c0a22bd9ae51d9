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

// Two fp32 operations in one instruction on a register pair (mul / fma
// .rn.f32x2, sm_100 and later): each half is the IEEE single-precision
// operation rounded to nearest even.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mul.rn.f32x2 x, x, y;\n mov.b64 {%0, %1}, x;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mov.b64 z, {%6, %7};\n"
        " fma.rn.f32x2 x, x, y, z;\n mov.b64 {%0, %1}, x;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 lo2(const float4 &v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4 &v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 cat2(float2 lo, float2 hi) { return make_float4(lo.x, lo.y, hi.x, hi.y); }

// dot of this thread's 16 entries with the staged vector x: two pair
// accumulators (pieces j = 0, 1 and j = 2, 3), each a chain of four fused
// pair operations, then their four lanes summed
__device__ __forceinline__ float dot16(const float4 (&s)[4], const float4 *x, int qe)
{
    float2 acc[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const float4 x0 = x[8 * (2 * h) + qe], x1 = x[8 * (2 * h + 1) + qe];
        acc[h] = fmul2(lo2(s[2 * h]), lo2(x0));
        acc[h] = ffma2(hi2(s[2 * h]), hi2(x0), acc[h]);
        acc[h] = ffma2(lo2(s[2 * h + 1]), lo2(x1), acc[h]);
        acc[h] = ffma2(hi2(s[2 * h + 1]), hi2(x1), acc[h]);
    }
    return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

// One token's update of this thread's 16 state entries (row vr, pieces 8j + e),
// with exp(g), k and q of the token staged in shared memory:
//   S' = S exp(g),  e = S' . k (over the row's eight threads),
//   S = S' + k beta (v - e),  returns S . q (over the row's eight threads).
// The decode step and the fold both run exactly this sequence of operations,
// so folding a tokens equals a decode steps bit for bit.  The entries go
// through the fp32 pipes two at a time (pairs of a float4).
__device__ __forceinline__ float token_step(float4 (&s)[4], const float4 *sa, const float4 *sk, const float4 *sq,
                                            int qe, float vv, float beta)
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float4 a = sa[8 * j + qe];
        s[j] = cat2(fmul2(lo2(s[j]), lo2(a)), fmul2(hi2(s[j]), hi2(a)));
    }
    float e = dot16(s, sk, qe);
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    e += __shfl_xor_sync(0xffffffffu, e, 2);
    e += __shfl_xor_sync(0xffffffffu, e, 4);
    const float u = beta * (vv - e);
    const float2 u2 = make_float2(u, u);
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float4 kk = sk[8 * j + qe];
        s[j] = cat2(ffma2(lo2(kk), u2, lo2(s[j])), ffma2(hi2(kk), u2, hi2(s[j])));
    }
    float o = 0.f;
    if (sq) {
        o = dot16(s, sq, qe);
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

// ---------------------------------------------------------------------------
// The decode step with the short conv fused in front of it.  One CTA of 256
// threads per (sequence, head) owns the whole head, so it alone reads and
// rewrites the head's channels of the sequence's window, and no other CTA
// waits on it.  Thread (part, c), part = tid / 128, convolves channel c of q
// (part 0) or k (part 1) over the window's three rows and the new projection
// row (optional SiLU), then channel c of v (part 0) or takes exp(g) of it
// (part 1); the thread that read a channel's taps writes its new taps (taps 1
// and 2 move down, the projection row becomes tap 2), since no other thread
// touches that channel.  q and k are scaled to unit L2 norm per head after a
// block reduction.  The 128 value rows are then stepped in four blocks of 32
// (eight threads a row, as in kda_decode_kernel, so token_step runs unchanged).
// All four blocks' state rows are requested before the conv and held in
// registers (64 a thread, two CTAs per SM), so that the whole 64 KB state is
// in flight while the slot ids, the window and the conv are dealt with
// (measured per 64 x 32-head step: 47.9 us; two blocks in flight at three
// CTAs per SM, 61.6 us; 512 threads a CTA, 52.0 us; 1024, 69 us).
// ---------------------------------------------------------------------------
struct DecodeConvParams {
    const uint16_t *xq, *xk, *xv;  // [N][H][128] bf16: this step's projections
    const float *w;                // [3][H*128][4] conv weights (stream, channel, tap)
    const int32_t *conv_slots;     // [N] or nullptr (entry n)
    uint16_t *conv_pool;           // [conv_num_slots][3 taps][3 streams][H*128] bf16
    const float *g, *beta;         // [N][H][128], [N][H]
    const int32_t *slots;          // [N] or nullptr (entry n)
    float *pool;                   // [num_slots][H][128][128]
    uint16_t *out;                 // [N][H][128] bf16
    int N, H, num_slots, conv_num_slots, act;
    float eps;
    int *err;
};

__device__ __forceinline__ float conv4(float4 w, uint16_t t0, uint16_t t1, uint16_t t2, uint16_t x, int act)
{
    float y = w.x * bf16_bits_to_float(t0);
    y = fmaf(w.y, bf16_bits_to_float(t1), y);
    y = fmaf(w.z, bf16_bits_to_float(t2), y);
    y = fmaf(w.w, bf16_bits_to_float(x), y);
    return act ? y / (1.f + dec_ex2(-y * kDecLog2e)) : y;
}

constexpr int kDcThreads = 256;   // 32 value rows x 8 threads, four row blocks in turn

__global__ void __launch_bounds__(kDcThreads, 2) kda_decode_conv_kernel(DecodeConvParams p)
{
    __shared__ float4 sa[32], sk[32], sq[32];   // exp(g), k, q of this (sequence, head), 128 each
    __shared__ float sv[128];                   // v
    __shared__ float red[8];                    // per-warp sums of y^2 (warps 0-3: q, 4-7: k)
    const int rh = blockIdx.x;                  // (sequence, head)
    const int n = rh / p.H, h = rh % p.H;
    const size_t row = (size_t)n * p.H + h;
    const size_t C = (size_t)p.H * 128;
    const int tid = threadIdx.x;
    const int part = tid >> 7, c = tid & 127;                  // 0: q then v, 1: k then g; channel
    const size_t ch = (size_t)h * 128 + c;
    const int slot = decode_slot(p.slots, n, p.num_slots, p.err);
    const int cslot = decode_slot(p.conv_slots, n, p.conv_num_slots, p.err);
    if (slot < 0 || cslot < 0) return;   // padded row: nothing is computed or written
    const int vl = tid >> 3, qe = tid & 7;      // value row vl of each block, its pieces 8j + qe
    float4 *st = reinterpret_cast<float4 *>(p.pool + (((size_t)slot * p.H + h) * 128 + vl) * 128);
    constexpr int kBlk = kDecRows * 128 / 4;    // float4 stride between row blocks
    // every block's state rows go out first: they do not depend on the conv
    float4 s0[4], s1[4], s2[4], s3[4];
#pragma unroll
    for (int j = 0; j < 4; j++) s0[j] = st[8 * j + qe];
#pragma unroll
    for (int j = 0; j < 4; j++) s1[j] = st[kBlk + 8 * j + qe];
#pragma unroll
    for (int j = 0; j < 4; j++) s2[j] = st[2 * kBlk + 8 * j + qe];
#pragma unroll
    for (int j = 0; j < 4; j++) s3[j] = st[3 * kBlk + 8 * j + qe];
    uint16_t *win = p.conv_pool + (size_t)cslot * 9 * C;       // [tap][stream][H*128]
    const float4 wq4 = *reinterpret_cast<const float4 *>(p.w + ((size_t)part * C + ch) * 4);
    float4 wv4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint16_t ax = (part ? p.xk : p.xq)[row * 128 + c];
    uint16_t bx = 0;
    float gc = 0.f;
    if (part == 0) {
        wv4 = *reinterpret_cast<const float4 *>(p.w + ((size_t)2 * C + ch) * 4);
        bx = p.xv[row * 128 + c];
    } else {
        gc = p.g[row * 128 + c];
    }
    const float beta = p.beta[row];
    const uint16_t a0 = win[part * C + ch], a1 = win[(3 + part) * C + ch], a2 = win[(6 + part) * C + ch];
    uint16_t b0 = 0, b1 = 0, b2 = 0;
    if (part == 0) { b0 = win[2 * C + ch]; b1 = win[5 * C + ch]; b2 = win[8 * C + ch]; }
    // the taps this thread read are read by no other thread: the new window now
    win[part * C + ch] = a1; win[(3 + part) * C + ch] = a2; win[(6 + part) * C + ch] = ax;
    if (part == 0) { win[2 * C + ch] = b1; win[5 * C + ch] = b2; win[8 * C + ch] = bx; }
    const float y = conv4(wq4, a0, a1, a2, ax, p.act);
    if (part == 0) sv[c] = conv4(wv4, b0, b1, b2, bx, p.act);
    else reinterpret_cast<float *>(sa)[c] = dec_ex2(gc * kDecLog2e);
    float y2 = y * y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) y2 += __shfl_xor_sync(0xffffffffu, y2, o);
    if ((tid & 31) == 0) red[tid >> 5] = y2;
    __syncthreads();
    {
        const float *r4 = red + 4 * part;
        const float n2 = (r4[0] + r4[1]) + (r4[2] + r4[3]);
        reinterpret_cast<float *>(part ? sk : sq)[c] = y / sqrtf(n2 + p.eps);
    }
    __syncthreads();
    uint16_t *out = p.out + row * 128 + vl;
    auto finish = [&](float4 (&s)[4], int b) {
        const float o = token_step(s, sa, sk, sq, qe, sv[kDecRows * b + vl], beta);
#pragma unroll
        for (int j = 0; j < 4; j++) st[kBlk * b + 8 * j + qe] = s[j];
        if (qe == 0) {
            const __nv_bfloat16 ob = __float2bfloat16_rn(o);
            out[kDecRows * b] = *reinterpret_cast<const uint16_t *>(&ob);
        }
    };
    finish(s0, 0);
    finish(s1, 1);
    finish(s2, 2);
    finish(s3, 3);
}

struct FoldParams {
    const uint16_t *k, *v;       // [N][W][H][128] bf16: each sequence's window of W tokens
    const float *g, *beta;       // [N][W][H][128], [N][W][H]
    const int32_t *accepted;     // [N]: fold the first accepted[n] tokens of the window
    const int32_t *slots;        // [N] or nullptr (entry n)
    float *pool;                 // [num_slots][H][128][128]
    int N, W, H, num_slots;
    int items;                   // 4 N H: (sequence, head, quarter of the value rows)
    int *err;
};

// Commit of a speculative round: the state takes the first accepted[n] tokens
// of sequence n's window, one token_step each.  A persistent CTA walks items
// (sequence, head, quarter of the value rows); while it steps one item's state
// (in registers) through its tokens, the next item's state rows are loading
// into registers and its tokens' g, k, v and beta are copying (cp.async) into
// the other of two raw buffers.  Before an item's steps its raw tokens become
// exp(g), k, v and beta in fp32 (the decode step's operands), so the steps
// wait on no memory.  Up to kFoldBatch tokens go ahead like this; further ones
// (windows longer than kFoldBatch) are staged batch by batch.
constexpr int kFoldBatch = 16;

struct FoldItem {
    int n, h, vq, slot, acc;     // acc 0: nothing to do (padded, bad id, or none accepted)
};

__device__ __forceinline__ FoldItem fold_item(const FoldParams &p, int q)
{
    FoldItem it;
    it.n = (q >> 2) / p.H;
    it.h = (q >> 2) % p.H;
    it.vq = q & 3;
    it.slot = decode_slot(p.slots, it.n, p.num_slots, p.err);
    it.acc = 0;
    if (it.slot >= 0) {
        int acc = p.accepted[it.n];
        if (acc < 0 || acc > p.W) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBadAccepted);
            acc = acc < 0 ? 0 : p.W;
        }
        it.acc = acc;
    }
    return it;
}

__device__ __forceinline__ uint32_t smem_addr(const void *ptr) { return (uint32_t)__cvta_generic_to_shared(ptr); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct FoldRaw {                 // one item's first kFoldBatch tokens as stored in global memory
    float g[kFoldBatch][128];
    uint16_t k[kFoldBatch][128];
    uint16_t v[kFoldBatch][kDecRows];   // this quarter's value rows only
    float beta[kFoldBatch];
};

__device__ __forceinline__ size_t fold_row(const FoldParams &p, const FoldItem &it, int t)
{
    return ((size_t)it.n * p.W + t) * p.H + it.h;
}

__device__ void fold_issue_tokens(const FoldParams &p, const FoldItem &it, FoldRaw &raw, int tid)
{
    const int nt = min(it.acc, kFoldBatch);
    for (int i = tid; i < nt * 32; i += kDecThreads) {     // g: 32 pieces of 16 B a token
        const int t = i >> 5, c = 4 * (i & 31);
        cp_async16(&raw.g[t][c], p.g + fold_row(p, it, t) * 128 + c);
    }
    for (int i = tid; i < nt * 16; i += kDecThreads) {     // k: 16 pieces
        const int t = i >> 4, c = 8 * (i & 15);
        cp_async16(&raw.k[t][c], p.k + fold_row(p, it, t) * 128 + c);
    }
    for (int i = tid; i < nt * 4; i += kDecThreads) {      // v of this quarter: 4 pieces
        const int t = i >> 2, c = 8 * (i & 3);
        cp_async16(&raw.v[t][c], p.v + fold_row(p, it, t) * 128 + kDecRows * it.vq + c);
    }
    if (tid < nt) cp_async4(&raw.beta[tid], p.beta + fold_row(p, it, tid));
}

__global__ void __launch_bounds__(kDecThreads, 4) kda_fold_kernel(FoldParams p)
{
    __shared__ FoldRaw raw[2];
    __shared__ float4 sa[kFoldBatch][32], sk[kFoldBatch][32];
    __shared__ float sv[kFoldBatch][kDecRows], sb[kFoldBatch];
    const int tid = threadIdx.x, qe = tid & 7, vl = tid >> 3;   // value row vl of the quarter
    auto state_rows = [&](const FoldItem &it) {
        return reinterpret_cast<float4 *>(p.pool + (((size_t)it.slot * p.H + it.h) * 128 + kDecRows * it.vq + vl) * 128);
    };
    int q = blockIdx.x, b = 0;
    FoldItem it = fold_item(p, q);
    float4 s[4];
    if (it.acc > 0) {
        const float4 *st = state_rows(it);
#pragma unroll
        for (int j = 0; j < 4; j++) s[j] = st[8 * j + qe];
        fold_issue_tokens(p, it, raw[0], tid);
    }
    cp_async_commit();
    while (q < p.items) {
        const int qn = q + gridDim.x;
        FoldItem nx;
        nx.acc = 0;
        if (qn < p.items) nx = fold_item(p, qn);
        if (it.acc > 0) {
            // this item's raw tokens have landed and the previous item's steps are
            // over: convert them into the step operands
            cp_async_wait_all();
            __syncthreads();
            const int nt = min(it.acc, kFoldBatch);
            for (int i = tid; i < nt * 128; i += kDecThreads) {
                const int t = i >> 7, c = i & 127;
                reinterpret_cast<float *>(sa[t])[c] = dec_ex2(raw[b].g[t][c] * kDecLog2e);
                reinterpret_cast<float *>(sk[t])[c] = bf16_bits_to_float(raw[b].k[t][c]);
            }
            for (int i = tid; i < nt * kDecRows; i += kDecThreads)
                sv[i / kDecRows][i % kDecRows] = bf16_bits_to_float(raw[b].v[i / kDecRows][i % kDecRows]);
            if (tid < nt) sb[tid] = raw[b].beta[tid];
            __syncthreads();
        }
        // the next item's state and tokens go out before this item's steps
        float4 sn[4];
        if (nx.acc > 0) {
            const float4 *st = state_rows(nx);
#pragma unroll
            for (int j = 0; j < 4; j++) sn[j] = st[8 * j + qe];
            fold_issue_tokens(p, nx, raw[b ^ 1], tid);
        }
        cp_async_commit();
        if (it.acc > 0) {
            const int nt = min(it.acc, kFoldBatch);
            for (int t = 0; t < nt; t++) token_step(s, sa[t], sk[t], nullptr, qe, sv[t][vl], sb[t]);
            for (int t0 = kFoldBatch; t0 < it.acc; t0 += kFoldBatch) {   // windows longer than kFoldBatch
                const int mt = min(kFoldBatch, it.acc - t0);
                __syncthreads();                 // the previous batch is no longer read
                for (int i = tid; i < mt * 128; i += kDecThreads) {
                    const int t = i >> 7, c = i & 127;
                    const size_t row = fold_row(p, it, t0 + t);
                    reinterpret_cast<float *>(sa[t])[c] = dec_ex2(p.g[row * 128 + c] * kDecLog2e);
                    reinterpret_cast<float *>(sk[t])[c] = bf16_bits_to_float(p.k[row * 128 + c]);
                    if (c < kDecRows) sv[t][c] = bf16_bits_to_float(p.v[row * 128 + kDecRows * it.vq + c]);
                    if (c == 0) sb[t] = p.beta[row];
                }
                __syncthreads();
                for (int t = 0; t < mt; t++) token_step(s, sa[t], sk[t], nullptr, qe, sv[t][vl], sb[t]);
            }
            float4 *st = state_rows(it);
#pragma unroll
            for (int j = 0; j < 4; j++) st[8 * j + qe] = s[j];
        }
#pragma unroll
        for (int j = 0; j < 4; j++) s[j] = sn[j];
        it = nx;
        q = qn;
        b ^= 1;
    }
    cp_async_wait_all();
}

}  // namespace

cudaError_t launch_kda_decode_conv_bf16_d128(const DecodeConvArgs &a)
{
    if (a.N == 0) return cudaSuccess;
    DecodeConvParams p;
    p.xq = (const uint16_t *)a.xq; p.xk = (const uint16_t *)a.xk; p.xv = (const uint16_t *)a.xv;
    p.w = a.conv_weight; p.conv_slots = a.conv_slots; p.conv_pool = (uint16_t *)a.conv_pool;
    p.g = a.g; p.beta = a.beta; p.slots = a.state_slots; p.pool = a.state_pool;
    p.out = (uint16_t *)a.out;
    p.N = a.N; p.H = a.H; p.num_slots = a.num_slots; p.conv_num_slots = a.conv_num_slots;
    p.act = a.activation; p.eps = a.eps;
    p.err = a.err_word;
    kda_decode_conv_kernel<<<a.N * a.H, kDcThreads, 0, a.stream>>>(p);
    return cudaGetLastError();
}

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
    p.items = (128 / kDecRows) * a.N * a.H;
    p.err = a.err_word;
    const int per_sm = 4;
    const int grid = a.num_sms > 0 && p.items > a.num_sms * per_sm ? a.num_sms * per_sm : p.items;
    kda_fold_kernel<<<grid, kDecThreads, 0, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
