// kda_conv.cu -- the short-conv + L2-norm prologue of a KDA layer over packed
// sequences, with each sequence's conv window carried across calls in a
// slot-addressed pool (kern-k3-pp-prefill README: section "P: the packed
// prefill" runs the KDA layers with per-sequence conv windows and states;
// section "D inside SGLang" keeps the window in the engine's pool, laid out
// [slot][tap][q | k | v] bf16 and indexed by the same slot ids as the state).
//
// For sequence n (rows bos .. eos-1, t counted from bos), stream s in
// {q, k, v} and channel c (flat over the H heads of 128 channels):
//     x_{-3}, x_{-2}, x_{-1}  = the window's taps 0, 1, 2 (oldest first)
//     y_t[c] = sum_{j=0..3} w[s][c][j] x_{t-3+j}[c]   (tap 3 weighs the row itself)
//     y_t    = act(y_t)                                (identity or SiLU)
//     q_t, k_t = y_t / sqrt(|y_t|^2 + eps)             (per head, 128 channels)
//     v_t    = y_t
// after which the window holds x_{L-3}, x_{L-2}, x_{L-1}: the last three rows
// of [old taps ; the sequence's L rows].
//
// kda_conv_kernel: one warp per (block of 64 rows, head, stream).  Lane l owns
// channels 4l .. 4l+3 of the head and holds their 16 weights.  Rows go in
// groups of four over a window of seven rows in registers (the three before
// the group and the group), with the next group's loads in flight; each row is
// one 256-byte load and one 256-byte store per warp.  The L2 norms of a
// group's four rows are one butterfly across the warp (ten shuffles).  The kernel is bound by instruction issue rather than by memory,
// so the per-row code is kept short (no per-row register shifts).  Only the warp that holds a sequence's first row reads the
// sequence's window (for that row's three predecessors), so that warp also
// writes the new window, right after reading the old one; the new taps are
// input rows (or, for sequences shorter than three rows, old taps it holds).
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_conv.h"

namespace kda {
namespace {

constexpr int kConvRows = 64;    // rows per warp when the sequences are long (see conv_rows)
constexpr int kConvWarps = 4;    // warps per CTA

struct ConvParams {
    const uint16_t *x[3];
    uint16_t *y[3];
    const float *w;
    const int32_t *cu, *slots;
    uint16_t *pool;
    int N, T, H, num_slots, act;
    int rows;                    // rows per warp
    float eps;
    int *err;
};

// Rows per warp: a warp walks its rows in order and pays two dependent loads
// (slot id, window) at each sequence start, so short sequences get short
// blocks (measured: 64 one-row sequences at H = 32 took 115 us in 64-row
// blocks); long ones keep 64-row blocks.  Any size >= 4 keeps at most one
// block edge among a sequence's first three rows.
inline int conv_rows(long long T, int N)
{
    return T >= 48LL * N ? kConvRows : T >= 12LL * N ? 16 : 4;
}

// stream s of a 3-array kept in the kernel parameters (a runtime index would
// copy the parameter block to local memory)
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[3], int s) { return s == 0 ? a[0] : s == 1 ? a[1] : a[2]; }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi)
{
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// SiLU(a) = a * sigmoid(a) = a / (1 + 2^(-a log2 e)).  ex2.approx and the
// approximate division keep it to a few units of fp32 rounding (the form
// (a/2)(1 + tanh(a/2)) through tanh.approx loses most of its digits for
// negative a, where 1 + tanh cancels).
__device__ __forceinline__ float silu(float a)
{
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-a * 1.4426950408889634f));
    return __fdividef(a, 1.f + e);
}

// cu_seqlens[i] clamped into [0, T]
__device__ __forceinline__ int cu_at(const int32_t *cu, int i, int T) { return min(max(cu[i], 0), T); }

// The last sequence n in [0, N) with cu[n] <= t (cu non-decreasing): a 32-way
// search, one load per lane and step.
__device__ int seq_of(const int32_t *cu, int N, int T, int t, int lane)
{
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + lane * step;
        const unsigned m = __ballot_sync(0xffffffffu, idx < hi && cu_at(cu, idx, T) <= t);
        lo += (m ? 31 - __clz(m) : 0) * step;
        hi = min(lo + step, hi);
    }
    return lo;
}

// Edge x of the row blocks, moved so that no block starts among a sequence's
// first three rows (whose predecessors are window taps): then only the warp
// that holds a sequence's first row reads its window.  Both warps that share
// an edge compute it the same way.
__device__ int block_edge(const ConvParams &p, int x, int lane)
{
    if (x >= p.T) return p.T;
    const int n = seq_of(p.cu, p.N, p.T, x, lane);
    const int b = cu_at(p.cu, n, p.T), e = cu_at(p.cu, n + 1, p.T);
    const int first3 = min(b + 3, e);
    return (b < x && x < first3) ? first3 : x;
}

__global__ void __launch_bounds__(kConvWarps * 32, 6) kda_conv_kernel(ConvParams p)
{
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * kConvWarps + (threadIdx.x >> 5);   // ((block * 3 + s) * H + h)
    if (item == 0) {                              // every sequence's bounds and id, checked once
        for (int m = lane; m <= p.N; m += 32) {
            if (p.cu[m] < 0 || p.cu[m] > p.T) atomicOr(p.err, kErrBadSeqlens);
            if (m < p.N) {
                const int sl = p.slots ? p.slots[m] : m;
                if (sl < -1 || sl >= p.num_slots) atomicOr(p.err, kErrBadSlot);
            }
        }
    }
    const int h = item % p.H, s = (item / p.H) % 3, b32 = (item / p.H / 3) * p.rows;
    if (b32 >= p.T) return;
    const int t0 = block_edge(p, b32, lane), t1 = block_edge(p, b32 + p.rows, lane);
    const size_t HC = (size_t)p.H * 128;         // elements per row of a stream
    const int gc = h * 128 + 4 * lane;            // this lane's first channel
    float wt[4][4];                               // [channel][tap]
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(p.w + (s * HC + gc + i) * 4));
        wt[i][0] = f.x; wt[i][1] = f.y; wt[i][2] = f.z; wt[i][3] = f.w;
    }
    const uint16_t *xs = pick(p.x, s);
    uint16_t *ys = pick(p.y, s);
    const int tend = cu_at(p.cu, p.N, p.T);       // rows from here on belong to no sequence
    int n = seq_of(p.cu, p.N, p.T, t0, lane);
    int bos = cu_at(p.cu, n, p.T), eos = cu_at(p.cu, n + 1, p.T);
    int t = t0;
    while (t < t1 && t < tend) {
        while (t >= eos && n < p.N - 1) {         // the sequence holding row t
            n++;
            bos = cu_at(p.cu, n, p.T);
            eos = cu_at(p.cu, n + 1, p.T);
        }
        if (t < bos || t >= eos) {                // malformed cu_seqlens: a row of no sequence
            t++;
            continue;
        }
        const int seg_end = min(eos, t1);
        const int slot = p.slots ? p.slots[n] : n;
        if (slot < 0 || slot >= p.num_slots) {    // padded (or an id outside the pool) -- skipped
            t = seg_end;
            continue;
        }
        // xa holds rows g-3 .. g+3 of a group of four rows g .. g+3 (floats, this
        // lane's four channels); the three rows before t are earlier rows of the
        // sequence or the window's taps
        float xa[7][4];
        uint16_t *win = p.pool + (size_t)slot * 9 * HC + (size_t)s * HC + gc;   // tap j at win + 3 * j * HC
        uint2 raw[3];
#pragma unroll
        for (int j = 0; j < 3; j++) {
            const int r = t - 3 + j;
            raw[j] = r >= bos ? __ldg(reinterpret_cast<const uint2 *>(xs + (size_t)r * HC + gc))
                              : *reinterpret_cast<const uint2 *>(win + (size_t)(3 * (r - bos + 3)) * HC);
            xa[j][0] = bf_lo(raw[j].x); xa[j][1] = bf_hi(raw[j].x); xa[j][2] = bf_lo(raw[j].y); xa[j][3] = bf_hi(raw[j].y);
        }
        if (t == bos) {
            // This warp holds the sequence's first row, so it alone reads the old
            // window (just done) and it writes the new one: the last three rows of
            // [old taps ; the L rows].
            const int L = eos - bos;
            uint2 nw[3];
#pragma unroll
            for (int j = 0; j < 3; j++) {
                const int r = L - 3 + j;          // row of new tap j; r < 0: old tap r + 3
                nw[j] = r >= 0 ? __ldg(reinterpret_cast<const uint2 *>(xs + (size_t)(bos + r) * HC + gc))
                               : r == -2 ? raw[1] : raw[2];
            }
#pragma unroll
            for (int j = 0; j < 3; j++) *reinterpret_cast<uint2 *>(win + (size_t)(3 * j) * HC) = nw[j];
        }
        const uint16_t *xrow = xs + (size_t)t * HC + gc;     // row g of this lane's channels
        uint16_t *yrow = ys + (size_t)t * HC + gc;
        uint2 ld[4];                                           // rows g .. g+3, then the next group's
#pragma unroll
        for (int i = 0; i < 4; i++)
            ld[i] = t + i < seg_end ? __ldg(reinterpret_cast<const uint2 *>(xrow + i * HC)) : make_uint2(0u, 0u);
#pragma unroll 1
        for (int g = t; g < seg_end; g += 4, xrow += 4 * HC, yrow += 4 * HC) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                xa[3 + i][0] = bf_lo(ld[i].x); xa[3 + i][1] = bf_hi(ld[i].x);
                xa[3 + i][2] = bf_lo(ld[i].y); xa[3 + i][3] = bf_hi(ld[i].y);
                ld[i] = g + 4 + i < seg_end ? __ldg(reinterpret_cast<const uint2 *>(xrow + (4 + i) * HC))
                                            : make_uint2(0u, 0u);
            }
            float y[4][4];                        // rows g .. g+3 (past the segment: zeros, not stored)
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    float a = wt[c][0] * xa[i][c];
                    a = fmaf(wt[c][1], xa[i + 1][c], a);
                    a = fmaf(wt[c][2], xa[i + 2][c], a);
                    a = fmaf(wt[c][3], xa[i + 3][c], a);
                    y[i][c] = p.act ? silu(a) : a;
                }
            float sc[4] = {1.f, 1.f, 1.f, 1.f};
            if (s < 2) {
                // the four rows' squared norms in one butterfly: lanes 0-15 gather rows
                // 0 and 1, lanes 16-31 rows 2 and 3, then bit 3 of the lane picks one
                // row; lane 16 r1 + 8 r0 ends up with row 2 r1 + r0
                float ss[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    ss[i] = y[i][0] * y[i][0];
                    ss[i] = fmaf(y[i][1], y[i][1], ss[i]);
                    ss[i] = fmaf(y[i][2], y[i][2], ss[i]);
                    ss[i] = fmaf(y[i][3], y[i][3], ss[i]);
                }
                const bool h16 = lane & 16, h8 = lane & 8;
                const float a0 = (h16 ? ss[2] : ss[0]) + __shfl_xor_sync(0xffffffffu, h16 ? ss[0] : ss[2], 16);
                const float a1 = (h16 ? ss[3] : ss[1]) + __shfl_xor_sync(0xffffffffu, h16 ? ss[1] : ss[3], 16);
                float b = (h8 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, h8 ? a0 : a1, 8);
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
#pragma unroll
                for (int i = 0; i < 4; i++) sc[i] = rsqrtf(__shfl_sync(0xffffffffu, b, 16 * (i >> 1) + 8 * (i & 1)) + p.eps);
            }
#pragma unroll
            for (int i = 0; i < 4; i++) {
                if (g + i >= seg_end) break;
                *reinterpret_cast<uint2 *>(yrow + i * HC) = make_uint2(pack_bf2(y[i][0] * sc[i], y[i][1] * sc[i]),
                                                                       pack_bf2(y[i][2] * sc[i], y[i][3] * sc[i]));
            }
#pragma unroll
            for (int j = 0; j < 3; j++)
#pragma unroll
                for (int c = 0; c < 4; c++) xa[j][c] = xa[4 + j][c];
        }
        t = seg_end;
    }
}

}  // namespace

cudaError_t launch_kda_conv_bf16_d128(const ConvArgs &a)
{
    ConvParams p;
    for (int s = 0; s < 3; s++) {
        p.x[s] = (const uint16_t *)a.x[s];
        p.y[s] = (uint16_t *)a.y[s];
    }
    p.w = a.weight;
    p.cu = a.cu_seqlens;
    p.slots = a.conv_slots;
    p.pool = (uint16_t *)a.conv_pool;
    p.N = a.N; p.T = a.T; p.H = a.H; p.num_slots = a.num_slots;
    p.act = a.activation;
    p.eps = a.eps;
    p.err = a.err_word;
    p.rows = conv_rows(a.T, a.N);
    const long long items = (long long)((a.T + p.rows - 1) / p.rows) * 3 * a.H;
    const long long blocks = items > 0 ? (items + kConvWarps - 1) / kConvWarps : 1;   // block 0 checks the ids
    kda_conv_kernel<<<(unsigned)blocks, kConvWarps * 32, 0, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
