// kda_simt.cu -- fp32 CUDA-core KDA chunked prefill.
//
// The plain SIMT form of the chunked method: one CTA per (sequence, head),
// fp32 throughout, no tensor cores.  It serves the fp32-input entry point
// (kda_chunk_prefill_f32, dk = dv = 64) and computes the same per-chunk steps,
// in the same order, as the tensor-core kernel.
//
// Per 64-row chunk of one (sequence, head), rows r < L valid (L <= 64):
//   G_r   = sum_{u<=r} g_u                                 (per channel)
//   m     = (L-1)/2, a_r = exp(G_r - G_m), b_r = exp(G_m - G_r)  (midpoint reference)
//   Kp = K*a, Km = K*b, Qp = Q*a                            (rows >= L are zero)
//   A_ij  = beta_i Kp_i . Km_j  (j < i)   == beta_i sum_c k_ic k_jc exp(G_ic - G_jc)
//   B_ri  = Qp_r . Km_i          (i <= r)  == sum_c q_rc k_ic exp(G_rc - G_ic)
//   M     = (I + A)^-1 diag(beta)
//   S'    = Diag(exp(G_m)) S0                               (state seen from row m)
//   Delta = M (V - Kp S')        == U - W S0 with U = M V, W = M (K*exp(G))
//   O     = Qp S' + B Delta      == (Q*exp(G)) S0 + B Delta
//   S1    = Diag(exp(G_{L-1} - G_m)) (S' + Km^T Delta)
//          == Diag(exp(G_{L-1})) S0 + sum_i (k_i*exp(G_{L-1}-G_i)) Delta_i^T
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kAStride = kChunk + 1;

template <int D>
struct SimtSmem {
    float S[D * D];                 // S'[c][v]
    float Kp[kChunk * D];           // [r][c]; later Delta[r][v]
    float Km[kChunk * D];           // [r][c]
    float Qp[kChunk * D];           // [r][c]
    float V[kChunk * D];            // [r][v]; later R = V - Kp S'
    float A[kChunk * kAStride];     // L -> T -> M, in place
    float B[kChunk * kAStride];
    float G[kChunk * D];            // [r][c]: g of the chunk, then its cumulative sum G
    float Kin[kChunk * D];          // [r][c]: k and q of the chunk as loaded
    float Qin[kChunk * D];
    float gm[D], gl[D], pend[D];
    float beta[kChunk];
};

template <typename Tin, typename Tout, int D>
__global__ void __launch_bounds__(kThreads, 1)
kda_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                const float *__restrict__ g, const float *__restrict__ beta,
                const int32_t *__restrict__ cu, const float *initial_state,
                Tout *__restrict__ out, float *final_state, int N, int T, int H, int *err)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<D> &sm = *reinterpret_cast<SimtSmem<D> *>(smem_raw);
    const int tid = threadIdx.x;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    int bos = clamp_row(cu[n], T, err);
    int eos = clamp_row(cu[n + 1], T, err);
    if (eos < bos) eos = bos;
    const size_t state_off = ((size_t)n * H + h) * D * D;

    for (int idx = tid; idx < D * D; idx += kThreads) {
        int c = idx / D, vv = idx % D;
        sm.S[idx] = initial_state ? initial_state[state_off + (size_t)vv * D + c] : 0.f;
    }
    for (int c = tid; c < D; c += kThreads) sm.pend[c] = 1.f;
    __syncthreads();

    for (int c0 = bos; c0 < eos; c0 += kChunk) {
        const int L = min(kChunk, eos - c0);
        const int m = (L - 1) / 2;
        // The chunk's g, k, q and v tiles into shared memory, all threads, one row
        // of D channels per warp pass (rows past the chunk zero).
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            const size_t off = ((size_t)(c0 + r) * H + h) * D + c;
            const bool in = r < L;
            sm.G[idx] = in ? g[off] : 0.f;
            sm.Kin[idx] = in ? load_in(k + off) : 0.f;
            sm.Qin[idx] = in ? load_in(q + off) : 0.f;
            sm.V[idx] = in ? load_in(v + off) : 0.f;
        }
        if (tid < kChunk) sm.beta[tid] = tid < L ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
        __syncthreads();
        // G = running sum of g over the rows, per channel; G_m and G_{L-1}.
        if (tid < D) {
            float acc = 0.f;
            for (int r = 0; r < L; r++) {
                acc += sm.G[r * D + tid];
                sm.G[r * D + tid] = acc;
            }
            sm.gm[tid] = sm.G[m * D + tid];
            sm.gl[tid] = acc;
        }
        __syncthreads();
        // S <- Diag(exp(G_m)) Diag(pend) S: first the previous chunk's pending
        // decay to its last row, then the view from row m.  Two separate
        // roundings, so a context split into calls (state stored after the
        // first multiply) reproduces the single-call bits.
        for (int idx = tid; idx < D * D; idx += kThreads) {
            int c = idx / D;
            sm.S[idx] = (sm.S[idx] * sm.pend[c]) * expf(sm.gm[c]);
        }
        // Decay-scaled operands, all threads over the tile.
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            float kp = 0.f, km = 0.f, qp = 0.f;
            if (r < L) {
                const float G = sm.G[idx];
                const float a = expf(G - sm.gm[c]);
                const float b = expf(sm.gm[c] - G);
                const float kv = sm.Kin[idx], qv = sm.Qin[idx];
                kp = kv * a;
                km = kv * b;
                qp = qv * a;
            }
            sm.Kp[idx] = kp;
            sm.Km[idx] = km;
            sm.Qp[idx] = qp;
        }
        __syncthreads();
        // A (strictly lower, beta-scaled) and B (lower incl. diagonal).  The
        // channel loop starts at a per-row offset so that a warp's reads of
        // different rows fall in different banks.
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
            const int i = idx / kChunk, j = idx % kChunk;
            float sa = 0.f, sb = 0.f;
            if (j <= i) {
                for (int cc = 0; cc < D; cc++) {
                    const int c = (cc + j) & (D - 1);
                    const float kmj = sm.Km[j * D + c];
                    sa += sm.Kp[i * D + c] * kmj;
                    sb += sm.Qp[i * D + c] * kmj;
                }
            }
            sm.A[i * kAStride + j] = (j < i) ? sm.beta[i] * sa : 0.f;
            sm.B[i * kAStride + j] = sb;
        }
        // (I + A)^-1 by right-looking forward substitution, in place: at step j
        // row j is final; rows i > j take -A_ij T_j.  Slot j of row i holds
        // A_ij until step j reads it, then T_ij.
        for (int j = 0; j < kChunk - 1; j++) {
            __syncthreads();
            const int i = tid;
            if (i > j && i < kChunk) {
                float a = sm.A[i * kAStride + j];
                sm.A[i * kAStride + j] = -a;
                for (int l = 0; l < j; l++) sm.A[i * kAStride + l] -= a * sm.A[j * kAStride + l];
            }
        }
        __syncthreads();
        // M = T diag(beta), T unit lower triangular.
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
            const int i = idx / kChunk, j = idx % kChunk;
            float t = (j < i) ? sm.A[i * kAStride + j] : (j == i ? 1.f : 0.f);
            sm.A[i * kAStride + j] = t * sm.beta[j];
        }
        __syncthreads();
        // R = V - Kp S'
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int r = idx / D, vv = idx % D;
            float s = 0.f;
            for (int c = 0; c < D; c++) s += sm.Kp[r * D + c] * sm.S[c * D + vv];
            sm.V[idx] -= s;
        }
        __syncthreads();
        // Delta = M R  (into the Kp buffer)
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int r = idx / D, vv = idx % D;
            float s = 0.f;
            for (int j = 0; j <= r; j++) s += sm.A[r * kAStride + j] * sm.V[j * D + vv];
            sm.Kp[idx] = s;
        }
        __syncthreads();
        // O = Qp S' + B Delta
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int r = idx / D, vv = idx % D;
            if (r < L) {
                float s = 0.f;
                for (int c = 0; c < D; c++) s += sm.Qp[r * D + c] * sm.S[c * D + vv];
                for (int i = 0; i <= r; i++) s += sm.B[r * kAStride + i] * sm.Kp[i * D + vv];
                store_out(out + ((size_t)(c0 + r) * H + h) * D + vv, s);
            }
        }
        __syncthreads();
        // S <- S' + Km^T Delta; the decay to row L-1 is applied lazily.
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int c = idx / D, vv = idx % D;
            float s = sm.S[idx];
            for (int j = 0; j < L; j++) s += sm.Km[j * D + c] * sm.Kp[j * D + vv];
            sm.S[idx] = s;
        }
        for (int c = tid; c < D; c += kThreads) sm.pend[c] = expf(sm.gl[c] - sm.gm[c]);
        __syncthreads();
    }
    if (final_state) {
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int vv = idx / D, c = idx % D;
            final_state[state_off + idx] = sm.S[c * D + vv] * sm.pend[c];
        }
    }
}

}  // namespace

template <typename Tin, typename Tout, int D>
static cudaError_t launch_simt(const KdaArgs &a)
{
    auto kern = kda_simt_kernel<Tin, Tout, D>;
    const int smem = (int)sizeof(SimtSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<a.N * a.H, kThreads, smem, a.stream>>>(
        (const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, a.g, a.beta, a.cu_seqlens,
        a.initial_state, (Tout *)a.out, a.final_state, a.N, a.T, a.H, a.err_word);
    return cudaGetLastError();
}

cudaError_t launch_kda_simt_f32_d64(const KdaArgs &a) { return launch_simt<float, float, 64>(a); }

}  // namespace kda
