// kda_simt.cu -- the full-range KDA chunked prefill on CUDA cores (fp32).
//
// One CTA of 512 threads per (sequence, head), fp32 throughout, no tensor
// cores.  It serves every (dk, dv) in {64, 128} x {64, 128} with bf16 or fp32
// q/k/v, and has no limit on the decay: every decay factor inside a chunk is
// formed directly from a difference of cumulative log-decays, never split
// into a product of a large and a small factor, so strong gates (alpha near
// 0) and mild growth (g > 0) are computed as the recurrence defines them.
//
// Per 64-row chunk of one (sequence, head), rows r < L valid (L <= 64), with
// G_r = sum_{u<=r} g_u (per key channel) and S0 the state at the chunk start
// (the chunked WY form of S_t = (I - b k k^T) Diag(exp(g_t)) S_{t-1} + b k v^T,
// o_t = S_t^T q_t):
//
//   A_ij  = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)      j < i   (strictly lower)
//   B_ri  =        sum_c q_rc k_ic exp(G_rc - G_ic)      i <= r  (lower, diagonal included)
//   T     = (I + A)^-1                                  (blocked forward substitution)
//   R     = diag(beta) (V - (K * exp(G)) S0)
//   Delta = T R                                         (== U - W S0)
//   O     = (Q * exp(G)) S0 + B Delta
//   S1    = Diag(exp(G_{L-1})) S0 + (K * exp(G_{L-1} - G))^T Delta
//
// Every exponent above is <= 0 when g <= 0; G is kept in base 2 (exp(x) =
// 2^(x log2 e)).  The state is complete at each chunk end, so a sequence split
// into calls at a multiple of 64 rows gives the same bits as one call.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kAS = kChunk + 1;   // row stride of the 64 x 64 matrices
constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the special-function unit: a relative error of a few units of fp32
// rounding, results below the normal range flushed to zero (such a decay
// factor is negligible next to the others of its row).  The pairwise decay
// products of A and B -- 266k of them a chunk at dk = 128 -- take it.
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct SimtParams {
    const void *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu;
    const float *s0;
    void *out;
    float *s1;
    int N, T, H;
    int *err;
    const int32_t *slots;   // [N] state entries (-1 padding), or nullptr (entry n)
    int num_slots;
};

// Shared memory, in floats.  S is the state S[c][v] (key channel major); K, Q
// and G hold the chunk's k, q and cumulative log-decay and are later turned,
// element by element, into K*exp(G_{L-1}-G), Q*exp(G) and beta*K*exp(G); V
// holds beta*V and then R; Delta reuses G's slot once R is formed.
template <int DK, int DV>
struct SimtLayout {
    static constexpr int S = 0;
    static constexpr int K = S + DK * DV;
    static constexpr int Q = K + kChunk * DK;
    static constexpr int G = Q + kChunk * DK;
    static constexpr int V = G + kChunk * (DK > DV ? DK : DV);
    static constexpr int A = V + kChunk * DV;
    static constexpr int B = A + kChunk * kAS;
    static constexpr int Beta = B + kChunk * kAS;
    static constexpr int GL = Beta + kChunk;     // G of the last valid row
    static constexpr int EL = GL + DK;           // exp(G of the last valid row)
    static constexpr int Floats = EL + DK;
    static constexpr int Bytes = Floats * 4;
};

template <int W>
__device__ __forceinline__ void load_vec(const float *p, float (&x)[W])
{
    if constexpr (W == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        x[0] = t.x; x[1] = t.y;
    }
}

// 16 bytes of a row as fp32: 8 bf16 or 4 floats
template <typename T> struct Piece;
template <> struct Piece<float> {
    static constexpr int n = 4;
    static __device__ __forceinline__ void get(const float *src, float *dst)
    {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
        dst[0] = x.x; dst[1] = x.y; dst[2] = x.z; dst[3] = x.w;
    }
};
template <> struct Piece<__nv_bfloat16> {
    static constexpr int n = 8;
    static __device__ __forceinline__ void get(const __nv_bfloat16 *src, float *dst)
    {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            dst[2 * e] = __uint_as_float(w[e] << 16);
            dst[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
};

// rows row0 .. row0+63 of one head of a [T][H][D] tensor -> [64][D] fp32 in
// shared memory (rows at and past L zero); each thread's pieces are all
// requested before the first is stored
template <typename T, int D>
__device__ __forceinline__ void load_tile(const T *src, float *dst, int row0, int L, size_t rs, int h, int tid)
{
    constexpr int P = Piece<T>::n, PR = D / P, N = (kChunk * PR + kThreads - 1) / kThreads;
    float x[N][P];
#pragma unroll
    for (int k = 0; k < N; k++) {
        const int i = tid + k * kThreads, r = i / PR, c = (i % PR) * P;
        if (i < kChunk * PR && r < L) {
            Piece<T>::get(src + ((size_t)(row0 + r) * rs + h) * D + c, x[k]);
        } else {
#pragma unroll
            for (int e = 0; e < P; e++) x[k][e] = 0.f;
        }
    }
#pragma unroll
    for (int k = 0; k < N; k++) {
        const int i = tid + k * kThreads;
        if (i < kChunk * PR) {
            float *d = dst + (i / PR) * D + (i % PR) * P;
#pragma unroll
            for (int e = 0; e < P; e += 4) *reinterpret_cast<float4 *>(d + e) = make_float4(x[k][e], x[k][e + 1], x[k][e + 2], x[k][e + 3]);
        }
    }
}

// T = (I + A)^-1 for the strictly lower A in As ([64][kAS]; its upper half
// zero).  T is unit lower triangular; T[i][j] (i > j) is written to As[j][i],
// the upper half, so that A stays readable throughout.  In 16 x 16 blocks: the
// diagonal blocks by forward substitution (two warps, a lane per column), then
// T_IJ = -T_II sum_{K=J..I-1} A_IK T_KJ for I - J = 1, 2, 3 (block row I of
// (I + A) T = I).  Callers synchronise before and after.
__device__ void invert_unit_lower(float *As, int tid)
{
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 2) {
        const int o = 16 * (2 * warp + (lane >> 4)), c = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            float s = r == c ? 1.f : 0.f;
#pragma unroll
            for (int l = 0; l < r; l++) s = fmaf(-As[(o + r) * kAS + o + l], x[l], s);
            x[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; r++)
            if (r > c) As[(o + c) * kAS + o + r] = x[r];
    }
    // T[16K + m][16J + c] for K >= J (transposed storage, unit diagonal implicit)
    auto tval = [&](int K, int J, int m, int c) -> float {
        if (K > J || m > c) return As[(16 * J + c) * kAS + 16 * K + m];
        return m == c ? 1.f : 0.f;
    };
    for (int d = 1; d < 4; d++) {
        __syncthreads();
        const int nb = 4 - d;                                // blocks (J + d, J), J < nb
        for (int e = tid; e < nb * 256; e += kThreads) {     // P_IJ[l][c] into T_IJ's place
            const int J = e >> 8, I = J + d, l = (e >> 4) & 15, c = e & 15;
            float s = 0.f;
            for (int K = J; K < I; K++)
#pragma unroll
                for (int m = 0; m < 16; m++) s = fmaf(As[(16 * I + l) * kAS + 16 * K + m], tval(K, J, m, c), s);
            As[(16 * J + c) * kAS + 16 * I + l] = s;
        }
        __syncthreads();
        if (tid < nb * 16) {                                 // T_IJ[:, c] = -T_II P_IJ[:, c]
            const int J = tid >> 4, I = J + d, c = tid & 15;
            float pcol[16];
#pragma unroll
            for (int l = 0; l < 16; l++) pcol[l] = As[(16 * J + c) * kAS + 16 * I + l];
#pragma unroll
            for (int r = 0; r < 16; r++) {
                float s = pcol[r];
#pragma unroll
                for (int l = 0; l < r; l++) s = fmaf(As[(16 * I + l) * kAS + 16 * I + r], pcol[l], s);
                As[(16 * J + c) * kAS + 16 * I + r] = -s;
            }
        }
    }
}

template <typename Tin, typename Tout, int DK, int DV, bool kSlots>
__global__ void __launch_bounds__(kThreads, 1) kda_simt_kernel(SimtParams p)
{
    using Lay = SimtLayout<DK, DV>;
    constexpr int VW = DV / 32;   // value columns per lane
    constexpr int CW = DK / kWarps;   // key channels per warp in the state update
    extern __shared__ __align__(16) float sm[];
    float *S = sm + Lay::S, *Ks = sm + Lay::K, *Qs = sm + Lay::Q, *Gs = sm + Lay::G, *Vs = sm + Lay::V;
    float *As = sm + Lay::A, *Bs = sm + Lay::B, *bs = sm + Lay::Beta, *gl = sm + Lay::GL, *el = sm + Lay::EL;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const Tin *q = static_cast<const Tin *>(p.q), *k = static_cast<const Tin *>(p.k), *v = static_cast<const Tin *>(p.v);
    Tout *out = static_cast<Tout *>(p.out);

    int st = n;
    if constexpr (kSlots) {
        st = p.slots[n];
        if (st < -1 || st >= p.num_slots) {
            if (tid == 0) atomicOr(p.err, kErrBadSlot);
            return;
        }
        if (st < 0) return;   // padding: nothing computed or written
    }
    const int bos = clamp_row(p.cu[n], p.T, p.err);
    int eos = clamp_row(p.cu[n + 1], p.T, p.err);
    if (eos < bos) eos = bos;
    const size_t soff = ((size_t)st * p.H + h) * DK * DV;   // [dv][dk] entry of this (sequence, head)

    for (int i = tid; i < DK * DV; i += kThreads) {          // i = v * DK + c (coalesced global reads)
        const int vv = i / DK, c = i % DK;
        S[c * DV + vv] = p.s0 ? p.s0[soff + i] : 0.f;
    }

    const size_t rs = (size_t)p.H;   // row stride in heads
    for (int row0 = bos; row0 < eos; row0 += kChunk) {
        const int L = min(kChunk, eos - row0);
        // ---- the chunk's tiles (rows past L zero): 16-byte pieces, every load of a
        //      tile issued before any is used ----
        load_tile<Tin, DK>(k, Ks, row0, L, rs, h, tid);
        load_tile<Tin, DK>(q, Qs, row0, L, rs, h, tid);
        load_tile<float, DK>(p.g, Gs, row0, L, rs, h, tid);
        load_tile<Tin, DV>(v, Vs, row0, L, rs, h, tid);
        if (tid < kChunk) bs[tid] = tid < L ? __ldg(p.beta + (size_t)(row0 + tid) * rs + h) : 0.f;
        __syncthreads();
        // ---- G = running sum of g over the rows, per key channel, kept in base 2
        //      (exp(x) = 2^(x log2 e)) ----
        if (tid < DK) {
            float acc = 0.f;
            for (int r = 0; r < kChunk; r++) {   // rows past L add zero
                acc += Gs[r * DK + tid];
                Gs[r * DK + tid] = acc * kLog2e;
            }
            gl[tid] = acc * kLog2e;
            el[tid] = exp2f(acc * kLog2e);
        }
        __syncthreads();
        // ---- A (beta-scaled, strictly lower) and B (lower with diagonal) ----
        // In 2 x 2 tiles of pairs: rows 2I, 2I+1 against rows 2J, 2J+1 (J <= I;
        // 528 tiles, thread tid takes tiles tid, tid + 512), so that each channel
        // step reads ten values for four pairs.  The channel loop is skewed by
        // the lane, so that the lanes of a warp read 32 different banks.
        for (int tl = tid; tl < (kChunk / 2) * (kChunk / 2 + 1) / 2; tl += kThreads) {
            int I = (int)((sqrtf(8.f * tl + 1.f) - 1.f) * 0.5f);
            if ((I + 1) * (I + 2) / 2 <= tl) I++;          // float rounding of the root
            if (I * (I + 1) / 2 > tl) I--;
            const int J = tl - I * (I + 1) / 2;
            const int i0 = 2 * I, j0 = 2 * J;
            float sa[2][2] = {}, sb[2][2] = {};
#pragma unroll 2
            for (int cc = 0; cc < DK; cc++) {
                const int c = (cc + lane) & (DK - 1);
                float ki[2], qi[2], gi[2], kj[2], gj[2];
#pragma unroll
                for (int a = 0; a < 2; a++) {
                    ki[a] = Ks[(i0 + a) * DK + c];
                    qi[a] = Qs[(i0 + a) * DK + c];
                    gi[a] = Gs[(i0 + a) * DK + c];
                    kj[a] = Ks[(j0 + a) * DK + c];
                    gj[a] = Gs[(j0 + a) * DK + c];
                }
#pragma unroll
                for (int a = 0; a < 2; a++)
#pragma unroll
                    for (int b2 = 0; b2 < 2; b2++) {
                        const float w = ex2_fast(gi[a] - gj[b2]) * kj[b2];
                        sa[a][b2] = fmaf(ki[a], w, sa[a][b2]);
                        sb[a][b2] = fmaf(qi[a], w, sb[a][b2]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 2; a++)
#pragma unroll
                for (int b2 = 0; b2 < 2; b2++) {
                    const int i = i0 + a, j = j0 + b2;
                    if (j > i) continue;                   // (the diagonal tile's upper corner)
                    As[i * kAS + j] = j < i ? bs[i] * sa[a][b2] : 0.f;
                    Bs[i * kAS + j] = sb[a][b2];
                }
        }
        for (int pr = tid; pr < kChunk * (kChunk - 1) / 2; pr += kThreads) {   // the upper triangles: zero
            int j = (int)((sqrtf(8.f * pr + 1.f) - 1.f) * 0.5f);
            if ((j + 1) * (j + 2) / 2 <= pr) j++;
            if (j * (j + 1) / 2 > pr) j--;
            const int i = pr - j * (j + 1) / 2;            // i < j + 1
            As[i * kAS + j + 1] = 0.f;
            Bs[i * kAS + j + 1] = 0.f;
        }
        __syncthreads();
        // ---- element-wise: K -> K*exp(G_L - G), Q -> Q*exp(G), G -> beta*K*exp(G);
        //      V -> beta*V ----
        for (int i = tid; i < kChunk * DK; i += kThreads) {
            const int r = i / DK, c = i % DK;
            const float x = Gs[i], kv = Ks[i];
            const float e = exp2f(x);
            Ks[i] = kv * exp2f(gl[c] - x);
            Qs[i] = Qs[i] * e;
            Gs[i] = bs[r] * (kv * e);
        }
        for (int i = tid; i < kChunk * DV; i += kThreads) Vs[i] *= bs[i / DV];
        __syncthreads();
        invert_unit_lower(As, tid);
        __syncthreads();
        const int r0 = 4 * warp, v0 = VW * lane;   // this thread's 4 rows x VW value columns
        // ---- R = beta*V - (beta*K*exp(G)) S0, in place over V ----
        {
            float acc[4][VW] = {};
            for (int c = 0; c < DK; c++) {
                float s[VW];
                load_vec<VW>(S + c * DV + v0, s);
#pragma unroll
                for (int a = 0; a < 4; a++) {
                    const float kg = Gs[(r0 + a) * DK + c];
#pragma unroll
                    for (int b = 0; b < VW; b++) acc[a][b] = fmaf(kg, s[b], acc[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; a++)   // this thread's own elements of V
#pragma unroll
                for (int b = 0; b < VW; b++) Vs[(r0 + a) * DV + v0 + b] -= acc[a][b];
        }
        __syncthreads();   // R complete, and every read of the KG slot done
        // ---- Delta = T R into G's slot ----
        float *D = Gs;
        {
            float acc[4][VW];
#pragma unroll
            for (int a = 0; a < 4; a++) load_vec<VW>(Vs + (r0 + a) * DV + v0, acc[a]);   // unit diagonal
            for (int j = 0; j < r0 + 3; j++) {
                float x[VW];
                load_vec<VW>(Vs + j * DV + v0, x);
#pragma unroll
                for (int a = 0; a < 4; a++) {
                    const float t = j < r0 + a ? As[j * kAS + r0 + a] : 0.f;   // T[r0+a][j], kept transposed
#pragma unroll
                    for (int b = 0; b < VW; b++) acc[a][b] = fmaf(t, x[b], acc[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < VW; b++) D[(r0 + a) * DV + v0 + b] = acc[a][b];
        }
        __syncthreads();
        // ---- O = (Q*exp(G)) S0 + B Delta -> out (rows < L) ----
        {
            float acc[4][VW] = {};
            for (int c = 0; c < DK; c++) {
                float s[VW];
                load_vec<VW>(S + c * DV + v0, s);
#pragma unroll
                for (int a = 0; a < 4; a++) {
                    const float qg = Qs[(r0 + a) * DK + c];
#pragma unroll
                    for (int b = 0; b < VW; b++) acc[a][b] = fmaf(qg, s[b], acc[a][b]);
                }
            }
            for (int j = 0; j <= r0 + 3; j++) {
                float x[VW];
                load_vec<VW>(D + j * DV + v0, x);
#pragma unroll
                for (int a = 0; a < 4; a++) {
                    const float bb = Bs[(r0 + a) * kAS + j];   // zero for j > r0 + a
#pragma unroll
                    for (int b = 0; b < VW; b++) acc[a][b] = fmaf(bb, x[b], acc[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; a++) {
                if (r0 + a < L) {
                    Tout *o = out + ((size_t)(row0 + r0 + a) * rs + h) * DV + v0;
#pragma unroll
                    for (int b = 0; b < VW; b++) store_out(o + b, acc[a][b]);
                }
            }
        }
        __syncthreads();
        // ---- S <- Diag(exp(G_L)) S + (K*exp(G_L - G))^T Delta ----
        {
            const int c0 = CW * warp;
            float acc[CW][VW];
#pragma unroll
            for (int a = 0; a < CW; a++) {
                float s[VW];
                load_vec<VW>(S + (c0 + a) * DV + v0, s);
#pragma unroll
                for (int b = 0; b < VW; b++) acc[a][b] = el[c0 + a] * s[b];
            }
            for (int r = 0; r < L; r++) {
                float x[VW];
                load_vec<VW>(D + r * DV + v0, x);
#pragma unroll
                for (int a = 0; a < CW; a++) {
                    const float ke = Ks[r * DK + c0 + a];
#pragma unroll
                    for (int b = 0; b < VW; b++) acc[a][b] = fmaf(ke, x[b], acc[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < CW; a++)
#pragma unroll
                for (int b = 0; b < VW; b++) S[(c0 + a) * DV + v0 + b] = acc[a][b];
        }
        __syncthreads();
    }
    if (p.s1) {
        __syncthreads();
        for (int i = tid; i < DK * DV; i += kThreads) {
            const int vv = i / DK, c = i % DK;
            p.s1[soff + i] = S[c * DV + vv];
        }
    }
}

template <typename Tin, typename Tout, int DK, int DV, bool kSlots>
cudaError_t launch_one(const KdaArgs &a)
{
    auto kern = kda_simt_kernel<Tin, Tout, DK, DV, kSlots>;
    constexpr int smem = SimtLayout<DK, DV>::Bytes;
    static_assert(smem <= 232448, "shared memory of the CUDA-core kernel");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    SimtParams p;
    p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.cu = a.cu_seqlens;
    p.s0 = a.initial_state; p.out = a.out; p.s1 = a.final_state;
    p.N = a.N; p.T = a.T; p.H = a.H; p.err = a.err_word;
    p.slots = a.state_slots; p.num_slots = a.num_slots;
    kern<<<(unsigned)((size_t)a.N * a.H), kThreads, smem, a.stream>>>(p);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, bool kSlots>
cudaError_t launch_dims(const KdaArgs &a)
{
    if (a.dk == 128 && a.dv == 128) return launch_one<Tin, Tout, 128, 128, kSlots>(a);
    if (a.dk == 128 && a.dv == 64) return launch_one<Tin, Tout, 128, 64, kSlots>(a);
    if (a.dk == 64 && a.dv == 128) return launch_one<Tin, Tout, 64, 128, kSlots>(a);
    if (a.dk == 64 && a.dv == 64) return launch_one<Tin, Tout, 64, 64, kSlots>(a);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_kda_simt(const KdaArgs &a, bool f32)
{
    const bool slots = a.state_slots != nullptr;
    if (f32) return slots ? launch_dims<float, float, true>(a) : launch_dims<float, float, false>(a);
    return slots ? launch_dims<__nv_bfloat16, __nv_bfloat16, true>(a)
                 : launch_dims<__nv_bfloat16, __nv_bfloat16, false>(a);
}

}  // namespace kda
