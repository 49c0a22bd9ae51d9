/*
 * kda_oracle.c -- plain fp64 CPU oracle for Kimi Delta Attention (KDA)
 * chunked packed-varlen prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What is computed (one (sequence, head) pair at a time, all pairs
 * independent).  KDA is the gated delta rule with a per-channel decay:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t,           alpha_t = exp(g_t)  (g is the per-token
 *                                                     log-decay, per channel)
 *
 * with S in R^{dk x dv}.  Packed sequences are separated by cu_seqlens, as in
 * the packed prefill of the kern-k3-pp-prefill README ("P: the packed
 * prefill": up to 16 sequences a call, back to back, split by cu_seqlens).
 * The recurrent state is stored per (sequence, head) as [dv][dk] fp32/fp64,
 * the SGLang pool layout [slot][head][v][k] named in the kern-k3-pp-prefill
 * README, section "D inside SGLang".
 *
 * Two independent routes are provided:
 *
 *  kda_oracle_recurrent  -- the definition written out token by token.
 *  kda_oracle_chunked    -- the chunked form, in the order the method is
 *                           described: per chunk of C rows the in-chunk
 *                           cumulative log-decay G, the strictly lower
 *                           A_kk = beta_i (k_i * exp(G_i - G_j)) . k_j, the
 *                           inverse of (I + A_kk) by forward substitution,
 *                           the WY factors W and U, the inter-chunk state
 *                           recurrence, and the outputs.  No blocking, no
 *                           factorisation of the exponentials, no fusion.
 *
 * Readings taken where the pages are silent:
 *  - no 1/sqrt(dk) query scale;  o_t reads the state after token t's write;
 *  - decay first, then erase and write with the decayed state;
 *  - g is per token (not cumulative) and is not clamped;
 *  - a zero-length sequence leaves final = initial (zeros if no initial);
 *  - chunks start at each sequence's first row; the last one is partial.
 *
 * Inputs are passed in their storage types (bf16 bits, fp32 or fp64) and
 * upcast exactly to double.  Arithmetic is fp64 throughout.
 *
 * Head selection: only the heads listed in `heads` (nsel of them, indices into
 * the H heads of the inputs) are computed; out is [T][nsel][dv] and
 * final_state is [N][nsel][dv][dk].  initial_state, when given, is
 * [N][nsel][dv][dk] too.  This lets tests check large workloads on a sample
 * of heads.
 *
 * Parallelism: (sequence, selected head) pairs are spread over `nthreads`
 * POSIX threads; each pair is computed by exactly one thread with the same
 * arithmetic, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 0, ORC_F32 = 1, ORC_F64 = 2 };

typedef struct {
    const void *q, *k, *v, *g, *beta;
    int qkv_dtype;            /* dtype of q, k, v */
    int gb_dtype;             /* dtype of g and beta */
    const int32_t *cu;        /* [N+1] */
    const double *init;       /* [N][nsel][dv][dk] or NULL */
    double *out;              /* [T][nsel][dv] */
    double *fin;              /* [N][nsel][dv][dk] or NULL */
    int N, T, H, dk, dv;
    const int32_t *heads;
    int nsel;
    int chunk;                /* 0 = token recurrence, else chunk size */
    int nthreads;
    int next;                 /* work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

static double load_val(const void *p, int dtype, size_t i)
{
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == ORC_F32)
        return (double)((const float *)p)[i];
    return ((const double *)p)[i];
}

/* Row t, head h, channel c of a [T][H][d] tensor. */
static double at3(const job_t *J, const void *p, int dtype, int t, int h, int c, int d)
{
    return load_val(p, dtype, ((size_t)t * J->H + h) * d + c);
}

static double beta_at(const job_t *J, int t, int h)
{
    return load_val(J->beta, J->gb_dtype, (size_t)t * J->H + h);
}

/* S is kept as S[c][v] (dk x dv), the orientation of the recurrence. */
static void load_state(const job_t *J, int n, int hs, double *S)
{
    int dk = J->dk, dv = J->dv;
    if (!J->init) {
        memset(S, 0, sizeof(double) * dk * dv);
        return;
    }
    const double *src = J->init + ((size_t)n * J->nsel + hs) * dv * dk;
    for (int c = 0; c < dk; c++)
        for (int v = 0; v < dv; v++)
            S[c * dv + v] = src[v * dk + c];
}

static void store_state(const job_t *J, int n, int hs, const double *S)
{
    int dk = J->dk, dv = J->dv;
    if (!J->fin)
        return;
    double *dst = J->fin + ((size_t)n * J->nsel + hs) * dv * dk;
    for (int v = 0; v < dv; v++)
        for (int c = 0; c < dk; c++)
            dst[v * dk + c] = S[c * dv + v];
}

/* ---- route 1: the recurrence, one token at a time ---------------------- */
static void run_recurrent(const job_t *J, int n, int hs, double *S, double *buf)
{
    int dk = J->dk, dv = J->dv, h = J->heads[hs];
    double *qq = buf, *kk = qq + dk, *al = kk + dk, *vv = al + dk, *e = vv + dv;
    int bos = J->cu[n], eos = J->cu[n + 1];
    load_state(J, n, hs, S);
    for (int t = bos; t < eos; t++) {
        for (int c = 0; c < dk; c++) {
            qq[c] = at3(J, J->q, J->qkv_dtype, t, h, c, dk);
            kk[c] = at3(J, J->k, J->qkv_dtype, t, h, c, dk);
            al[c] = exp(at3(J, J->g, J->gb_dtype, t, h, c, dk));
        }
        for (int v = 0; v < dv; v++)
            vv[v] = at3(J, J->v, J->qkv_dtype, t, h, v, dv);
        double b = beta_at(J, t, h);
        /* S <- Diag(alpha_t) S */
        for (int c = 0; c < dk; c++)
            for (int v = 0; v < dv; v++)
                S[c * dv + v] *= al[c];
        /* e = S^T k : what the decayed state recalls for key k */
        for (int v = 0; v < dv; v++)
            e[v] = 0.0;
        for (int c = 0; c < dk; c++)
            for (int v = 0; v < dv; v++)
                e[v] += kk[c] * S[c * dv + v];
        /* S <- S + beta k (v - e)^T  ==  (I - beta k k^T) S + beta k v^T */
        for (int v = 0; v < dv; v++)
            e[v] = b * (vv[v] - e[v]);
        for (int c = 0; c < dk; c++)
            for (int v = 0; v < dv; v++)
                S[c * dv + v] += kk[c] * e[v];
        /* o_t = S_t^T q_t */
        double *o = J->out + ((size_t)t * J->nsel + hs) * dv;
        for (int v = 0; v < dv; v++)
            o[v] = 0.0;
        for (int c = 0; c < dk; c++)
            for (int v = 0; v < dv; v++)
                o[v] += qq[c] * S[c * dv + v];
    }
    store_state(J, n, hs, S);
}

/* ---- route 2: the chunked form, step by step ---------------------------- */
static void run_chunked(const job_t *J, int n, int hs, double *S, double *buf)
{
    int dk = J->dk, dv = J->dv, h = J->heads[hs], C = J->chunk;
    /* scratch carving */
    double *G = buf;                       /* [C][dk] cumulative log-decay */
    double *K = G + (size_t)C * dk;        /* [C][dk] */
    double *Q = K + (size_t)C * dk;        /* [C][dk] */
    double *V = Q + (size_t)C * dk;        /* [C][dv] */
    double *bt = V + (size_t)C * dv;       /* [C] beta */
    double *A = bt + C;                    /* [C][C] strictly lower A_kk */
    double *Tm = A + (size_t)C * C;        /* [C][C] (I + A)^-1 */
    double *W = Tm + (size_t)C * C;        /* [C][dk] */
    double *U = W + (size_t)C * dk;        /* [C][dv] */
    double *D = U + (size_t)C * dv;        /* [C][dv] Delta = U - W S0 */
    double *B = D + (size_t)C * dv;        /* [C][C] lower A_qk incl. diagonal */
    double *Sn = B + (size_t)C * C;        /* [dk][dv] next state */

    int bos = J->cu[n], eos = J->cu[n + 1];
    load_state(J, n, hs, S);
    for (int s0 = bos; s0 < eos; s0 += C) {
        int L = eos - s0 < C ? eos - s0 : C;
        /* inputs of the chunk */
        for (int r = 0; r < L; r++) {
            for (int c = 0; c < dk; c++) {
                K[r * dk + c] = at3(J, J->k, J->qkv_dtype, s0 + r, h, c, dk);
                Q[r * dk + c] = at3(J, J->q, J->qkv_dtype, s0 + r, h, c, dk);
            }
            for (int v = 0; v < dv; v++)
                V[r * dv + v] = at3(J, J->v, J->qkv_dtype, s0 + r, h, v, dv);
            bt[r] = beta_at(J, s0 + r, h);
        }
        /* step 1: G_r = sum_{u <= r} g_u, per channel (inclusive prefix) */
        for (int c = 0; c < dk; c++) {
            double acc = 0.0;
            for (int r = 0; r < L; r++) {
                acc += at3(J, J->g, J->gb_dtype, s0 + r, h, c, dk);
                G[r * dk + c] = acc;
            }
        }
        /* step 2: A_ij = beta_i sum_c k_ic k_jc exp(G_ic - G_jc), j < i */
        for (int i = 0; i < L; i++)
            for (int j = 0; j < L; j++) {
                double s = 0.0;
                if (j < i)
                    for (int c = 0; c < dk; c++)
                        s += K[i * dk + c] * K[j * dk + c] * exp(G[i * dk + c] - G[j * dk + c]);
                A[i * C + j] = bt[i] * s;
            }
        /* step 3: T = (I + A)^-1, forward substitution on the unit diagonal:
         * row i of T is e_i - sum_{j<i} A_ij T_j */
        for (int i = 0; i < L; i++) {
            for (int j = 0; j < L; j++)
                Tm[i * C + j] = (i == j) ? 1.0 : 0.0;
            for (int j = 0; j < i; j++) {
                double a = A[i * C + j];
                for (int l = 0; l <= j; l++)
                    Tm[i * C + l] -= a * Tm[j * C + l];
            }
        }
        /* step 4: WY factors  W = T diag(beta) (K * exp(G)),  U = T diag(beta) V */
        for (int i = 0; i < L; i++) {
            for (int c = 0; c < dk; c++) {
                double s = 0.0;
                for (int j = 0; j <= i; j++)
                    s += Tm[i * C + j] * bt[j] * K[j * dk + c] * exp(G[j * dk + c]);
                W[i * dk + c] = s;
            }
            for (int v = 0; v < dv; v++) {
                double s = 0.0;
                for (int j = 0; j <= i; j++)
                    s += Tm[i * C + j] * bt[j] * V[j * dv + v];
                U[i * dv + v] = s;
            }
        }
        /* step 5: Delta = U - W S0 */
        for (int i = 0; i < L; i++)
            for (int v = 0; v < dv; v++) {
                double s = 0.0;
                for (int c = 0; c < dk; c++)
                    s += W[i * dk + c] * S[c * dv + v];
                D[i * dv + v] = U[i * dv + v] - s;
            }
        /* step 6: B_ri = sum_c q_rc k_ic exp(G_rc - G_ic), i <= r */
        for (int r = 0; r < L; r++)
            for (int i = 0; i < L; i++) {
                double s = 0.0;
                if (i <= r)
                    for (int c = 0; c < dk; c++)
                        s += Q[r * dk + c] * K[i * dk + c] * exp(G[r * dk + c] - G[i * dk + c]);
                B[r * C + i] = s;
            }
        /* step 7: o_r = (q_r * exp(G_r))^T S0 + sum_{i<=r} B_ri Delta_i */
        for (int r = 0; r < L; r++) {
            double *o = J->out + ((size_t)(s0 + r) * J->nsel + hs) * dv;
            for (int v = 0; v < dv; v++) {
                double s = 0.0;
                for (int c = 0; c < dk; c++)
                    s += Q[r * dk + c] * exp(G[r * dk + c]) * S[c * dv + v];
                for (int i = 0; i <= r; i++)
                    s += B[r * C + i] * D[i * dv + v];
                o[v] = s;
            }
        }
        /* step 8: S <- Diag(exp(G_last)) S0 + sum_i (k_i * exp(G_last - G_i)) Delta_i^T */
        const double *Gl = G + (size_t)(L - 1) * dk;
        for (int c = 0; c < dk; c++)
            for (int v = 0; v < dv; v++) {
                double s = exp(Gl[c]) * S[c * dv + v];
                for (int i = 0; i < L; i++)
                    s += K[i * dk + c] * exp(Gl[c] - G[i * dk + c]) * D[i * dv + v];
                Sn[c * dv + v] = s;
            }
        memcpy(S, Sn, sizeof(double) * dk * dv);
    }
    store_state(J, n, hs, S);
}

static size_t scratch_doubles(const job_t *J)
{
    size_t dk = J->dk, dv = J->dv, C = J->chunk;
    if (C == 0)
        return 3 * dk + 2 * dv;
    return C * dk * 4 + C * dv * 4 + C + C * C * 3 + dk * dv;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * J->dk * J->dv);
    double *buf = (double *)malloc(sizeof(double) * scratch_doubles(J));
    int total = J->N * J->nsel;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int w = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (w >= total)
            break;
        int n = w / J->nsel, hs = w % J->nsel;
        if (J->chunk == 0)
            run_recurrent(J, n, hs, S, buf);
        else
            run_chunked(J, n, hs, S, buf);
    }
    free(S);
    free(buf);
    return NULL;
}

static int check_args(const job_t *J)
{
    if (!J->q || !J->k || !J->v || !J->g || !J->beta || !J->cu || !J->out || !J->heads)
        return 1;
    if (J->N < 1 || J->T < 0 || J->H < 1 || J->dk < 1 || J->dv < 1 || J->nsel < 1 || J->chunk < 0)
        return 2;
    if (J->cu[0] != 0 || J->cu[J->N] != J->T)
        return 2;
    for (int n = 0; n < J->N; n++)
        if (J->cu[n + 1] < J->cu[n])
            return 2;
    for (int i = 0; i < J->nsel; i++)
        if (J->heads[i] < 0 || J->heads[i] >= J->H)
            return 2;
    return 0;
}

static int run_job(job_t *J)
{
    int rc = check_args(J);
    if (rc)
        return rc;
    int nt = J->nthreads < 1 ? 1 : J->nthreads;
    if (nt > J->N * J->nsel)
        nt = J->N * J->nsel;
    pthread_mutex_init(&J->mu, NULL);
    J->next = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    for (int i = 0; i < nt; i++)
        pthread_create(&th[i], NULL, worker, J);
    for (int i = 0; i < nt; i++)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->mu);
    return 0;
}

/*
 * Public entry points.  Return 0 on success, 1 for a NULL required pointer,
 * 2 for bad sizes or cu_seqlens.  The caller owns every buffer.
 */
int kda_oracle_recurrent(const void *q, const void *k, const void *v, int qkv_dtype,
                         const void *g, const void *beta, int gb_dtype,
                         const int32_t *cu_seqlens, const double *initial_state,
                         double *out, double *final_state,
                         int N, int T, int H, int dk, int dv,
                         const int32_t *heads, int nsel, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.qkv_dtype = qkv_dtype; J.gb_dtype = gb_dtype;
    J.cu = cu_seqlens; J.init = initial_state; J.out = out; J.fin = final_state;
    J.N = N; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.heads = heads; J.nsel = nsel; J.chunk = 0; J.nthreads = nthreads;
    return run_job(&J);
}

int kda_oracle_chunked(const void *q, const void *k, const void *v, int qkv_dtype,
                       const void *g, const void *beta, int gb_dtype,
                       const int32_t *cu_seqlens, const double *initial_state,
                       double *out, double *final_state,
                       int N, int T, int H, int dk, int dv,
                       const int32_t *heads, int nsel, int chunk, int nthreads)
{
    if (chunk < 1)
        return 2;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.qkv_dtype = qkv_dtype; J.gb_dtype = gb_dtype;
    J.cu = cu_seqlens; J.init = initial_state; J.out = out; J.fin = final_state;
    J.N = N; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.heads = heads; J.nsel = nsel; J.chunk = chunk; J.nthreads = nthreads;
    return run_job(&J);
}
