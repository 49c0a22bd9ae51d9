/*
 * synthetic_gen.c -- seeded, counter-based input generator for the KDA
 * workloads (host code, plain C11 + POSIX threads).
 *
 * It draws inputs only and holds none of the method's arithmetic; the CUDA
 * path and the CPU oracle both take their inputs from it.
 *
 * Element i of stream s under seed `seed` is mix64(mix64(seed) + s*2^48 + i),
 * where mix64 is the splitmix64 output function.  Uniforms use the top 53
 * bits, (x + 0.5) * 2^-53, so they lie in the open interval (0, 1).  Normal
 * deviates use Box-Muller (cosine branch) on the uniforms of indices 2i and
 * 2i + 1.  Every value depends only on its flat index in the full logical
 * tensor, so any row range or head subset can be drawn on its own.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline double uniform(uint64_t key, uint64_t stream, uint64_t i)
{
    uint64_t x = mix64(key + stream * (1ull << 48) + i);
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal(uint64_t key, uint64_t stream, uint64_t i)
{
    double u1 = uniform(key, stream, 2 * i), u2 = uniform(key, stream, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t b;
    memcpy(&b, &f, 4);
    return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

enum { KIND_Q = 0, KIND_K = 1, KIND_V = 2, KIND_G = 3, KIND_BETA = 4, KIND_STATE = 5 };
enum { OUT_BF16 = 0, OUT_F32 = 1 };

typedef struct {
    int kind, out_dtype, H, d, nh;
    uint64_t key;
    int64_t row_lo, nrows;
    const int32_t *heads;
    void *out;
    int64_t lo, hi;   /* this worker's slice of rows (or states) */
} task_t;

static void put(const task_t *t, size_t pos, double x)
{
    if (t->out_dtype == OUT_BF16)
        ((uint16_t *)t->out)[pos] = to_bf16(x);
    else
        ((float *)t->out)[pos] = (float)x;
}

static void *work(void *arg)
{
    const task_t *t = (const task_t *)arg;
    double buf[1024];
    for (int64_t r = t->lo; r < t->hi; r++) {
        for (int hs = 0; hs < t->nh; hs++) {
            uint64_t h = (uint64_t)t->heads[hs];
            if (t->kind == KIND_BETA) {
                uint64_t idx = (uint64_t)(t->row_lo + r) * t->H + h;
                double z = normal(t->key, 5, idx);
                ((float *)t->out)[(size_t)r * t->nh + hs] = (float)(1.0 / (1.0 + exp(-z)));
                continue;
            }
            if (t->kind == KIND_STATE) {
                /* r is the sequence index; d*d values in [dv][dk] order */
                uint64_t base = ((uint64_t)r * t->H + h) * (uint64_t)t->d * t->d;
                size_t pos = ((size_t)r * t->nh + hs) * (size_t)t->d * t->d;
                for (int i = 0; i < t->d * t->d; i++)
                    ((float *)t->out)[pos + i] = (float)(0.02 * normal(t->key, 6, base + i));
                continue;
            }
            uint64_t base = ((uint64_t)(t->row_lo + r) * t->H + h) * (uint64_t)t->d;
            size_t pos = ((size_t)r * t->nh + hs) * (size_t)t->d;
            if (t->kind == KIND_G) {
                for (int c = 0; c < t->d; c++)
                    ((float *)t->out)[pos + c] = (float)(-0.2 * uniform(t->key, 4, base + c));
                continue;
            }
            uint64_t stream = t->kind == KIND_Q ? 1 : (t->kind == KIND_K ? 2 : 3);
            double ss = 0.0;
            for (int c = 0; c < t->d; c++) {
                buf[c] = normal(t->key, stream, base + c);
                ss += buf[c] * buf[c];
            }
            double scale = (t->kind == KIND_V) ? 1.0 : 1.0 / sqrt(ss);
            for (int c = 0; c < t->d; c++)
                put(t, pos + c, buf[c] * scale);
        }
    }
    return NULL;
}

/*
 * Fill `out` with rows [row_lo, row_lo + nrows) of one input tensor, for the
 * heads listed in `heads` (nh of them, out of H): q, k, v are [nrows][nh][d]
 * (bf16 bits or fp32), g is [nrows][nh][d] fp32, beta is [nrows][nh] fp32.
 * For KIND_STATE, rows are sequences and out is [nrows][nh][d][d] fp32.
 * Returns 0, or 1 on bad arguments.
 */
int syn_fill(int kind, uint64_t seed, int64_t row_lo, int64_t nrows, const int32_t *heads, int nh,
             int H, int d, void *out, int out_dtype, int nthreads)
{
    if (!heads || !out || nh < 1 || H < 1 || d < 1 || d > 1024 || nrows < 0 || kind < 0 || kind > 5)
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;
    task_t *ts = (task_t *)calloc((size_t)nthreads, sizeof(task_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    uint64_t key = mix64((uint64_t)seed);
    for (int i = 0; i < nthreads; i++) {
        task_t t = {kind, out_dtype, H, d, nh, key, row_lo, nrows, heads, out,
                    nrows * i / nthreads, nrows * (i + 1) / nthreads};
        ts[i] = t;
        pthread_create(&th[i], NULL, work, &ts[i]);
    }
    for (int i = 0; i < nthreads; i++)
        pthread_join(th[i], NULL);
    free(ts);
    free(th);
    return 0;
}

/* Uniform deviates of stream `stream`, indices [0, n), as doubles. */
int syn_uniform(uint64_t seed, uint64_t stream, int64_t n, double *out)
{
    uint64_t key = mix64(seed);
    for (int64_t i = 0; i < n; i++)
        out[i] = uniform(key, stream, (uint64_t)i);
    return 0;
}
