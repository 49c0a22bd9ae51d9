// kda_tc.cu -- the fused tensor-core KDA chunked packed-varlen prefill for
// GB300 (sm_103a): one persistent kernel, TMA-staged tiles, tcgen05 MMAs with
// fp32 accumulators in TMEM, warp-specialised prep / chain / load roles.
//
// What one (sequence, head) "unit" computes, per 64-row chunk with L valid
// rows (KDA recurrence S_t = (I - b k k^T) Diag(exp(g_t)) S_{t-1} + b k v^T,
// o_t = S_t^T q_t, in the chunked WY form: cumulative log-decay G, strictly
// lower A_kk = beta_i (k_i * exp(G_i - G_j)) . k_j, the inverse of (I + A_kk),
// the factors W and U, the inter-chunk state recurrence, the outputs):
//
//   G_r  = sum_{u<=r} g_u,  m = (L-1)/2,  a_r = exp(G_r - G_m), b_r = 1/a_r
//   Kp = beta*K*a, Qp = Q*a, Km = K*b            (fp16, in shared memory)
//   [A_kk ; A_qk] = [Kp ; Qp] Km^T               MMA-a  (M=128, N=64, K=128)
//   T  = (I + strict(A_kk))^-1                   CUDA cores + warp MMA
//   W'^T = Kp^T T^T,  U^T = (beta*V)^T T^T       MMA-b  (M=128, N=64, K=64)
//   S' = Diag(exp(G_m)) S                        (state seen from row m)
//   [Delta^T | O^T] = [U^T | 0] + S'^T [-W' ; Qp]^T   MMA1 (one N=128 MMA, A = S'^T from TMEM)
//   O^T += Delta^T tril(A_qk)^T, S^T += Delta^T Km  MMA3 (one N=192 MMA over
//                                                [tril(A_qk)^T | Km]; the state stays fp32 in TMEM)
//   S   <- Diag(exp(G_{L-1} - G_m)) S            (applied at the next chunk start)
//
// Everything is kept "v-major" (TMEM lane = value channel v) so that every MMA
// has M = 128 and the state S^T = [dv][dk] lives in TMEM in exactly the
// layout of the [slot][head][v][k] state pool.  MMA operands are fp16 (fp32
// accumulate): bf16 operands would cost ~2e-3 relative error, fp16 costs
// ~2e-4; the midpoint reference m keeps every scaled operand within fp16 range
// for half-chunk log-decays above about -11.
//
// Roles (512 threads, 16 warps):
//   warps 0-3    chain: state rescaling and its fp16 copy, MMA1, the Delta
//                conversion, MMA3, output and final-state stores; its first
//                thread requests the k/q/v tiles and issues the chain MMAs;
//                warp 0 allocates TMEM
//   warps 4-11   group E: cumulative log-decay, decay-scaled operands, MMA-a,
//                beta*V; requests the next chunk's g and claims units
//   warps 12-15  group I: A readout, the 64x64 inverse (16x16 diagonal blocks
//                by forward substitution, block merges on the warp MMA), MMA-b,
//                -W' out of TMEM into the stage as MMA1's operand
// Two shared-memory stages let the prep of chunk c+1 overlap the chain of
// chunk c.  Every mbarrier wait is bounded; on timeout the kernel records
// kErrWaitTimeout in the device error word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

// Optional phase timestamps of CTA 0 (compiled in only with -DKDA_TRACE).
#ifdef KDA_TRACE
#ifndef KDA_TRACE_CTA
#define KDA_TRACE_CTA 0
#endif
__device__ unsigned long long g_kda_trace[3][128][16];
__device__ unsigned long long g_kda_cta[1024][4];   // per CTA: start, end (global timer), items, units
__device__ __forceinline__ unsigned long long kda_gtimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define KDA_PHASE(role, item, point)                                                  \
    do {                                                                              \
        if (blockIdx.x == KDA_TRACE_CTA && (item) < 128) g_kda_trace[role][item][point] = clock64(); \
    } while (0)
#else
#define KDA_PHASE(role, item, point) \
    do {                             \
    } while (0)
#endif

// Poll limit of the chain's wait for MMA1.  A test build of the library sets
// it to 0, so that the wait gives up at once although its MMA does complete:
// that drives the kernel through its timeout path (error bit, wind-down,
// TMEM freed after every MMA and copy in flight has landed) on the GPU.
#ifndef KDA_WAIT_LIMIT_MMA1
#define KDA_WAIT_LIMIT_MMA1 (1u << 18)
#endif

constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kChainThreads = 128;
constexpr int kEThreads = 256;                      // prep group E (warps 4-11)
constexpr int kGroupThreads = 128;                  // prep group I (warps 12-15)
constexpr int kBarChain = 1, kBarE = 2, kBarI = 3;   // named barriers
constexpr int kMaxSortedSeqs = 256;

// ---- shared memory map (bytes from a 1024-aligned base) ----------------------
// Two 72 KB stages hold what lives from a chunk's k/q/v loads until the chain's
// MMAs on it are done; g, T16 and group I's fp32 blocks are single shared
// buffers because only one chunk at a time uses them.
constexpr uint32_t kStageBytes = 73728;
// k and q: [kb][128 rows][64 channels], 2 x 16 KB, K rows first in stage 0 and
// Q rows first in stage 1 (so that MMA1's [Delta | O] output follows the TMEM
// order below); the K rows later hold -W' [r][c]
constexpr uint32_t kOffKQ = 0;
constexpr uint32_t kOffV = 32768;       // V (fp16 in place of bf16), 2 x 8 KB
// Km [kb][r][c] (2 x 8 KB) and tril(A_qk)^T [i][r] (8 KB): three 64-column
// blocks, adjacent in the order of the TMEM columns MMA3 accumulates into --
// stage 0 [tril(A_qk)^T | Km], stage 1 [Km | tril(A_qk)^T] -- so that MMA3 reads
// one N = 192 operand (MN-major) from here
constexpr uint32_t kOffMma3 = 49152;
__device__ __forceinline__ uint32_t off_k(int s) { return s ? 8192u : 0u; }        // K rows in a kb block
__device__ __forceinline__ uint32_t off_q(int s) { return s ? 0u : 8192u; }        // Q rows in a kb block
__device__ __forceinline__ uint32_t off_km(int s) { return s ? 49152u : 57344u; }   // Km
__device__ __forceinline__ uint32_t off_bq(int s) { return s ? 65536u : 49152u; }   // tril(A_qk)^T
// (the functions above take a layout bit lb: the stage index s in the fused
// kernel, whose chain merges its MMAs across the two layouts; in split mode
// the parity of the chunk's index in its sequence, so that a chain CTA sees
// the layouts alternate -- see layout_bit)
constexpr uint32_t kOffG = 2 * kStageBytes;     // g slot ([64][128] fp32, unswizzled), read once by the decay scan
constexpr uint32_t kOffT16 = kOffG + 32768;     // T = (I + A_kk)^-1 [r][j] fp16, 8 KB (MMA-b operand)
constexpr uint32_t kOffTmp = kOffT16 + 8192;    // group I fp32 blocks of the inverse, 16 KB
constexpr uint32_t kOffEScr = kOffTmp + 16384;  // group E scan exchange, 2 KB
constexpr uint32_t kOffP = kOffEScr + 2048;     // group I merge temporaries, 6 KB
constexpr uint32_t kOffConst = kOffP + 6144;    // per stage: fm[128] | unused | beta[64]
constexpr uint32_t kConstBytes = 1280;
constexpr uint32_t kOffGm = kOffConst + 2 * kConstBytes;   // G_m[128], G_last[128]
constexpr uint32_t kOffOrder = kOffGm + 1024;              // sorted order, then {bos, eos} per sequence
constexpr uint32_t kOffBar = kOffOrder + 12 * kMaxSortedSeqs;
constexpr uint32_t kOffMisc = kOffBar + 256;     // TMEM base, abort flag, schedule length, schedule
// pend = exp(G_last - G_m) of chunk i lives in slot i % 3: the chain reads it at
// the start of chunk i+1 (or at the end of the unit), and only chunk i+3's
// decay scan, which waits for chunk i+1's stage, can overwrite it.
constexpr uint32_t kOffPend = kOffMisc + 128;
// output rows 32-63 of a chunk, bf16 [2 channel blocks][32 rows][64], 128B-swizzled
// (rows 0-31 go to the stage's tril(A_qk) buffer, free once MMA3 is done)
constexpr uint32_t kOffOT = (kOffPend + 3 * 512 + 1023) & ~1023u;
constexpr uint32_t kSmemBytes = kOffOT + 8192 + 1024;   // + alignment slack

// ---- split mode: chunk preparation and the state chain on separate SMs ----
// For calls with few (sequence, head) units -- one long sequence, say -- one
// unit per SM leaves most SMs idle and each unit's chunks run one after
// another at the pace of a whole prep pipeline.  Only the state chain (the
// rescale, MMA1, Delta, MMA3, outputs) depends on the previous chunk; the
// decay scan, the operands, A, the inverse, W' and beta*V do not.  In split
// mode CTA b < chains runs the chain of unit b alone -- 16 compute warps, a
// loader warp and an MMA-issuer warp (576 threads for every CTA); with half
// chains, CTAs 2u and 2u + 1 each keep 64 of unit u's value channels -- and
// every other CTA prepares chunks -- any unit's, in the order (chunk index,
// unit) -- with the prep roles unchanged and ships each finished stage through
// a ring in global memory (kRingSlots slots per unit, in L2 in practice):
// producer and chain hand over through flags with release/acquire ordering.
constexpr int kSortChunks = 3;                          // the producers' deal: one chunk per claim
constexpr int kRingSlots = 4;
// each ring slot's two flags in cache lines of their own (128 B apart, the
// next slot 256 B on), so that the polling spreads over L2 (measured: with
// the flags packed together, long_65536 took 18 % longer in some runs)
constexpr int kFlagSlotStride = 64;                     // ints per ring slot: ready at +0, freed at +32
constexpr uint32_t kSlotT16 = kStageBytes;              // slot: the stage | T16 | fm, pend
constexpr uint32_t kSlotHdr = kStageBytes + 8192;
constexpr uint32_t kSlotBytes = kSlotHdr + 1024;
// the chain CTA's shared memory: two slot buffers, then two output staging
// buffers (16 KB each), then the
// pend of the last two chunks; barriers and misc at the usual offsets
constexpr uint32_t kCOut = 2 * kSlotBytes;
constexpr uint32_t kCPend = kCOut + 2 * 16384;
static_assert(kCPend + 1024 <= kOffOrder, "chain layout overlaps the unit table");

// mbarrier slots ([2] = one per stage)
constexpr int kBarKQFull = 0;      // [2]: k, q tiles landed
constexpr int kBarVFull = 2;       // [2]: v tile landed
constexpr int kBarPrepDone = 4;    // [2]: MMA-b of a chunk is done (W'^T and U^T in TMEM)
constexpr int kBarAFull = 6;       // [2]: MMA-a done
constexpr int kBarEDone = 8;       // [2]: group E has written a chunk's beta*V (256 arrivals; not with the fused prologue)
constexpr int kBarODone = 10;      // [2]: the chain has read a chunk's outputs (TMEM P_s free)
constexpr int kBarFmReady = 12;    // [2]: the chunk's decay constants are written (128 arrivals)
constexpr int kBarKmFree = 14;     // [2]: the chain's MMAs on the stage are done (Km, B free)
constexpr int kBarGFull = 16;      // g slot landed
constexpr int kBarMma1 = 18, kBarMma3 = 20, kBarDrain = 21;
constexpr int kBarWReady = 22;     // [2]: -W' is in the stage's K rows, TMEM output columns zeroed (128 arrivals)

// TMEM columns: [Delta_0 | O_0 | S | O_1 | Delta_1 | S'h | Delta h].  The O_s
// columns take A (MMA-a), then W'^T (MMA-b), then the outputs; Delta_s takes
// U^T (MMA-b), then Delta^T.  MMA1 writes [Delta_0 | O_0] or [O_1 | Delta_1]
// (N = 128), MMA3 [O_0 | S] or [S | O_1] (N = 192).
constexpr uint32_t kTmS = 128, kTmS0h = 384, kTmDh = 448, kTmCols = 512;
__device__ __forceinline__ uint32_t tm_o(int s) { return s ? 256u : 64u; }
__device__ __forceinline__ uint32_t tm_d(int s) { return s ? 320u : 0u; }

constexpr uint32_t kKQBytes = 4 * 8192;        // k and q tiles (bf16)
constexpr uint32_t kVBytes = 2 * 8192;         // v tile (bf16)
constexpr uint32_t kGBytes = 4 * 8192;         // g tile (fp32)

struct TcParams {
    const int32_t *cu;
    const float *beta;
    const float *s0;
    __nv_bfloat16 *out;
    float *s1;
    int N, T, H;
    const int *g_order;
    const int2 *g_rows;
    const int *g_une;
    int *err;
    unsigned int *sched;   // dynamic deal: [claim counter, finished CTAs], or nullptr
    const int *slots;      // [N] state-pool entry of each sequence (-1: padding), or nullptr (entry n)
    int num_slots;         // entries in the state pool when slots is set
};

// The fused short-conv prologue's arguments (read by kConv builds only; a
// separate kernel argument, so that the other builds' parameters and code
// stay as they are).  The tensor maps then read the raw projections.
struct ConvParams {
    const uint16_t *x[3];  // x_q, x_k, x_v [T][H][128] bf16, for the rows before a chunk
    const float *w;        // [3][H*128][4] fp32 (stream, channel, tap)
    uint16_t *pool;        // [entries][3 taps][3 streams][H*128] bf16, the windows, updated in place
    int H;
    int act;               // 0 identity, 1 SiLU
    float eps;
};

// Split mode's hand-over (zeroed by the host before each launch).
struct SplitParams {
    uint8_t *ring;         // [units][kRingSlots][kSlotBytes]
    int *ready;            // per slot (stride kFlagSlotStride): 2 (j + 1) + layout bit once chunk j is in the slot
    int *freed;            // per slot (stride kFlagSlotStride): j + 1 once the chain is done with chunk j
                           // (half chains: +1 from each of the two for every chunk of the slot)
    int *abort;            // set by a CTA whose wait on another CTA ran out
    int chains;            // CTAs 0 .. chains-1 run the chains, one unit (or half unit) each, in sorted order
};

struct Smem {
    uint8_t *base;
    __device__ uint32_t u32(uint32_t off) const { return smem_u32(base + off); }
    template <typename T> __device__ T *ptr(uint32_t off) const { return reinterpret_cast<T *>(base + off); }
    __device__ uint32_t bar(int i) const { return u32(kOffBar + 8 * i); }
    __device__ volatile int *abort_flag() const { return ptr<volatile int>(kOffMisc + 4); }
    __device__ uint32_t *tmem_base() const { return ptr<uint32_t>(kOffMisc); }
    // dynamic unit deal
    __device__ volatile int *published() const { return ptr<volatile int>(kOffMisc + 12); }   // dynamic: units in the ring
    __device__ volatile int *claim_done() const { return ptr<volatile int>(kOffMisc + 16); }  // dynamic: no more claims
    __device__ int *units_nonempty() const { return ptr<int>(kOffMisc + 20); }
    __device__ int *sched() const { return ptr<int>(kOffMisc + 24); }      // ring [8] of claimed units
    __device__ int *split_parity() const { return ptr<int>(kOffMisc + 56); }   // split chain: [2] per buffer
    __device__ int *producers() const { return ptr<int>(kOffMisc + 64); }      // split: producer CTAs
};

__device__ __forceinline__ bool role_any(bool pred, int id, int n)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// State-pool entry of sequence n: n itself, or its id in the slot table.  A
// padded sequence (id -1) has none, and neither has an id outside
// [-1, num_slots), which is also reported; such a sequence is skipped.  The
// kernel is built twice, with and without the slot table, so that the dense
// form carries none of this code.
template <bool kSlots>
__device__ __forceinline__ int state_index(const TcParams &p, int n)
{
    if (!kSlots) return n;
    const int s = __ldg(p.slots + n);
    if (s >= 0 && s < p.num_slots) return s;
    if (s != -1) atomicOr(p.err, kErrBadSlot);
    return -1;
}

// Unit u (in this CTA's schedule order) -> (sequence, head, rows, state entry).
struct Unit {
    int n, h, bos, eos, nchunks, st;
};

template <bool kSlots, int kSort>
__device__ __forceinline__ Unit get_unit(const TcParams &p, const int *order, int u)
{
    Unit x;
    const int su = u / p.H;
    x.h = u % p.H;
    int b, e;
    if constexpr (kSort == kSortChunks) {
        // a producer's claim: chunk j of unit uu (sorted order), packed (j << 8) | uu
        const int j = u >> 8, uu = u & 255;
        x.n = order[uu / p.H];
        x.h = uu % p.H;
        const int2 be = reinterpret_cast<const int2 *>(order + kMaxSortedSeqs)[x.n];
        x.bos = be.x + kChunk * j;
        x.eos = min(x.bos + kChunk, be.y);
        x.nchunks = 1;
        x.st = -1;   // producers touch no state
        return x;
    } else if constexpr (kSort == 1) {
        // order[] is followed in shared memory by the clamped {bos, eos} rows
        x.n = order[su];
        const int2 be = reinterpret_cast<const int2 *>(order + kMaxSortedSeqs)[x.n];
        b = be.x;
        e = be.y;
    } else if constexpr (kSort == 2) {
        x.n = p.g_order[su];
        const int2 be = p.g_rows[x.n];
        b = be.x;
        e = be.y;
    } else {
        x.n = su;
        b = min(max(p.cu[x.n], 0), p.T);
        e = min(max(p.cu[x.n + 1], 0), p.T);
    }
    x.st = state_index<kSlots>(p, x.n);
    if (e < b || (kSlots && x.st < 0)) e = b;
    x.bos = b;
    x.eos = e;
    x.nchunks = (e - b + kChunk - 1) / kChunk;
    return x;
}

// Layout bit of a stage (off_k etc.): the stage index s, or for a split-mode
// producer the parity of the chunk's index in its sequence
template <int kSort>
__device__ __forceinline__ int layout_bit(const int *order, const Unit &un, int s)
{
    if constexpr (kSort == kSortChunks) {
        const int2 be = reinterpret_cast<const int2 *>(order + kMaxSortedSeqs)[un.n];
        return ((un.bos - be.x) / kChunk) & 1;
    } else {
        return s;
    }
}

// Dynamic deal: unit k of this CTA once group E's first thread has published
// it (units are claimed one ahead of the furthest loader); after the last
// claim, the CTA's share of the empty units (dealt round-robin) follows.
__device__ __noinline__ int dyn_unit(const Smem &sm, int k, int U)
{
    for (uint32_t it = 0; it < (1u << 22); it++) {
        const int pub = *sm.published();
        __threadfence_block();
        if (k < pub) return reinterpret_cast<volatile int *>(sm.sched())[k & 7];
        if (*sm.claim_done()) {
            const int u = *sm.units_nonempty() + (int)blockIdx.x + (k - pub) * (int)gridDim.x;
            return u < U ? u : -1;
        }
        if (*sm.abort_flag()) return -1;
        __nanosleep(64);
    }
    *sm.abort_flag() = 1;
    return -1;
}

// k-th unit of this CTA, -1 when exhausted: the dynamic deal of the
// length-sorted units, or (unsorted) a boustrophedon ("snake") deal over the grid.
template <int kSort>
__device__ __forceinline__ int cta_unit(const Smem &sm, int k, int U)
{
    if constexpr (kSort != 0) {
        return dyn_unit(sm, k, kSort == kSortChunks ? 0 : U);   // producers get no empty units
    } else {
        const int G = gridDim.x, b = blockIdx.x;
        const int u = k * G + ((k & 1) ? (G - 1 - b) : b);
        return u < U ? u : -1;
    }
}


// The producers' claims, in order: claim i is chunk j of unit u, where the
// chunks are counted by index j first and then by unit (sorted order, so the
// units that still have a chunk j are the first cnt(j) = H * (sequences with
// more than j chunks)).  A producer's claims only grow, so a cursor over j
// decodes them.
struct ChunkDeal {
    int j = 0, base = 0;   // chunks of index < j
    int m = -1;            // sequences (sorted) with more than j chunks
    __device__ int decode(const int *order, int N, int H, int i)
    {
        const int2 *rows = reinterpret_cast<const int2 *>(order + kMaxSortedSeqs);
        auto nch = [&](int su) { const int2 be = rows[order[su]]; return (be.y - be.x + kChunk - 1) / kChunk; };
        if (m < 0) {
            m = N;
            while (m > 0 && nch(m - 1) <= 0) m--;
        }
        while (i >= base + H * m) {
            base += H * m;
            j++;
            while (m > 0 && nch(m - 1) <= j) m--;
        }
        return (j << 8) | (i - base);
    }
};

// k-th unit of this CTA if it is already known (-1: exhausted, -2: not yet
// claimed); never waits.
template <int kSort>
__device__ __forceinline__ int cta_unit_peek(const Smem &sm, int k, int U)
{
    if constexpr (kSort == 0) return cta_unit<kSort>(sm, k, U);
    const int pub = *sm.published();
    __threadfence_block();
    if (k < pub) return reinterpret_cast<volatile int *>(sm.sched())[k & 7];
    if (!*sm.claim_done()) return -2;
    const int u = *sm.units_nonempty() + (int)blockIdx.x + (k - pub) * (int)gridDim.x;
    return u < U ? u : -1;
}

// byte offset of 16-byte chunk `ch` of row `r` in a 128B-swizzled tile
__device__ __forceinline__ uint32_t sw128_chunk(int r, int ch) { return r * 128 + ((ch ^ (r & 7)) << 4); }

// Two fp32 operations in one instruction on a register pair (mul / sub / add
// .rn.f32x2, sm_100 and later): each half is the IEEE single-precision
// operation rounded to nearest even, so the results are the scalar ones, for
// half the instructions on the issue slots the roles of a CTA share.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mul.rn.f32x2 x, x, y;\n mov.b64 {%0, %1}, x;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n sub.rn.f32x2 x, x, y;\n mov.b64 {%0, %1}, x;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n add.rn.f32x2 x, x, y;\n mov.b64 {%0, %1}, x;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 2^x on the special-function unit (approximate, subnormal results flushed to
// zero).  The decay pass keeps its log-decays in base 2: exp(G) = 2^(G log2 e).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;   // 1 / ln 2
// Largest |G_r - G_m| (base 2) of a chunk's operand factors.  At 2^15 an
// operand beta*k*a stays below fp16's largest value 65504 for |beta k| <= 1,
// and a factor of 2^-15 keeps a typical |k| ~ 2^-3.5 at 2^-18.5, whose fp16
// subnormal still carries ~6 significant bits in the few products that pair
// it with a factor of 2^15.
constexpr float kMaxFactorLog2 = 15.f;

__device__ __forceinline__ void record_error(const TcParams &p, const Smem &sm, int code)
{
    atomicOr(p.err, code);
    *sm.abort_flag() = 1;
}

// ---- small products on the warp MMA (tf32) ------------------------------------------
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d += A[16x8] * B[8x8] with both operands rounded to tf32 (10-bit mantissa,
// the precision of the fp16 operand T16 the merged blocks end up in)
__device__ __forceinline__ void mma_1xtf32(float (&d)[4], const float (&a)[4], const float (&b)[2])
{
    const uint32_t ah[4] = {to_tf32(a[0]), to_tf32(a[1]), to_tf32(a[2]), to_tf32(a[3])};
    const uint32_t bh[2] = {to_tf32(b[0]), to_tf32(b[1])};
    mma_tf32(d, ah, bh);
}

// One m16n8 tile of D = sum_k A[r0 + .][ka + k] * B[kb + k][c0 + .] over k-steps
// [ks0, ks1) of 8, A and B read from fp32 smem through `la` / `lb` (row, col)
// index functions; tf32 on the warp MMA.
template <typename FA, typename FB>
__device__ __forceinline__ void tile_mma(float (&d)[4], FA la, FB lb, int ks0, int ks1, int lane)
{
    const int g = lane >> 2, t = lane & 3;
    for (int ks = ks0; ks < ks1; ks++) {
        const float a[4] = {la(g, 8 * ks + t), la(g + 8, 8 * ks + t), la(g, 8 * ks + t + 4), la(g + 8, 8 * ks + t + 4)};
        const float b[2] = {lb(8 * ks + t, g), lb(8 * ks + t + 4, g)};
        mma_1xtf32(d, a, b);
    }
}

// =============================================================================
// TMA loads.  The chain's elected thread loads k, q and v into the stages (the
// first two chunks at the start, then chunk i+2 as soon as chunk i has released
// the regions: v once MMA-b is done, k and q once MMA1 is done); group E's
// first thread loads g into the single g slot as soon as the operand pass has
// read the previous chunk's G.
// =============================================================================
struct Maps {
    const CUtensorMap *q, *k, *v, *g, *o;
};

// Walks this CTA's chunks in schedule order.
struct LoadCursor {
    int k = -1, c = 0, item = 0;
    bool done = false;
    Unit un = {0, 0, 0, 0, 0};
    int row0 = 0;
};

// Advances to the next chunk (its coordinates: row0, un.h; its index: item - 1);
// false when the schedule is exhausted.
template <bool kSlots, int kSort>
__device__ bool cursor_next(LoadCursor &L, const TcParams &p, const Smem &sm, const int *order, int U)
{
    while (!L.done && L.c >= L.un.nchunks) {
        const int u = cta_unit<kSort>(sm, ++L.k, U);
        if (u < 0) {
            L.done = true;
            break;
        }
        L.un = get_unit<kSlots, kSort>(p, order, u);
        L.c = 0;
    }
    if (L.done) return false;
    L.row0 = L.un.bos + L.c * kChunk;
    L.c++;
    L.item++;
    return true;
}

// k and q of chunk `item`: one 3-D box per 64-channel half (the halves of k and
// q interleave in shared memory)
__device__ void issue_kq(const Smem &sm, const Maps &m, int item, int row0, int h, int lb)
{
    const uint32_t st = sm.u32((item & 1) * kStageBytes);
    const uint32_t bar = sm.bar(kBarKQFull + (item & 1));
    KDA_PHASE(2, item, 0);
    mbar_arrive_expect_tx(bar, kKQBytes);
    for (int kb = 0; kb < 2; kb++) {
        tma_load_3d(st + kOffKQ + kb * 16384 + off_k(lb), m.k, 64 * kb, h, row0, bar);
        tma_load_3d(st + kOffKQ + kb * 16384 + off_q(lb), m.q, 64 * kb, h, row0, bar);
    }
}

// v of chunk `item`: one 4-D box, channel blocks outermost
__device__ void issue_v(const Smem &sm, const Maps &m, int item, int row0, int h)
{
    const uint32_t bar = sm.bar(kBarVFull + (item & 1));
    mbar_arrive_expect_tx(bar, kVBytes);
    tma_load_4d(sm.u32((item & 1) * kStageBytes + kOffV), m.v, 0, row0, 0, h, bar);
}

// g of the next chunk into the g slot: one 3-D box, each row's 512 bytes
// contiguous in memory and in the slot (measured: 1.3 % faster than four
// 128-byte swizzled channel blocks, which fetch every row in four passes)
__device__ void issue_g(const Smem &sm, const Maps &m, int row0, int h)
{
    const uint32_t bar = sm.bar(kBarGFull);
    mbar_arrive_expect_tx(bar, kGBytes);
    tma_load_3d(sm.u32(kOffG), m.g, 0, h, row0, bar);
}

// =============================================================================
// prep, group E (warps 4-11): cumulative log-decay, the decay-scaled operands,
// MMA-a and beta*V.  Loops are kept rolled: each warp runs its loop bodies
// once per chunk next to two other roles, so compact code matters more than
// unrolling.
// =============================================================================

// -----------------------------------------------------------------------------
// The fused short-conv prologue (kConv builds).  The stage's raw projection
// tiles become q, k and v in place: group E converts q and k before its
// operand pass, group I the value rows (straight to beta*V, i_conv_v) before
// it takes the chunk; q, k and v never reach global memory.  Per row t of a
// sequence and channel c, with x_{-3..-1} the window's taps:
// y_t = sum_j w_j x_{t-3+j}, SiLU if asked, and q, k scaled to unit L2 norm
// over the head's 128 channels, y / sqrt(|y|^2 + eps).
// -----------------------------------------------------------------------------
// SiLU(a) = a sigmoid(a) = a / (1 + 2^(-a log2 e)); ex2.approx and the
// approximate division keep it to a few units of fp32 rounding
__device__ __forceinline__ float conv_silu(float a) { return __fdividef(a, 1.f + ex2(-a * kLog2e)); }

// One stream over rows 8w .. 8w+7 of the chunk (w: the group E warp) and this
// lane's channels 4l .. 4l+3 of the head, in place in the stage tile whose two
// 64-channel blocks are `blk` apart from `tile` (bf16 in and out; rows at and
// past L become zero); with kNorm each row is scaled to unit L2 norm over the
// head's 128 channels -- the 32 lanes of the warp hold all of them, so the sum
// needs no other warp.  halo[j]: row 8w - 3 + j of the chunk (for warp 0 the
// sequence's previous rows, or its window's taps on its first chunk); a warp
// reads from the tile only the rows it rewrites, so the warps need no barrier
// here.  win (only on a sequence's last chunk): tap 0 of the stream's window
// at this lane's channels, taps tap_stride apart; it receives the last three
// raw rows of [old taps ; the sequence's rows] (warp 0 read the old taps into
// its halo before the decay pass's barriers).
template <bool kNorm>
__device__ void e_conv_stream(uint8_t *tile, uint32_t blk, const uint2 (&halo)[3], const float (&w)[4][4], int L,
                              int et, int act, float eps, uint16_t *win, size_t tap_stride)
{
    const int lane = et & 31, w8 = et >> 5;
    uint8_t *base = tile + (lane >> 4) * blk + 8 * (lane & 1);
    const int ch = (lane & 15) >> 1;                   // 16-byte chunk of channel 4l in its block row
    uint2 raw[11];                                     // rows 8w - 3 .. 8w + 7
#pragma unroll
    for (int j = 0; j < 3; j++) raw[j] = halo[j];
#pragma unroll
    for (int t = 0; t < 8; t++) raw[3 + t] = *reinterpret_cast<const uint2 *>(base + sw128_chunk(8 * w8 + t, ch));
    if (win) {
#pragma unroll 1
        for (int j = 0; j < 3; j++) {
            const int r = L - 3 + j;                     // chunk row of new tap j (< 0: in the halo)
            if ((r >= 0 ? (r >> 3) : 0) == w8) {
                const int idx = 3 + r - 8 * w8;
                uint2 val = make_uint2(0u, 0u);
#pragma unroll
                for (int i = 0; i < 11; i++) val = i == idx ? raw[i] : val;
                *reinterpret_cast<uint2 *>(win + j * tap_stride) = val;
            }
        }
    }
    float y[8][4];
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const float x[4][4] = {{bf16lo(raw[t].x), bf16hi(raw[t].x), bf16lo(raw[t].y), bf16hi(raw[t].y)},
                               {bf16lo(raw[t + 1].x), bf16hi(raw[t + 1].x), bf16lo(raw[t + 1].y), bf16hi(raw[t + 1].y)},
                               {bf16lo(raw[t + 2].x), bf16hi(raw[t + 2].x), bf16lo(raw[t + 2].y), bf16hi(raw[t + 2].y)},
                               {bf16lo(raw[t + 3].x), bf16hi(raw[t + 3].x), bf16lo(raw[t + 3].y), bf16hi(raw[t + 3].y)}};
#pragma unroll
        for (int c = 0; c < 4; c++) {                 // tap j weighs row t - 3 + j; the order of the sum is the prologue's
            float a = w[c][0] * x[0][c];
            a = fmaf(w[c][1], x[1][c], a);
            a = fmaf(w[c][2], x[2][c], a);
            a = fmaf(w[c][3], x[3][c], a);
            y[t][c] = act ? conv_silu(a) : a;
        }
    }
    if constexpr (kNorm) {
        // the 8 rows' squared norms: a reduce-scatter over the warp leaves lane l
        // with row l/4 (9 shuffles), then each row's total comes back by shuffle
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; t++) {
            v[t] = y[t][0] * y[t][0];
            v[t] = fmaf(y[t][1], y[t][1], v[t]);
            v[t] = fmaf(y[t][2], y[t][2], v[t]);
            v[t] = fmaf(y[t][3], y[t][3], v[t]);
        }
        float a4[4], a2[2];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const bool up = lane & 16;
            a4[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, up ? v[i] : v[i + 4], 16);
        }
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const bool up = lane & 8;
            a2[i] = (up ? a4[i + 2] : a4[i]) + __shfl_xor_sync(0xffffffffu, up ? a4[i] : a4[i + 2], 8);
        }
        const bool up = lane & 4;
        float tot = (up ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, up ? a2[0] : a2[1], 4);
        tot += __shfl_xor_sync(0xffffffffu, tot, 2);
        tot += __shfl_xor_sync(0xffffffffu, tot, 1);       // lane l: row l/4, all 128 channels
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const float sc = rsqrtf(__shfl_sync(0xffffffffu, tot, 4 * t) + eps);
#pragma unroll
            for (int c = 0; c < 4; c++) y[t][c] *= sc;
        }
    }
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const bool in = 8 * w8 + t < L;
        const uint2 out = in ? make_uint2(pack_bf16x2(y[t][0], y[t][1]), pack_bf16x2(y[t][2], y[t][3]))
                             : make_uint2(0u, 0u);
        *reinterpret_cast<uint2 *>(base + sw128_chunk(8 * w8 + t, ch)) = out;
    }
}

// the three rows before a group E warp's first row, per stream (q, k), at a
// lane's four channels; nothing in builds without the prologue
template <bool kConv> struct ConvHalo {
    uint2 r[2][3] = {};
};
template <> struct ConvHalo<false> {};

// where a group E lane's four channels (4l .. 4l+3 of the head) of a unit's
// window live: tap = the distance between taps, and the window of stream s on
// the unit's last chunk (null on the others)
struct ConvAt {
    uint16_t *base;   // tap 0, stream 0 at this lane's channels, or null
    size_t tap, stream;
    int c0;
    __device__ uint16_t *window(int s) const { return base ? base + s * stream : nullptr; }
};
__device__ __forceinline__ ConvAt conv_at(const ConvParams &cp, const Unit &un, int c, int et)
{
    ConvAt a;
    const size_t HC = (size_t)cp.H * kD;
    a.c0 = 4 * (et & 31);
    a.tap = 3 * HC;
    a.stream = HC;
    a.base = c == un.nchunks - 1 ? cp.pool + (size_t)un.st * 9 * HC + (size_t)un.h * kD + a.c0 : nullptr;
    return a;
}

// conv weights of stream s at channels h*128 + c0 .. + 3
__device__ __forceinline__ void conv_weights(const ConvParams &cp, int s, int h, int c0, float (&w)[4][4])
{
    const float4 *src = reinterpret_cast<const float4 *>(cp.w + ((size_t)s * cp.H * kD + (size_t)h * kD + c0) * 4);
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const float4 a = __ldg(src + c);
        w[c][0] = a.x; w[c][1] = a.y; w[c][2] = a.z; w[c][3] = a.w;
    }
}

// Group E's decay pass over one chunk (256 threads); `beta_r` is the beta of
// row et (zero past the chunk), loaded a chunk ahead.  Thread = (row group
// ew: rows 16*ew .. +15) x (channel half chh) x (key channels c0 = 64*chh +
// 2*lane, +1).  The row prefix of g * log2(e) runs in registers and the four
// row groups exchange their totals once; from then on the g slot is no longer
// read (`released` runs: the next chunk's g may be requested) and G, in base
// 2, stays in registers.  With G_m the G of the middle row m, Kp = beta*K*
// 2^(G - G_m), Qp = Q*2^(G - G_m) and Km = K*2^(G_m - G) become fp16 in place
// over the bf16 tiles (rows past the chunk zero).  Returns false if a wait ran
// out.
template <class F, class V, class C>
__device__ bool e_pass(const Smem &sm, int s, int lb, int item, int L, int et, float beta_r, int *err, F &&released,
                       V &&before_kq, C &&conv_qk)
{
    const int lane = et & 31;
    const uint32_t st = s * kStageBytes;
    float *cst = sm.ptr<float>(kOffConst + s * kConstBytes);
    float *gmx = sm.ptr<float>(kOffGm), *glx = gmx + 128;
    const int m = (L - 1) >> 1;
    const int ew = (et >> 5) & 3, chh = et >> 7;
    const int c0 = 64 * chh + 2 * lane;                      // this thread's two channels
    float *xchg = sm.ptr<float>(kOffEScr);                   // [4 row groups][128 channels]
    float2 x[16];
    {
        const uint8_t *gb = sm.base + kOffG + 4 * c0;    // [64 rows][128 channels], rows 512 B apart
#pragma unroll
        for (int t = 0; t < 16; t++) {
            const int r = 16 * ew + t;
            const float2 g2 = r < L ? *reinterpret_cast<const float2 *>(gb + 512 * r) : make_float2(0.f, 0.f);
            x[t] = fmul2(g2, make_float2(kLog2e, kLog2e));   // base-2 log-decay
        }
    }
#pragma unroll
    for (int t = 1; t < 16; t++) x[t] = fadd2(x[t], x[t - 1]);
    *reinterpret_cast<float2 *>(xchg + ew * 128 + c0) = x[15];
    fence_proxy_async_smem();   // the reads of the g slot come before a load that overwrites it
    named_bar(kBarE, kEThreads);
    released();
    float2 pre = make_float2(0.f, 0.f);
    for (int w = 0; w < ew; w++) {
        const float2 y = *reinterpret_cast<const float2 *>(xchg + w * 128 + c0);
        pre.x += y.x; pre.y += y.y;
    }
#pragma unroll
    for (int t = 0; t < 16; t++) {
        x[t] = fadd2(x[t], pre);
        const int r = 16 * ew + t;
        if (r == m) *reinterpret_cast<float2 *>(gmx + c0) = x[t];
        if (r == L - 1) *reinterpret_cast<float2 *>(glx + c0) = x[t];
    }
    if (et < kChunk) cst[256 + et] = beta_r;
    named_bar(kBarE, kEThreads);
    if (!before_kq()) return false;
    // k and q of this chunk have landed -- so the chain is past its MMA1 of chunk
    // item-2 and no longer reads that chunk's fm or pend slot -- and Km of chunk
    // item-2 is no longer read
    if (et == 0) KDA_PHASE(0, item, 15);
    bool ok = mbar_wait(sm.bar(kBarKQFull + s), (item >> 1) & 1, sm.abort_flag());
    if (ok && item >= 2) ok = mbar_wait(sm.bar(kBarKmFree + s), ((item >> 1) - 1) & 1, sm.abort_flag());
    if (role_any(!ok, kBarE, kEThreads)) return false;
    if (et == 0) KDA_PHASE(0, item, 14);
    conv_qk();        // the fused prologue's q and k (nothing in other builds)
    if (et < 128) {   // chain constants, one thread per key channel
        cst[et] = ex2(gmx[et]);                                                  // view from row m
        sm.ptr<float>(kOffPend)[(item % 3) * 128 + et] = ex2(glx[et] - gmx[et]);  // row m -> last row
        mbar_arrive(sm.bar(kBarFmReady + s));
    }
    if (et == 0) KDA_PHASE(0, item, 10);
    const float2 gm = *reinterpret_cast<const float2 *>(gmx + c0);
    float worst = 0.f;   // largest |G_r - G_m| of this thread's rows r < L
    uint8_t *kt = sm.base + st + kOffKQ + chh * 16384 + off_k(lb);   // this channel half's 64-channel block
    uint8_t *qt = sm.base + st + kOffKQ + chh * 16384 + off_q(lb);
    uint8_t *kmt = sm.base + st + off_km(lb) + chh * 8192;
    const int jk = lane >> 2;                            // 16-byte chunk of channel c0 in the row
    const uint32_t cb = 4 * (lane & 3);                  // byte of channel c0 in that chunk
#pragma unroll 1
    for (int half = 0; half < 2; half++) {
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const int r = 16 * ew + 8 * half + t;
            const uint32_t off = sw128_chunk(r, jk) + cb;
            const uint32_t kw = *reinterpret_cast<const uint32_t *>(kt + off);
            const uint32_t qw = *reinterpret_cast<const uint32_t *>(qt + off);
            const float br = cst[256 + r];               // zero past the chunk
            float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
            if (r < L) {
                const float2 d = fsub2(x[t], gm);
                a.x = ex2(d.x);
                a.y = ex2(d.y);
                b.x = ex2(-d.x);
                b.y = ex2(-d.y);
                worst = fmaxf(worst, fmaxf(fabsf(d.x), fabsf(d.y)));
            }
            const float2 kk = make_float2(bf16lo(kw), bf16hi(kw));
            const float2 qq = make_float2(bf16lo(qw), bf16hi(qw));
            const float2 kp = fmul2(kk, fmul2(a, make_float2(br, br)));
            const float2 qp = fmul2(qq, a), km = fmul2(kk, b);
            *reinterpret_cast<uint32_t *>(kt + off) = pack_f16x2(kp.x, kp.y);
            *reinterpret_cast<uint32_t *>(qt + off) = pack_f16x2(qp.x, qp.y);
            *reinterpret_cast<uint32_t *>(kmt + off) = pack_f16x2(km.x, km.y);
        }
#pragma unroll
        for (int t = 0; t < 8; t++) x[t] = x[t + 8];
    }
    // every factor 2^(G_r - G_m) must lie in [2^-kMaxFactorLog2, 2^kMaxFactorLog2]:
    // beyond it the fp16 operands overflow or lose their precision, and the
    // chunk is reported (its results are not to be used)
    if (worst > kMaxFactorLog2) atomicOr(err, kErrDecayRange);
    if (et == 0) KDA_PHASE(0, item, 11);
    return true;
}

// value tile bf16 -> beta_r * v as fp16, in place; rows past the chunk become zero
__device__ void e_convert_v(const Smem &sm, int s, int L, int et)
{
    uint8_t *vt = sm.base + s * kStageBytes + kOffV;
    const float *bt = sm.ptr<float>(kOffConst + s * kConstBytes) + 256;
#pragma unroll 1
    for (int i = 0; i < 4; i++) {
        const int idx = et + kEThreads * i;        // 16-byte chunk index in the 16 KB tile
        const int r = (idx >> 3) & 63;
        uint4 *ptr = reinterpret_cast<uint4 *>(vt + idx * 16);
        const uint4 w = *ptr;
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
        const float br = bt[r];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float2 y = fmul2(make_float2(bf16lo(in[e]), bf16hi(in[e])), make_float2(br, br));
            o[e] = r < L ? pack_f16x2(y.x, y.y) : 0u;
        }
        *ptr = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// (unrolled, unlike the other issue loops: group E, which issues it, sets the
// cadence, and the unrolled issue is faster; measured)
__device__ void issue_mma_a(const Smem &sm, int s, int lb, uint32_t tmem)
{
    const uint32_t st = sm.u32(s * kStageBytes);
    const uint32_t id = idesc_f16(128, 64, 0, 0);
#pragma unroll
    for (int ks = 0; ks < 8; ks++) {
        const int kb = ks >> 2, kin = ks & 3;
        const uint64_t ad = smem_desc_sw128(st + kOffKQ + kb * 16384 + kin * 32, 16, 1024);
        const uint64_t bd = smem_desc_sw128(st + off_km(lb) + kb * 8192 + kin * 32, 16, 1024);
        mma_ss(tmem + tm_o(s), ad, bd, id, ks > 0);
    }
}

__device__ __forceinline__ float load_beta(const TcParams &p, const LoadCursor &c, int et)
{
    const int L = min(kChunk, c.un.eos - c.row0);
    return et < L ? __ldg(p.beta + (size_t)(c.row0 + et) * p.H + c.un.h) : 0.f;
}

template <bool kSlots, int kSort, bool kConv>
__device__ void e_role(const TcParams &p, const ConvParams &cp, const Smem &sm, const int *order, int U,
                       const Maps &maps)
{
    const int et = threadIdx.x - kChainThreads;
    const uint32_t tmem = *sm.tmem_base();
    // g and the betas run one chunk ahead: `ahead` is the chunk whose g is in
    // flight (every thread walks it; thread 0 issues the load)
    LoadCursor ahead;
    float beta_next = 0.f;
    // dynamic deal: when the g loads reach the last chunk of a unit, thread 0
    // claims the next unit, and publishes the claim (to the ring in shared
    // memory) one step later -- late enough that a CTA only takes more work
    // when it is about to run out, early enough to hide the atomic's latency
    constexpr bool dyn = kSort != 0;
    unsigned claim = 0;
    int claim_slot = -1;
    ChunkDeal deal;   // split mode's producers: claims -> chunks
    auto publish = [&]() {
        if (claim_slot >= 0) {
            int u = (int)gridDim.x + (int)claim;
            bool more = u < *sm.units_nonempty();
            if constexpr (kSort == kSortChunks) {
                const int i = *sm.producers() + (int)claim;
                more = i < *sm.units_nonempty();
                if (more) u = deal.decode(order, p.N, p.H, i);
            }
            if (more) {
                reinterpret_cast<volatile int *>(sm.sched())[claim_slot & 7] = u;
                __threadfence_block();
                *sm.published() = claim_slot + 1;
            } else {
                __threadfence_block();
                *sm.claim_done() = 1;
            }
            claim_slot = -1;
        }
    };
    auto maybe_claim = [&](int k) {   // the g loads have just reached the last chunk of unit k
        if (dyn && et == 0 && claim_slot < 0 && !*sm.claim_done() && *sm.published() == k + 1) {
            claim = atomicAdd(p.sched, 1u);
            claim_slot = k + 1;
        }
    };
    if (cursor_next<kSlots, kSort>(ahead, p, sm, order, U)) {
        if (ahead.c == ahead.un.nchunks) maybe_claim(ahead.k);
        if (et == 0) {
            KDA_PHASE(2, 0, 1);
            issue_g(sm, maps, ahead.row0, ahead.un.h);
        }
        beta_next = load_beta(p, ahead, et);
    }
    int item = 0;
    // after a wait ran out: the g load in flight (chunk ahead.item - 1, one past
    // the last chunk whose g was waited for) lands before the role returns
    auto drain_g = [&]() {
        if (et == 0 && ahead.item > item) mbar_wait_drain(sm.bar(kBarGFull), (ahead.item - 1) & 1);
    };
    for (int k = 0;; k++) {
        const int u = cta_unit<kSort>(sm, k, U);
        if (u < 0) break;
        const Unit un = get_unit<kSlots, kSort>(p, order, u);
        for (int c = 0; c < un.nchunks; c++, item++) {
            const int s = item & 1;
            const uint32_t ph = (item >> 1) & 1;
            const int L = min(kChunk, un.eos - (un.bos + c * kChunk));
            const float beta_r = beta_next;
            if (et == 0) publish();
            // fused prologue: the three rows before each warp's first row, in flight
            // during the decay scan -- for warp 0 the sequence's previous rows, or
            // its window's taps on its first chunk; for the others rows of the chunk
            // (zero past its end), read from global memory so that no warp reads
            // rows another rewrites
            ConvHalo<kConv> halo;
            if constexpr (kConv) {
                const size_t HC = (size_t)p.H * kD;
                const int cc0 = 4 * (et & 31);                        // this lane's first channel
                const int row0 = un.bos + c * kChunk;
                const int rh = 8 * (et >> 5) - 3;                     // chunk row of halo row 0
#pragma unroll
                for (int sx = 0; sx < 2; sx++)
#pragma unroll
                    for (int j = 0; j < 3; j++) {
                        const uint2 *src = reinterpret_cast<const uint2 *>(cp.x[sx] + (size_t)(row0 + rh + j) * HC + (size_t)un.h * kD + cc0);
                        if (rh < 0)
                            halo.r[sx][j] = c == 0
                                ? *reinterpret_cast<const uint2 *>(cp.pool + ((size_t)un.st * 9 + 3 * j + sx) * HC +
                                                                   (size_t)un.h * kD + cc0)
                                : __ldg(src);
                        else
                            halo.r[sx][j] = rh + j < L ? __ldg(src) : make_uint2(0u, 0u);
                    }
            }
            bool ok = mbar_wait(sm.bar(kBarGFull), item & 1, sm.abort_flag());
            if (role_any(!ok, kBarE, kEThreads)) {
                if (et == 0) record_error(p, sm, kErrWaitTimeout);
                drain_g();
                return;
            }
            if (et == 0) KDA_PHASE(0, item, 0);
            // the next chunk's g is requested as soon as this chunk's g is read
            auto next_g = [&]() {
                if (cursor_next<kSlots, kSort>(ahead, p, sm, order, U)) {
                    if (ahead.c == ahead.un.nchunks) maybe_claim(ahead.k);
                    if (et == 0) {
                        KDA_PHASE(2, ahead.item - 1, 1);
                        issue_g(sm, maps, ahead.row0, ahead.un.h);
                    }
                    beta_next = load_beta(p, ahead, et);
                }
            };
            // beta*V as soon as v has landed (the betas are in place after the scan):
            // before the wait for k and q, so that MMA-b never waits for it (builds
            // with the fused prologue: group I does it, i_conv_v)
            auto convert_v = [&]() -> bool {
                if constexpr (kConv) {
                    return true;   // group I maps the raw value rows (i_conv_v)
                } else {
                    const bool okv = mbar_wait(sm.bar(kBarVFull + s), ph, sm.abort_flag());
                    if (role_any(!okv, kBarE, kEThreads)) return false;
                    e_convert_v(sm, s, L, et);
                    fence_proxy_async_smem();
                    mbar_arrive(sm.bar(kBarEDone + s));
                    return true;
                }
            };
            auto conv_qk = [&]() {
                if constexpr (kConv) {
                    const ConvAt at = conv_at(cp, un, c, et);
                    uint8_t *kq = sm.base + s * kStageBytes + kOffKQ;
                    float w[4][4];
                    conv_weights(cp, 1, un.h, at.c0, w);
                    e_conv_stream<true>(kq + off_k(s), 16384, halo.r[1], w, L, et, cp.act, cp.eps, at.window(1),
                                        at.tap);
                    conv_weights(cp, 0, un.h, at.c0, w);
                    e_conv_stream<true>(kq + off_q(s), 16384, halo.r[0], w, L, et, cp.act, cp.eps, at.window(0),
                                        at.tap);
                    named_bar(kBarE, kEThreads);   // q and k in place before the operand pass reads them
                }
            };
            const int lb = layout_bit<kSort>(order, un, s);
            if (!e_pass(sm, s, lb, item, L, et, beta_r, p.err, next_g, convert_v, conv_qk)) {
                if (et == 0) record_error(p, sm, kErrWaitTimeout);
                // this chunk's g was waited for (item + 1 of them); the next one may be in flight
                item++;
                drain_g();
                return;
            }
            fence_proxy_async_smem();
            named_bar(kBarE, kEThreads);                   // operands written
            if (et == 0) {
                KDA_PHASE(0, item, 1);
                // TMEM P_s is free once the chain has read chunk item-2's outputs
                if (item >= 2 && !mbar_wait(sm.bar(kBarODone + s), ((item >> 1) - 1) & 1, sm.abort_flag()))
                    record_error(p, sm, kErrWaitTimeout);
                KDA_PHASE(0, item, 2);
                tc_fence_after();
                issue_mma_a(sm, s, lb, tmem);
                mma_commit(sm.bar(kBarAFull + s));
                KDA_PHASE(2, item, 2);
            }
            if (et == 0) publish();
            if (et == 0) KDA_PHASE(0, item, 4);
        }
    }
}

// =============================================================================
// prep, group I (warps 12-15): the A readout, the inverse T = (I + A_kk)^-1,
// MMA-b and the -W' conversion (and, with the fused prologue, the value rows)
// =============================================================================
// fp32 blocks of the inverse in the shared kOffTmp region (float offsets):
//   D0 = T[0:32, 0:32], D1 = T[32:64, 32:64]  dense [32][36] (upper-right 16x16 zero)
//   L2 = L[32:64, 0:32] [32][36],  L10 = L[16:32, 0:16], L32 = L[48:64, 32:48] [16][20]
// and, in the kOffP region while the diagonal blocks are solved, the four
// 16x16 diagonal blocks of L, [4][16][20].  Row strides keep warp-MMA
// fragment loads conflict-free.
constexpr int kD0 = 0, kD1 = 1152, kL2 = 2304, kL10 = 3456, kL32 = 3776;

// Inverse of the unit lower-triangular 16x16 block (I + Lb) by forward
// substitution, one column per lane: x[r] = e_c[r] - sum_{j<r} Lb[r][j] x[j].
// Lb is read from shared memory (rows zero right of the diagonal).
__device__ __forceinline__ void solve_column16(const float *Lb, int c, float (&x)[16])
{
#pragma unroll
    for (int r = 0; r < 16; r++) x[r] = 0.f;
#pragma unroll
    for (int r = 0; r < 16; r++) {
        float s0 = (r == c) ? 1.f : 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j = 0; j < r; j += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(Lb + r * 20 + j);
            s0 -= l4.x * x[j];
            s1 -= l4.y * x[j + 1];
            s2 -= l4.z * x[j + 2];
            s3 -= l4.w * x[j + 3];
        }
        x[r] = (s0 + s1) + (s2 + s3);
    }
}

// A readout (A in TMEM: lane = row of [Kp ; Qp], stage 1 [Qp ; Kp]).  The two
// A_qk warps (query rows r): the lower part, diagonal included, goes to the
// MMA3 operand tril(A_qk)^T [i][r] (fp16, each 8 x 8 block stored transposed).
// The two A_kk warps (rows i; beta_i is folded into Kp, so this already is the
// beta-scaled A_kk): the strictly lower part goes to the L blocks; the 16x16
// diagonal blocks are inverted column by column into D0/D1 and, as fp16, into
// T16.
// T = (I + A_kk)^-1 as the fp16 MMA-b operand: one buffer, or in split mode
// one per stage (the producer's shipper copies it out with the stage)
template <bool kSplit>
__device__ __forceinline__ uint32_t t16_off(int s) { return (kSplit && s) ? kOffOT : kOffT16; }

template <bool kSplit>
__device__ void i_read_a(const Smem &sm, int s, int lb, uint32_t tmem, int it, int item)
{
    const int ew = it >> 5, lane = it & 31;
    const int hw = ew & 1;                        // which 32 rows of A_kk or A_qk
    const uint32_t src = tmem + tm_o(s) + ((uint32_t)(32 * ew) << 16);
    if ((ew >= 2) != (lb == 1)) {                 // A_qk: lanes 64-127 in layout 0, 0-63 in layout 1
        const uint32_t bt = sm.u32(s * kStageBytes + off_bq(lb));
        const int mi = lane >> 3, k8 = lane & 7;  // this thread's stored matrix and row
#pragma unroll 1
        for (int hl = 0; hl < 2; hl++) {
            uint32_t f[4][8];                     // [16-column block][fragment]
#pragma unroll
            for (int cb = 0; cb < 4; cb++) tmem_ld16x256_x2(src + ((uint32_t)(16 * hl) << 16) + 16 * cb, f[cb]);
            tmem_wait_ld();
            const int r0 = 32 * hw + 16 * hl + (lane >> 2);              // query rows of the fragments: r0, r0 + 8
            const int rs = 32 * hw + 16 * hl + ((mi & 1) ? 8 : 0);       // first query row of the stored block
#pragma unroll
            for (int cb = 0; cb < 4; cb++) {
                float x[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int r = r0 + ((j & 2) ? 8 : 0), i = 16 * cb + 8 * (j >> 2) + 2 * (lane & 3) + (j & 1);
                    x[j] = i <= r ? __uint_as_float(f[cb][j]) : 0.f;
                }
                const int row = 16 * cb + ((mi & 2) ? 8 : 0) + k8;           // key row i of the stored block
                stmatrix_x4_trans(bt + sw128_chunk(row, rs >> 3), pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]),
                                  pack_f16x2(x[4], x[5]), pack_f16x2(x[6], x[7]));
            }
        }
        return;
    }
    uint32_t a[64];
    tmem_ld32(src, *reinterpret_cast<uint32_t(*)[32]>(a));
    tmem_ld32(src + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
    tmem_wait_ld();
    const int i = 32 * hw + lane, blk = i >> 4, a16 = i & 15;
    auto lval = [&](int j) { return (j < i) ? __uint_as_float(a[j]) : 0.f; };
    float *W = sm.ptr<float>(kOffTmp);
    float *Ld = sm.ptr<float>(kOffP) + blk * 320 + a16 * 20;
    if (hw == 0) {
#pragma unroll
        for (int q = 0; q < 4; q++)
            *reinterpret_cast<float4 *>(Ld + 4 * q) =
                (lane & 16) ? make_float4(lval(16 + 4 * q), lval(17 + 4 * q), lval(18 + 4 * q), lval(19 + 4 * q))
                            : make_float4(lval(4 * q), lval(1 + 4 * q), lval(2 + 4 * q), lval(3 + 4 * q));
        if (lane >= 16) {                          // rows 16-31: L10 = L[16:32, 0:16]
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<float4 *>(W + kL10 + (i - 16) * 20 + 4 * q) =
                    make_float4(lval(4 * q), lval(4 * q + 1), lval(4 * q + 2), lval(4 * q + 3));
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; q++)
            *reinterpret_cast<float4 *>(Ld + 4 * q) =
                (lane & 16) ? make_float4(lval(48 + 4 * q), lval(49 + 4 * q), lval(50 + 4 * q), lval(51 + 4 * q))
                            : make_float4(lval(32 + 4 * q), lval(33 + 4 * q), lval(34 + 4 * q), lval(35 + 4 * q));
        // rows 32-63: L[32:64, 0:32]; rows 48-63 also L32
#pragma unroll
        for (int q = 0; q < 8; q++)
            *reinterpret_cast<float4 *>(W + kL2 + (i - 32) * 36 + 4 * q) =
                make_float4(lval(4 * q), lval(4 * q + 1), lval(4 * q + 2), lval(4 * q + 3));
        if (lane >= 16) {
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<float4 *>(W + kL32 + (i - 48) * 20 + 4 * q) =
                    make_float4(lval(32 + 4 * q), lval(33 + 4 * q), lval(34 + 4 * q), lval(35 + 4 * q));
        }
    }
    __syncwarp();
    if (it == 0) KDA_PHASE(0, item, 12);
    {   // lane = column c of diagonal block bb (this warp's two blocks)
        const int c = lane & 15, bb = 2 * hw + (lane >> 4);
        float x[16];
        solve_column16(sm.ptr<float>(kOffP) + bb * 320, c, x);
        float *D = W + (hw ? kD1 : kD0) + (lane >> 4) * (16 * 36 + 16);
#pragma unroll
        for (int r = 0; r < 16; r++) D[r * 36 + c] = x[r];
    }
    __syncwarp();
    if (it == 0) KDA_PHASE(0, item, 13);
    {   // row i of its diagonal block -> fp16 T16 (two 16-byte chunks)
        const float *Dr = W + (hw ? kD1 : kD0) + lane * 36 + (lane >> 4) * 16;
        uint32_t h[8];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float4 v4 = *reinterpret_cast<const float4 *>(Dr + 4 * q);
            h[2 * q] = pack_f16x2(v4.x, v4.y);
            h[2 * q + 1] = pack_f16x2(v4.z, v4.w);
        }
        uint8_t *T16 = sm.base + t16_off<kSplit>(s);
        *reinterpret_cast<uint4 *>(T16 + sw128_chunk(i, 2 * blk)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(T16 + sw128_chunk(i, 2 * blk + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// Block merges of (I + L)^-1 on the warp MMA (tf32 operands, fp32 accumulate),
// on the dense fp32 blocks; the merged blocks go to the fp16 operand T16, whose
// own rounding is of the same size as the tf32 operand rounding (the fp32
// diagonal inverses are exact to fp32).
//   level 1: T10 = -X1 (L10 X0),  T32 = -X3 (L32 X2)       (into D0 / D1)
//   level 2: T[32:64, 0:32] = -D1 (L[32:64, 0:32] D0)
template <bool kSplit>
__device__ void i_merge(const Smem &sm, int s, int it)
{
    const int iw = it >> 5, lane = it & 31, g = lane >> 2, t = lane & 3;
    float *W = sm.ptr<float>(kOffTmp);
    uint8_t *T16 = sm.base + t16_off<kSplit>(s);
    float *P1 = sm.ptr<float>(kOffP);            // [2][16][24]
    float *P2 = P1;                              // [32][40] once P1 is dead
    auto put16 = [&](int r, int c, float v0, float v1) {   // c even
        *reinterpret_cast<uint32_t *>(T16 + sw128_chunk(r, c >> 3) + 2 * (c & 7)) = pack_f16x2(v0, v1);
    };
    {
        const int bl = iw >> 1, nt = iw & 1;
        float *D = W + (bl ? kD1 : kD0);
        const float *Lb = W + (bl ? kL32 : kL10);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(d, [&](int rr, int kk) { return Lb[rr * 20 + kk]; },
                 [&](int kk, int cc) { return D[kk * 36 + 8 * nt + cc]; }, nt, 2, lane);
        float *P = P1 + bl * 384;
        *reinterpret_cast<float2 *>(P + g * 24 + 8 * nt + 2 * t) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(P + (g + 8) * 24 + 8 * nt + 2 * t) = make_float2(d[2], d[3]);
        named_bar(kBarI, kGroupThreads);
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(e, [&](int rr, int kk) { return D[(16 + rr) * 36 + 16 + kk]; },
                 [&](int kk, int cc) { return P[kk * 24 + 8 * nt + cc]; }, 0, 2, lane);
        *reinterpret_cast<float2 *>(D + (16 + g) * 36 + 8 * nt + 2 * t) = make_float2(-e[0], -e[1]);
        *reinterpret_cast<float2 *>(D + (24 + g) * 36 + 8 * nt + 2 * t) = make_float2(-e[2], -e[3]);
        const int r0 = 32 * bl + 16, c0 = 32 * bl;
        put16(r0 + g, c0 + 8 * nt + 2 * t, -e[0], -e[1]);
        put16(r0 + g + 8, c0 + 8 * nt + 2 * t, -e[2], -e[3]);
    }
    named_bar(kBarI, kGroupThreads);
    // level 2: each warp one 16-row slab mt and two 8-column tiles n0, n0+1
    // sharing the A fragment (two independent accumulation chains)
    const int mt = iw >> 1, n0 = 2 * (iw & 1);
    {
        const float *L2 = W + kL2, *D0 = W + kD0;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int ks = n0; ks < 4; ks++) {           // D0 is zero above its diagonal
            const int r = 16 * mt + g, k0 = 8 * ks + t;
            const float a[4] = {L2[r * 36 + k0], L2[(r + 8) * 36 + k0], L2[r * 36 + k0 + 4], L2[(r + 8) * 36 + k0 + 4]};
            const float b0[2] = {D0[k0 * 36 + 8 * n0 + g], D0[(k0 + 4) * 36 + 8 * n0 + g]};
            const float b1[2] = {D0[k0 * 36 + 8 * n0 + 8 + g], D0[(k0 + 4) * 36 + 8 * n0 + 8 + g]};
            mma_1xtf32(d0, a, b0);
            mma_1xtf32(d1, a, b1);
        }
        const int r = 16 * mt + g;
        *reinterpret_cast<float2 *>(P2 + r * 40 + 8 * n0 + 2 * t) = make_float2(d0[0], d0[1]);
        *reinterpret_cast<float2 *>(P2 + (r + 8) * 40 + 8 * n0 + 2 * t) = make_float2(d0[2], d0[3]);
        *reinterpret_cast<float2 *>(P2 + r * 40 + 8 * n0 + 8 + 2 * t) = make_float2(d1[0], d1[1]);
        *reinterpret_cast<float2 *>(P2 + (r + 8) * 40 + 8 * n0 + 8 + 2 * t) = make_float2(d1[2], d1[3]);
    }
    named_bar(kBarI, kGroupThreads);
    {
        const float *D1 = W + kD1;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int ks = 0; ks <= 2 * mt + 1; ks++) {   // D1 is zero above its diagonal
            const int rr = 16 * mt + g, k0 = 8 * ks + t;
            const float a[4] = {D1[rr * 36 + k0], D1[(rr + 8) * 36 + k0], D1[rr * 36 + k0 + 4], D1[(rr + 8) * 36 + k0 + 4]};
            const float b0[2] = {P2[k0 * 40 + 8 * n0 + g], P2[(k0 + 4) * 40 + 8 * n0 + g]};
            const float b1[2] = {P2[k0 * 40 + 8 * n0 + 8 + g], P2[(k0 + 4) * 40 + 8 * n0 + 8 + g]};
            mma_1xtf32(d0, a, b0);
            mma_1xtf32(d1, a, b1);
        }
        const int r = 32 + 16 * mt + g;
        put16(r, 8 * n0 + 2 * t, -d0[0], -d0[1]);
        put16(r + 8, 8 * n0 + 2 * t, -d0[2], -d0[3]);
        put16(r, 8 * n0 + 8 + 2 * t, -d1[0], -d1[1]);
        put16(r + 8, 8 * n0 + 8 + 2 * t, -d1[2], -d1[3]);
    }
}

template <bool kSplit>
__device__ void issue_mma_b(const Smem &sm, int s, int lb, uint32_t tmem)
{
    const uint32_t st = sm.u32(s * kStageBytes);
    const uint32_t id = idesc_f16(128, 64, 1, 0);
#pragma unroll 1
    for (int ks = 0; ks < 4; ks++) {
        const uint64_t bd = smem_desc_sw128(sm.u32(t16_off<kSplit>(s)) + ks * 32, 16, 1024);
        const uint64_t aw = smem_desc_sw128(st + kOffKQ + off_k(lb) + ks * 2048, 16384, 1024);  // Kp^T, MN-major
        const uint64_t au = smem_desc_sw128(st + kOffV + ks * 2048, 8192, 1024);                // V^T, MN-major
        mma_ss(tmem + tm_o(s), aw, bd, id, ks > 0);
        mma_ss(tmem + tm_d(s), au, bd, id, ks > 0);
    }
}

// -W'^T (TMEM, lane = key channel c, column = row r) -> -W' as fp16 K-major
// [r][c] in the stage's K rows (Kp is dead once MMA-b is done), so that
// [-W' ; Qp] is one 128-row operand for MMA1.  TMEM is read in the warp-MMA
// fragment layout and each 8 x 8 block is stored transposed (stmatrix.trans).
// Then the TMEM columns MMA1 accumulates the output into are zeroed.
__device__ void i_read_w(const Smem &sm, int s, int lb, uint32_t tmem, int it)
{
    const int iw = it >> 5, lane = it & 31;
    const int mi = lane >> 3, k8 = lane & 7;              // this thread's stored matrix and row
    const uint32_t src = tmem + tm_o(s) + ((uint32_t)(32 * iw) << 16);
    const uint32_t kq = sm.u32(s * kStageBytes + kOffKQ + off_k(lb));
#pragma unroll 1
    for (int hl = 0; hl < 2; hl++) {
        uint32_t f[4][8];                                 // [16-column block][fragment]
#pragma unroll
        for (int cb = 0; cb < 4; cb++) tmem_ld16x256_x2(src + ((uint32_t)(16 * hl) << 16) + 16 * cb, f[cb]);
        tmem_wait_ld();
        const int c = 32 * iw + 16 * hl + ((mi & 1) ? 8 : 0);          // first key channel of the block
        const uint32_t base = kq + (c >> 6) * 16384;
#pragma unroll
        for (int cb = 0; cb < 4; cb++) {
            const int r = 16 * cb + ((mi & 2) ? 8 : 0) + k8;
            stmatrix_x4_trans(base + sw128_chunk(r, (c & 63) >> 3),
                              pack_f16x2(-__uint_as_float(f[cb][0]), -__uint_as_float(f[cb][1])),
                              pack_f16x2(-__uint_as_float(f[cb][2]), -__uint_as_float(f[cb][3])),
                              pack_f16x2(-__uint_as_float(f[cb][4]), -__uint_as_float(f[cb][5])),
                              pack_f16x2(-__uint_as_float(f[cb][6]), -__uint_as_float(f[cb][7])));
        }
    }
    uint32_t z[32];
#pragma unroll
    for (int j = 0; j < 32; j++) z[j] = 0u;
    tmem_st32(src, z);
    tmem_st32(src + 32, z);
    tmem_wait_st();
}

// The fused prologue's value stream (kConv builds), done by group I on the
// chunk it is about to take, before it waits for that chunk's MMA-a (group E
// has the q and k streams and the decay pass): the conv (and SiLU) of the raw
// v rows, rounded to bf16 as the prologue's own outputs are, then beta_r * v
// as fp16 in place -- the bytes of e_conv_stream followed by e_convert_v.
// Warp w takes rows 16w .. 16w+15 in two passes of 8 rows, lane l channels
// 4l .. 4l+3 of the head.  A warp reads from shared memory only the rows it
// rewrites itself, and the three rows before its first row from global memory
// (warp 0 on a sequence's first chunk: the window's taps), so the warps never
// wait for one another; warp 0 also rewrites the window, after it has read
// the old taps.
__device__ void i_conv_v(const TcParams &p, const ConvParams &cp, const Smem &sm, int s, const Unit &un, int c, int L,
                         int it)
{
    const int lane = it & 31, iw = it >> 5;
    const size_t HC = (size_t)p.H * kD;
    const int c0 = 4 * lane;
    const int row0 = un.bos + c * kChunk;
    uint8_t *base = sm.base + s * kStageBytes + kOffV + (lane >> 4) * 8192 + 8 * (lane & 1);
    const int ch = (lane & 15) >> 1;                              // 16-byte chunk of channel c0 in its block row
    const uint16_t *xv = cp.x[2] + (size_t)un.h * kD + c0;        // row r of the projection at xv + r * HC
    uint2 raw[11];                                                // rows r0 - 3 .. r0 + 7 of a pass
    {
        uint16_t *win = cp.pool + ((size_t)un.st * 9 + 2) * HC + (size_t)un.h * kD + c0;   // tap j at win + 3 j HC
#pragma unroll
        for (int j = 0; j < 3; j++) {
            const int r = 16 * iw - 3 + j;
            const uint2 *src = reinterpret_cast<const uint2 *>(xv + (size_t)(row0 + r) * HC);
            if (r < 0)
                raw[j] = c == 0 ? *reinterpret_cast<const uint2 *>(win + 3 * j * HC) : __ldg(src);
            else
                raw[j] = r < L ? __ldg(src) : make_uint2(0u, 0u);
        }
        if (iw == 0 && c == un.nchunks - 1) {
            // the new window: the last three raw rows of [old taps ; the sequence's
            // rows], all read before the first is written
            uint2 nt[3];
#pragma unroll
            for (int j = 0; j < 3; j++) {
                const int r = L - 3 + j;                          // < 0 on a first chunk: old tap j + L
                nt[j] = r >= 0 || c > 0 ? __ldg(reinterpret_cast<const uint2 *>(xv + (size_t)(row0 + r) * HC))
                                        : *reinterpret_cast<const uint2 *>(win + 3 * (j + L) * HC);
            }
#pragma unroll
            for (int j = 0; j < 3; j++) *reinterpret_cast<uint2 *>(win + 3 * j * HC) = nt[j];
        }
    }
    // beta of row 16w + l at lane l < 16 (zero past the chunk), shuffled out per row
    const int rb = 16 * iw + (lane & 15);
    const float bl = rb < L ? __ldg(p.beta + (size_t)(row0 + rb) * p.H + un.h) : 0.f;
    float w[4][4];
    conv_weights(cp, 2, un.h, c0, w);
#pragma unroll 1
    for (int hp = 0; hp < 2; hp++) {   // rolled: one copy of the code (it runs once a chunk)
        const int r0 = 16 * iw + 8 * hp;
        if (hp) {
#pragma unroll
            for (int j = 0; j < 3; j++) raw[j] = raw[8 + j];
        }
#pragma unroll
        for (int t = 0; t < 8; t++) raw[3 + t] = *reinterpret_cast<const uint2 *>(base + sw128_chunk(r0 + t, ch));
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const float x[4][4] = {{bf16lo(raw[t].x), bf16hi(raw[t].x), bf16lo(raw[t].y), bf16hi(raw[t].y)},
                                   {bf16lo(raw[t + 1].x), bf16hi(raw[t + 1].x), bf16lo(raw[t + 1].y), bf16hi(raw[t + 1].y)},
                                   {bf16lo(raw[t + 2].x), bf16hi(raw[t + 2].x), bf16lo(raw[t + 2].y), bf16hi(raw[t + 2].y)},
                                   {bf16lo(raw[t + 3].x), bf16hi(raw[t + 3].x), bf16lo(raw[t + 3].y), bf16hi(raw[t + 3].y)}};
            float y[4];
#pragma unroll
            for (int cc = 0; cc < 4; cc++) {                      // the same order of the sum as e_conv_stream
                float a = w[cc][0] * x[0][cc];
                a = fmaf(w[cc][1], x[1][cc], a);
                a = fmaf(w[cc][2], x[2][cc], a);
                a = fmaf(w[cc][3], x[3][cc], a);
                y[cc] = cp.act ? conv_silu(a) : a;
            }
            const uint32_t b0 = pack_bf16x2(y[0], y[1]), b1 = pack_bf16x2(y[2], y[3]);
            const float b = __shfl_sync(0xffffffffu, bl, 8 * hp + t);
            const float2 v0 = fmul2(make_float2(bf16lo(b0), bf16hi(b0)), make_float2(b, b));
            const float2 v1 = fmul2(make_float2(bf16lo(b1), bf16hi(b1)), make_float2(b, b));
            const uint2 out = r0 + t < L ? make_uint2(pack_f16x2(v0.x, v0.y), pack_f16x2(v1.x, v1.y))
                                         : make_uint2(0u, 0u);
            *reinterpret_cast<uint2 *>(base + sw128_chunk(r0 + t, ch)) = out;
        }
    }
}

template <bool kSlots, int kSort, bool kConv>
__device__ void i_role(const TcParams &p, const ConvParams *cp, const Smem &sm, const int *order, int U)
{
    const int it = threadIdx.x - kChainThreads - kEThreads;
    const uint32_t tmem = *sm.tmem_base();
    constexpr bool kSplit = kSort == kSortChunks;
    {   // zeros that stay for the whole kernel: T16's 16-byte chunks right of each
        // row's diagonal block, and the upper-right 16x16 blocks of D0 and D1
        for (int b = 0; b < (kSplit ? 2 : 1); b++) {
            uint8_t *T16 = sm.base + t16_off<kSplit>(b);
            for (int idx = it; idx < 64 * 8; idx += kGroupThreads) {
                const int r = idx >> 3, q = idx & 7;
                if (q > 2 * (r >> 4) + 1)
                    *reinterpret_cast<uint4 *>(T16 + sw128_chunk(r, q)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float *W = sm.ptr<float>(kOffTmp);
        for (int idx = it; idx < 2 * 16 * 16; idx += kGroupThreads) {
            const int b = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
            W[(b ? kD1 : kD0) + r * 36 + 16 + c] = 0.f;
        }
        fence_proxy_async_smem();
    }
    int item = 0;
    for (int k = 0;; k++) {
        const int u = cta_unit<kSort>(sm, k, U);
        if (u < 0) break;
        const Unit un = get_unit<kSlots, kSort>(p, order, u);
        for (int c = 0; c < un.nchunks; c++, item++) {
            const int s = item & 1;
            const int lb = layout_bit<kSort>(order, un, s);
            const uint32_t ph = (item >> 1) & 1;
            if constexpr (kConv) {   // the value rows, once landed: beta*V for MMA-b
                const bool okv = mbar_wait(sm.bar(kBarVFull + s), ph, sm.abort_flag());
                if (role_any(!okv, kBarI, kGroupThreads)) { if (it == 0) record_error(p, sm, kErrWaitTimeout); return; }
                i_conv_v(p, *cp, sm, s, un, c, min(kChunk, un.eos - (un.bos + c * kChunk)), it);
            }
            // MMA-a done implies group E's operand pass is over (MMA-b of the previous
            // chunk, the last reader of T16, was waited for below)
            bool ok = mbar_wait(sm.bar(kBarAFull + s), ph, sm.abort_flag());
            if (role_any(!ok, kBarI, kGroupThreads)) { if (it == 0) record_error(p, sm, kErrWaitTimeout); return; }
            if (it == 0) KDA_PHASE(0, item, 5);
            tc_fence_after();
            i_read_a<kSplit>(sm, s, lb, tmem, it, item);
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(kBarI, kGroupThreads);
            if (it == 0) KDA_PHASE(0, item, 3);
            i_merge<kSplit>(sm, s, it);
            if (it == 0) KDA_PHASE(0, item, 6);
            fence_proxy_async_smem();
            named_bar(kBarI, kGroupThreads);
            if (it == 0) {
                if (!kConv && !mbar_wait(sm.bar(kBarEDone + s), ph, sm.abort_flag())) {   // group E's beta*V
                    record_error(p, sm, kErrWaitTimeout);
                } else {
                    KDA_PHASE(0, item, 7);
                    tc_fence_after();
                    issue_mma_b<kSplit>(sm, s, lb, tmem);
                    mma_commit(sm.bar(kBarPrepDone + s));
                    KDA_PHASE(0, item, 8);
                }
            }
            // -W' out of TMEM into the K rows of the stage (and the output columns
            // zeroed) for the chain's MMA1
            ok = mbar_wait(sm.bar(kBarPrepDone + s), ph, sm.abort_flag());
            if (role_any(!ok, kBarI, kGroupThreads)) { if (it == 0) record_error(p, sm, kErrWaitTimeout); return; }
            tc_fence_after();
            i_read_w(sm, s, lb, tmem, it);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(sm.bar(kBarWReady + s));
            if (it == 0) KDA_PHASE(0, item, 9);
        }
    }
}

// =============================================================================
// chain role: warps 0-3 (thread v owns TMEM lane v = value channel v)
// =============================================================================
// O^T (TMEM, lane v, column r) -> out[row0 + r][h][v] (bf16), rows r < L.
// TMEM is read in the warp-MMA fragment layout (16x256b) and stmatrix.trans
// writes each 8 x 8 block transposed into two 128B-swizzled tiles of 32 rows:
// rows 0-31 into the stage's tril(A_qk) buffer (MMA3 is done with it), rows
// 32-63 into the output buffer.  The first thread stores each full tile with
// one bulk tensor copy; the rows r < L of a partial tile are stored by every
// thread, 16 bytes at a time.  The first thread later waits until the copies
// have read the tiles and only then hands TMEM P_s and the tril(A_qk) buffer
// back to the prep (o_done).
__device__ void chain_store_out(const TcParams &p, const Smem &sm, const Maps &maps, uint32_t tmem, int s, int row0,
                                int L, int h, int v, int item)
{
    const int w = v >> 5, lane = v & 31;
    uint32_t o[2][4][8];                                  // [16-lane half][16-column block][fragment]
    const uint32_t src = tmem + tm_o(s) + ((uint32_t)(32 * w) << 16);
#pragma unroll
    for (int hl = 0; hl < 2; hl++)
#pragma unroll
        for (int cb = 0; cb < 4; cb++) tmem_ld16x256_x2(src + ((uint32_t)(16 * hl) << 16) + 16 * cb, o[hl][cb]);
    tmem_wait_ld();
    tc_fence_before();
    if (v == 0) KDA_PHASE(1, item, 8);
    const uint32_t tile0 = sm.u32(s * kStageBytes + off_bq(s)), tile1 = sm.u32(kOffOT);
    const int mi = lane >> 3, k8 = lane & 7;              // this thread's stored matrix and row
#pragma unroll
    for (int cb = 0; cb < 4; cb++) {                      // output rows 16*cb .. +15
#pragma unroll
        for (int hl = 0; hl < 2; hl++) {
            const uint32_t *f = o[hl][cb];
            const int rl = 16 * (cb & 1) + ((mi & 2) ? 8 : 0) + k8;      // row within the tile
            const int vc = 32 * w + 16 * hl + ((mi & 1) ? 8 : 0);      // first value channel
            stmatrix_x4_trans((cb < 2 ? tile0 : tile1) + (vc >> 6) * 4096 + sw128_chunk(rl, (vc & 63) >> 3),
                              pack_bf16x2(__uint_as_float(f[0]), __uint_as_float(f[1])),
                              pack_bf16x2(__uint_as_float(f[2]), __uint_as_float(f[3])),
                              pack_bf16x2(__uint_as_float(f[4]), __uint_as_float(f[5])),
                              pack_bf16x2(__uint_as_float(f[6]), __uint_as_float(f[7])));
        }
    }
    fence_proxy_async_smem();
    named_bar(kBarChain, kChainThreads);
    if (v == 0) {
        if (L >= 32) tma_store_4d(maps.o, 0, row0, 0, h, tile0);
        if (L == kChunk) tma_store_4d(maps.o, 0, row0 + 32, 0, h, tile1);
        bulk_commit();
    }
    if (L < kChunk) {                                     // the partial tile, row by row
        const int half = L < 32 ? 0 : 1, nr = L - 32 * half;
        const uint8_t *tb = sm.base + (half ? kOffOT : s * kStageBytes + off_bq(s));
        const size_t row_stride = (size_t)p.H * kD;
        __nv_bfloat16 *dst = p.out + ((size_t)(row0 + 32 * half) * p.H + h) * kD;
        for (int idx = v; idx < nr * 16; idx += kChainThreads) {
            const int r = idx >> 4, q = idx & 15;
            *reinterpret_cast<uint4 *>(dst + (size_t)r * row_stride + 8 * q) =
                *reinterpret_cast<const uint4 *>(tb + (q >> 3) * 4096 + sw128_chunk(r, q & 7));
        }
    }
    if (v == 0) KDA_PHASE(1, item, 9);
}

// ---- states between global memory and TMEM -------------------------------------
// A state row (value channel v: 128 key channels, 512 contiguous bytes) lives
// in TMEM lane v.  This warp's 32 state rows <-> TMEM columns tm .. tm+127 of its lanes, in the
// 16x256b fragment layout: thread t holds rows t/4 and 8 + t/4 of each 16-lane
// half and, in each group of 32 columns, columns 8b + 2 (t%4), +1 -- so the
// four threads of a row move 32 contiguous bytes, a whole sector, and no
// staging is needed.  Groups go two at a time (one in flight while the other
// is written).
__device__ void chain_load_state(const float *src, uint32_t tm, int lane)
{
    if (!src) {   // zeros: straight into TMEM
        uint32_t z[16];
#pragma unroll
        for (int j = 0; j < 16; j++) z[j] = 0u;
#pragma unroll
        for (int r = 0; r < 8; r++) tmem_st16(tm + 16 * r, z);
        tmem_wait_st();
        return;
    }
    const int rr = lane >> 2, cc = 2 * (lane & 3);
    float2 v[2][8];
    auto fetch = [&](int gi, float2 (&d)[8]) {   // group gi: half gi >> 2, columns 32 (gi & 3) ..
        const float *base = src + (16 * (gi >> 2) + rr) * kD + 32 * (gi & 3) + cc;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            d[2 * b] = *reinterpret_cast<const float2 *>(base + 8 * b);
            d[2 * b + 1] = *reinterpret_cast<const float2 *>(base + 8 * kD + 8 * b);
        }
    };
    fetch(0, v[0]);
#pragma unroll
    for (int gi = 0; gi < 8; gi++) {
        if (gi + 1 < 8) fetch(gi + 1, v[(gi + 1) & 1]);
        const float2 *d = v[gi & 1];
        uint32_t x[16];
#pragma unroll
        for (int b = 0; b < 4; b++) {
            x[4 * b] = __float_as_uint(d[2 * b].x); x[4 * b + 1] = __float_as_uint(d[2 * b].y);
            x[4 * b + 2] = __float_as_uint(d[2 * b + 1].x); x[4 * b + 3] = __float_as_uint(d[2 * b + 1].y);
        }
        tmem_st16x256_x4(tm + ((uint32_t)(16 * (gi >> 2)) << 16) + 32 * (gi & 3), x);
    }
    tmem_wait_st();
}

// TMEM columns tm .. tm+127 of this warp's lanes, times pend per key channel ->
// its 32 state rows at dst (the same fragment layout)
__device__ void chain_store_state(float *dst, const float *pend, uint32_t tm, int lane)
{
    const int rr = lane >> 2, cc = 2 * (lane & 3);
    uint32_t x[2][16];
    auto ld = [&](int gi, uint32_t (&d)[16]) {
        tmem_ld16x256_x4(tm + ((uint32_t)(16 * (gi >> 2)) << 16) + 32 * (gi & 3), d);
    };
    ld(0, x[0]);
    tmem_wait_ld();
#pragma unroll
    for (int gi = 0; gi < 8; gi++) {
        if (gi + 1 < 8) ld(gi + 1, x[(gi + 1) & 1]);
        const uint32_t *y = x[gi & 1];
        float *base = dst + (16 * (gi >> 2) + rr) * kD + 32 * (gi & 3) + cc;
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const float2 pe = *reinterpret_cast<const float2 *>(pend + 32 * (gi & 3) + 8 * b + cc);
            *reinterpret_cast<float2 *>(base + 8 * b) =
                make_float2(__fmul_rn(__uint_as_float(y[4 * b]), pe.x), __fmul_rn(__uint_as_float(y[4 * b + 1]), pe.y));
            *reinterpret_cast<float2 *>(base + 8 * kD + 8 * b) =
                make_float2(__fmul_rn(__uint_as_float(y[4 * b + 2]), pe.x), __fmul_rn(__uint_as_float(y[4 * b + 3]), pe.y));
        }
        if (gi + 1 < 8) tmem_wait_ld();
    }
}

// S <- (S * pend) * fm column by column (pend may be null), written back, and
// its fp16 copy S'h (two per 32-bit column) for the chain MMAs.
__device__ void chain_scale_state(uint32_t tmem, uint32_t lane_off, const float *fm, const float *pend, int item)
{
#pragma unroll 1
    for (int q = 0; q < 4; q++) {                       // 32 key channels at a time
        uint32_t x[32];
        tmem_ld32(tmem + kTmS + lane_off + 32 * q, x);
        tmem_wait_ld();
        if (lane_off == 0 && threadIdx.x == 0) {
            if (q == 0) KDA_PHASE(1, item, 15);
            if (q == 3) KDA_PHASE(1, item, 10);
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 f4 = *reinterpret_cast<const float4 *>(fm + 32 * q + j);
            const float4 p4 = pend ? *reinterpret_cast<const float4 *>(pend + 32 * q + j)
                                   : make_float4(1.f, 1.f, 1.f, 1.f);
            float2 lo = make_float2(__uint_as_float(x[j]), __uint_as_float(x[j + 1]));
            float2 hi = make_float2(__uint_as_float(x[j + 2]), __uint_as_float(x[j + 3]));
            if (pend) {
                lo = fmul2(lo, make_float2(p4.x, p4.y));
                hi = fmul2(hi, make_float2(p4.z, p4.w));
            }
            lo = fmul2(lo, make_float2(f4.x, f4.y));
            hi = fmul2(hi, make_float2(f4.z, f4.w));
            x[j] = __float_as_uint(lo.x); x[j + 1] = __float_as_uint(lo.y);
            x[j + 2] = __float_as_uint(hi.x); x[j + 3] = __float_as_uint(hi.y);
        }
        uint32_t h[16];
#pragma unroll
        for (int j = 0; j < 16; j++) h[j] = pack_f16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
        tmem_st32(tmem + kTmS + lane_off + 32 * q, x);
        tmem_st16(tmem + kTmS0h + lane_off + 16 * q, h);
    }
    if (lane_off == 0 && threadIdx.x == 0) KDA_PHASE(1, item, 14);
    tmem_wait_st();
}

// kq_pending (thread 0): chunk cur.item-1's v is requested, its k and q not yet
template <bool kSlots, int kSort>
__device__ void chain_units(const TcParams &p, const Smem &sm, const int *order, int U, const Maps &maps,
                            LoadCursor &cur, bool &kq_pending, uint32_t tmem, uint32_t lane_off, int v)
{
    int item = 0;
    int o_pending = -1;       // thread 0: stage whose output copies may still read their tiles
    // this warp's first state row of a unit
    auto warp_rows = [&](const Unit &x) { return (((size_t)x.st * p.H + x.h) * kD + (v & ~31)) * kD; };
    for (int k = 0;; k++) {
        const int u = cta_unit<kSort>(sm, k, U);
        if (u < 0) break;
        const Unit un = get_unit<kSlots, kSort>(p, order, u);
        const size_t soff = (((size_t)un.st * p.H + un.h) * kD + v) * kD;   // used only when st >= 0
        if (un.nchunks == 0) {
            if (p.s1 && (!kSlots || un.st >= 0)) {
                for (int c = 0; c < kD; c += 4) {
                    float4 x = p.s0 ? *reinterpret_cast<const float4 *>(p.s0 + soff + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(p.s1 + soff + c) = x;
                }
            }
            continue;
        }
        // initial state -> S (TMEM, lane v, columns = key channels)
        chain_load_state(p.s0 ? p.s0 + warp_rows(un) : nullptr, tmem + kTmS + lane_off, v & 31);
        for (int c = 0; c < un.nchunks; c++, item++) {
            const int s = item & 1;
            const uint32_t ph = (item >> 1) & 1;
            const int row0 = un.bos + c * kChunk;
            const int L = min(kChunk, un.eos - row0);
            // the state is rescaled as soon as the chunk's decay constants exist,
            // while the prep still works on the chunk's inverse and W'
            bool ok = mbar_wait(sm.bar(kBarFmReady + s), ph, sm.abort_flag());
            if (role_any(!ok, kBarChain, kChainThreads)) { if (v == 0) record_error(p, sm, kErrWaitTimeout); return; }
            if (v == 0) KDA_PHASE(1, item, 0);
            if (v == 0 && p.s0 && c == un.nchunks - 1) {
                // the next unit's initial state heads for L2 during this last chunk
                const int un2 = cta_unit_peek<kSort>(sm, k + 1, U);
                if (un2 >= 0) {
                    const Unit nx = get_unit<kSlots, kSort>(p, order, un2);
                    if (!kSlots || nx.st >= 0) {
                        const float *src = p.s0 + ((size_t)nx.st * p.H + nx.h) * kD * kD;
                        for (int part = 0; part < 4; part++) prefetch_l2(src + part * 4096, 16384);
                    }
                }
            }
            tc_fence_after();
            chain_scale_state(tmem, lane_off, sm.ptr<float>(kOffConst + s * kConstBytes),
                              c > 0 ? sm.ptr<float>(kOffPend) + ((item - 1) % 3) * 128 : nullptr, item);
            if (v == 0) KDA_PHASE(1, item, 6);
            if (v == 0 && o_pending >= 0) {
                // the previous chunk's output copies have read their tiles (long since)
                bulk_wait_read0();
                mbar_arrive(sm.bar(kBarODone + o_pending));
                o_pending = -1;
            }
            tc_fence_before();
            // group I has put -W' into the stage (so MMA-b is done) -- and the
            // barrier orders every lane's S'h stores before MMA1
            ok = mbar_wait(sm.bar(kBarWReady + s), ph, sm.abort_flag());
            if (role_any(!ok, kBarChain, kChainThreads)) { if (v == 0) record_error(p, sm, kErrWaitTimeout); return; }
            if (v == 0) {
                KDA_PHASE(1, item, 11);
                // MMA-b is done with V: chunk item+2's v may land
                if (cursor_next<kSlots, kSort>(cur, p, sm, order, U)) {
                    issue_v(sm, maps, cur.item - 1, cur.row0, cur.un.h);
                    kq_pending = true;
                }
                KDA_PHASE(1, item, 12);
                tc_fence_after();
                const uint32_t st = sm.u32(s * kStageBytes);
                // [U^T | 0] += S'^T [-W' ; Qp]^T: the Delta half and the output half in
                // one N = 128 MMA (the K rows of each stage block hold -W', the Q rows
                // Qp; in stage 1 Q rows first, output half first)
                const uint32_t id1 = idesc_f16(128, 128, 0, 0);
#pragma unroll 1
                for (int ks = 0; ks < 8; ks++) {
                    const int kb = ks >> 2, kin = ks & 3;
                    const uint64_t bwq = smem_desc_sw128(st + kOffKQ + kb * 16384 + kin * 32, 16, 1024);
                    mma_ts(tmem + (s ? tm_o(1) : tm_d(0)), tmem + kTmS0h + 8 * ks, bwq, id1, 1);
                }
                mma_commit(sm.bar(kBarMma1));
                KDA_PHASE(1, item, 1);
            }
            ok = mbar_wait(sm.bar(kBarMma1), item & 1, sm.abort_flag(), KDA_WAIT_LIMIT_MMA1);
            if (role_any(!ok, kBarChain, kChainThreads)) { if (v == 0) record_error(p, sm, kErrWaitTimeout); return; }
            if (v == 0) {
                KDA_PHASE(1, item, 2);
                if (kq_pending) {                             // -W' and Qp have been read
                    issue_kq(sm, maps, cur.item - 1, cur.row0, cur.un.h, (cur.item - 1) & 1);
                    kq_pending = false;
                }
            }
            tc_fence_after();
            // Delta^T (fp32, TMEM) -> fp16 A operand
            {
                uint32_t x[64];
                tmem_ld32(tmem + tm_d(s) + lane_off, *reinterpret_cast<uint32_t(*)[32]>(x));
                tmem_ld32(tmem + tm_d(s) + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
                tmem_wait_ld();
                uint32_t h0[16], h1[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    h0[j] = pack_f16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
                    h1[j] = pack_f16x2(__uint_as_float(x[32 + 2 * j]), __uint_as_float(x[32 + 2 * j + 1]));
                }
                tmem_st16(tmem + kTmDh + lane_off, h0);
                tmem_st16(tmem + kTmDh + lane_off + 16, h1);
            }
            tmem_wait_st();
            if (v == 0) KDA_PHASE(1, item, 7);
            tc_fence_before();
            named_bar(kBarChain, kChainThreads);
            if (v == 0) {
                tc_fence_after();
                const uint32_t st = sm.u32(s * kStageBytes);
                // the state update and the rest of the output in one N = 192 MMA:
                // [O^T | S^T] += Delta^T [tril(A_qk)^T | Km] in stage 0,
                // [S^T | O^T] += Delta^T [Km | tril(A_qk)^T] in stage 1 (B MN-major)
                const uint32_t id3 = idesc_f16(128, 192, 0, 1);
#pragma unroll 1
                for (int ks = 0; ks < 4; ks++) {
                    const uint64_t b3 = smem_desc_sw128(st + kOffMma3 + ks * 2048, 8192, 1024);
                    mma_ts(tmem + (s ? kTmS : tm_o(0)), tmem + kTmDh + 8 * ks, b3, id3, 1);
                }
                mma_commit(sm.bar(kBarMma3));
                KDA_PHASE(1, item, 13);
                KDA_PHASE(1, item, 3);
            }
            // every MMA of this chunk is done: Km and B are free, O^T is final
            ok = mbar_wait(sm.bar(kBarMma3), item & 1, sm.abort_flag());
            if (role_any(!ok, kBarChain, kChainThreads)) { if (v == 0) record_error(p, sm, kErrWaitTimeout); return; }
            if (v == 0) {
                KDA_PHASE(1, item, 4);
                mbar_arrive(sm.bar(kBarKmFree + s));
            }
            tc_fence_after();
            chain_store_out(p, sm, maps, tmem, s, row0, L, un.h, v, item);
            if (v == 0) o_pending = s;
            if (v == 0) KDA_PHASE(1, item, 5);
        }
#ifdef KDA_TRACE
        if (v == 0 && blockIdx.x < 1024) { g_kda_cta[blockIdx.x][2] = item; g_kda_cta[blockIdx.x][3] = k + 1; }
#endif
        // unit end: the last chunk's output copies have read the tile buffers
        // (then TMEM P_s and the buffers go back to the prep at once), and the
        // final state = S * pend of the unit's last chunk leaves from TMEM
        if (v == 0 && o_pending >= 0) {
            bulk_wait_read0();
            mbar_arrive(sm.bar(kBarODone + o_pending));
            o_pending = -1;
        }
        named_bar(kBarChain, kChainThreads);
        if (p.s1)
            chain_store_state(p.s1 + warp_rows(un), sm.ptr<float>(kOffPend) + ((item - 1) % 3) * 128,
                              tmem + kTmS + lane_off, v & 31);
    }
}

template <bool kSlots, int kSort>
__device__ void chain_role(const TcParams &p, const Smem &sm, const int *order, int U, const Maps &maps)
{
    const int v = threadIdx.x;
    const int w = v >> 5;
    const uint32_t tmem = *sm.tmem_base();
    const uint32_t lane_off = (uint32_t)(32 * w) << 16;
    LoadCursor cur;
    bool kq_pending = false;
    if (v == 0) {
        for (int i = 0; i < 2 && cursor_next<kSlots, kSort>(cur, p, sm, order, U); i++) {
            issue_kq(sm, maps, cur.item - 1, cur.row0, cur.un.h, (cur.item - 1) & 1);
            issue_v(sm, maps, cur.item - 1, cur.row0, cur.un.h);
        }
    }
    chain_units<kSlots, kSort>(p, sm, order, U, maps, cur, kq_pending, tmem, lane_off, v);
    if (v == 0) {
        bulk_wait0();   // the output copies are complete
        // copies still in flight land before the CTA exits: normally none (every
        // requested chunk has been consumed); after a wait ran out, up to the
        // last two requested chunks (the k and q of the last one only if issued)
        for (int back = 1; back <= 2 && cur.item - back >= 0; back++) {
            const int it = cur.item - back;
            if (!(back == 1 && kq_pending)) mbar_wait_drain(sm.bar(kBarKQFull + (it & 1)), (it >> 1) & 1);
            mbar_wait_drain(sm.bar(kBarVFull + (it & 1)), (it >> 1) & 1);
        }
    }
}

// =============================================================================
// split mode
// =============================================================================
// Bounded wait, by one thread, until another CTA's flag reaches `target`
// (acquire).  Gives up after about a second, or at once when this CTA or the
// launch is winding down; false then.
__device__ bool flag_wait(const int *flag, int target, const SplitParams &sp, volatile int *abort, int *seen = nullptr)
{
    for (uint32_t it = 0; it < (1u << 22); it++) {
        const int x = ld_acquire_gpu(flag);
        if (x >= target) {
            if (seen) *seen = x;
            return true;
        }
        if ((it & 15) == 15 && (*abort || *reinterpret_cast<volatile int *>(sp.abort))) return false;
        __nanosleep(it < 64 ? 32 : 256);
    }
    return false;
}

// a wait on another CTA ran out, or this CTA is winding down: every CTA of the
// launch stops waiting for the others
__device__ __forceinline__ void split_abort(const TcParams &p, const SplitParams &sp, const Smem &sm)
{
    record_error(p, sm, kErrWaitTimeout);
    atomicExch(sp.abort, 1);
}

// A producer's warps 0-3 (the chain's place in the fused kernel): once a stage
// is finished -- -W' and Qp in its k/q rows, beta*V, Km and tril(A_qk)^T, T in
// its T16 buffer, the decay constants written -- and the ring slot of its
// chunk is free, copy it there in three groups, in the order the chunk two
// ahead needs the regions back (v, which group E reads first; k and q; the
// rest), request that chunk's v and its k and q as soon as their regions have
// been read, hand the stage back to the prep roles, and publish the slot.
template <bool kSlots, bool kHalf>
__device__ void ship_role(const TcParams &p, const SplitParams &sp, const Smem &sm, const int *order,
                          const Maps &maps)
{
    const int v = threadIdx.x;
    LoadCursor cur;
    if (v == 0) {
        for (int i = 0; i < 2 && cursor_next<kSlots, kSortChunks>(cur, p, sm, order, 0); i++) {
            issue_kq(sm, maps, cur.item - 1, cur.row0, cur.un.h, layout_bit<kSortChunks>(order, cur.un, 0));
            issue_v(sm, maps, cur.item - 1, cur.row0, cur.un.h);
        }
    }
    bool failed = false;
    for (int item = 0;; item++) {
        const int u = cta_unit<kSortChunks>(sm, item, 0);
        if (u < 0) break;
        const int s = item & 1;
        const uint32_t ph = (item >> 1) & 1;
        const int j = u >> 8, uu = u & 255;
        const int slot = uu * kRingSlots + j % kRingSlots;
        if (v == 0) KDA_PHASE(1, item, 0);
#ifdef KDA_TRACE
        if (v == 0 && blockIdx.x == KDA_TRACE_CTA && item < 128) g_kda_trace[1][item][15] = (unsigned long long)u;
#endif
        bool ok = mbar_wait(sm.bar(kBarFmReady + s), ph, sm.abort_flag()) &&
                  mbar_wait(sm.bar(kBarWReady + s), ph, sm.abort_flag());
        if (v == 0) KDA_PHASE(1, item, 1);
        // the chain has read the chunk kRingSlots back from this slot (half
        // chains: both have counted every chunk of the slot up to that one)
        if (ok && v == 0 && j >= kRingSlots)
            ok = flag_wait(sp.freed + slot * kFlagSlotStride, kHalf ? 2 * (j / kRingSlots) : j - kRingSlots + 1, sp,
                           sm.abort_flag());
        if (role_any(!ok, kBarChain, kChainThreads)) {
            failed = true;
            break;
        }
        if (v == 0) KDA_PHASE(1, item, 2);
        uint8_t *dst = sp.ring + (size_t)slot * kSlotBytes;
        float *hdr = reinterpret_cast<float *>(dst + kSlotHdr);
        hdr[v] = sm.ptr<float>(kOffConst + s * kConstBytes)[v];          // fm: view from the middle row
        hdr[128 + v] = sm.ptr<float>(kOffPend)[(item % 3) * 128 + v];    // pend: middle row -> last row
        if (v == 0) {
            const uint32_t st = sm.u32(s * kStageBytes);
            bulk_store(dst + kOffV, st + kOffV, kVBytes);                    // group 1: beta*V
            bulk_commit();
            bulk_store(dst + kOffKQ, st + kOffKQ, 16384);                    // group 2: -W' and Qp
            bulk_store(dst + kOffKQ + 16384, st + kOffKQ + 16384, 16384);
            bulk_commit();
            bulk_store(dst + kOffMma3, st + kOffMma3, 16384);                // group 3: Km, tril(A_qk)^T, T16
            bulk_store(dst + kOffMma3 + 16384, st + kOffMma3 + 16384, kStageBytes - kOffMma3 - 16384);
            bulk_store(dst + kSlotT16, sm.u32(t16_off<true>(s)), 8192);
            bulk_commit();
            const bool more = cursor_next<kSlots, kSortChunks>(cur, p, sm, order, 0);
            bulk_wait_read2();
            if (more) issue_v(sm, maps, cur.item - 1, cur.row0, cur.un.h);
            bulk_wait_read1();
            if (more)
                issue_kq(sm, maps, cur.item - 1, cur.row0, cur.un.h, layout_bit<kSortChunks>(order, cur.un, 0));
            bulk_wait_read0();
            KDA_PHASE(1, item, 3);
            // the stage is the prep's again: Km and tril(A_qk)^T, TMEM P_s
            mbar_arrive(sm.bar(kBarKmFree + s));
            mbar_arrive(sm.bar(kBarODone + s));
            bulk_wait0();
            KDA_PHASE(1, item, 4);
        }
        // every thread's header stores and thread 0's copies are done; one
        // release after the block barrier publishes them all
        named_bar(kBarChain, kChainThreads);
        if (v == 0) {
            __threadfence();
            fence_proxy_async_global();
            st_release_gpu(sp.ready + slot * kFlagSlotStride, 2 * (j + 1) + (j & 1));   // + the stage's layout bit
            KDA_PHASE(1, item, 5);
        }
    }
    if (v == 0) {
        if (failed) split_abort(p, sp, sm);
        bulk_wait0();
        // loads still in flight land before the CTA exits (normally none: every
        // requested chunk was consumed)
        for (int back = 1; back <= 2 && cur.item - back >= 0; back++) {
            const int it = cur.item - back;
            mbar_wait_drain(sm.bar(kBarKQFull + (it & 1)), (it >> 1) & 1);
            mbar_wait_drain(sm.bar(kBarVFull + (it & 1)), (it >> 1) & 1);
        }
    }
}

// ---- the split chain: one unit, 16 compute warps -------------------------------
// Warp w owns TMEM lanes 32 (w % 4) .. +31 (value channels) and the quarter
// cg = w / 4 of each lane's columns.  States move as in chain_load_state /
// chain_store_state, in the 16x256b fragment layout, here over the warp's 32
// columns and its kRows rows: 32, or 16 in a half chain (its rows sit in lanes
// 0-15 of the warp's 32).
template <int kRows>
__device__ void split_load_state(const float *src, uint32_t tm, int lane, int cg)
{
    const int rr = lane >> 2, cc = 2 * (lane & 3);
#pragma unroll
    for (int gi = 0; gi < kRows / 16; gi++) {
        uint32_t x[16];
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const float *r0 = src ? src + (16 * gi + rr) * kD + 32 * cg + 8 * b + cc : nullptr;
            const float2 lo = r0 ? *reinterpret_cast<const float2 *>(r0) : make_float2(0.f, 0.f);
            const float2 hi = r0 ? *reinterpret_cast<const float2 *>(r0 + 8 * kD) : make_float2(0.f, 0.f);
            x[4 * b] = __float_as_uint(lo.x); x[4 * b + 1] = __float_as_uint(lo.y);
            x[4 * b + 2] = __float_as_uint(hi.x); x[4 * b + 3] = __float_as_uint(hi.y);
        }
        tmem_st16x256_x4(tm + ((uint32_t)(16 * gi) << 16) + 32 * cg, x);
    }
    tmem_wait_st();
}

template <int kRows>
__device__ void split_store_state(float *dst, const float *pend, uint32_t tm, int lane, int cg)
{
    const int rr = lane >> 2, cc = 2 * (lane & 3);
#pragma unroll
    for (int gi = 0; gi < kRows / 16; gi++) {
        uint32_t x[16];
        tmem_ld16x256_x4(tm + ((uint32_t)(16 * gi) << 16) + 32 * cg, x);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const float2 pe = *reinterpret_cast<const float2 *>(pend + 32 * cg + 8 * b + cc);
            float *r0 = dst + (16 * gi + rr) * kD + 32 * cg + 8 * b + cc;
            *reinterpret_cast<float2 *>(r0) =
                make_float2(__fmul_rn(__uint_as_float(x[4 * b]), pe.x), __fmul_rn(__uint_as_float(x[4 * b + 1]), pe.y));
            *reinterpret_cast<float2 *>(r0 + 8 * kD) =
                make_float2(__fmul_rn(__uint_as_float(x[4 * b + 2]), pe.x), __fmul_rn(__uint_as_float(x[4 * b + 3]), pe.y));
        }
    }
}

// S <- (S * pend) * fm on this warp's 32 columns, and their fp16 copy S'h (the
// arithmetic of chain_scale_state)
__device__ __forceinline__ void split_scale_state(uint32_t tmem, uint32_t lane_off, int cg, const float *fm,
                                                  const float *pend)
{
    uint32_t x[32];
    tmem_ld32(tmem + kTmS + lane_off + 32 * cg, x);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 f4 = *reinterpret_cast<const float4 *>(fm + 32 * cg + j);
        const float4 p4 = pend ? *reinterpret_cast<const float4 *>(pend + 32 * cg + j) : make_float4(1.f, 1.f, 1.f, 1.f);
        float2 lo = make_float2(__uint_as_float(x[j]), __uint_as_float(x[j + 1]));
        float2 hi = make_float2(__uint_as_float(x[j + 2]), __uint_as_float(x[j + 3]));
        if (pend) {
            lo = fmul2(lo, make_float2(p4.x, p4.y));
            hi = fmul2(hi, make_float2(p4.z, p4.w));
        }
        lo = fmul2(lo, make_float2(f4.x, f4.y));
        hi = fmul2(hi, make_float2(f4.z, f4.w));
        x[j] = __float_as_uint(lo.x); x[j + 1] = __float_as_uint(lo.y);
        x[j + 2] = __float_as_uint(hi.x); x[j + 3] = __float_as_uint(hi.y);
    }
    uint32_t h[16];
#pragma unroll
    for (int j = 0; j < 16; j++) h[j] = pack_f16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
    tmem_st32(tmem + kTmS + lane_off + 32 * cg, x);
    tmem_st16(tmem + kTmS0h + lane_off + 16 * cg, h);
}

// The same for a half chain (M = 64: value row i in TMEM lane
// (i % 16) + 32 (i / 16), so the 16 rows of sub-partition q sit in its lanes
// 0-15): this warp's 16 rows x 32 columns in the 16x256b fragment layout
// (thread t: rows t/4 and 8 + t/4, columns 8b + 2 (t%4), +1), and the fp16
// copy in the 16x128b layout, where thread t writes exactly the packed columns
// 4b + t%4 of those two rows -- the pairs it holds.
__device__ __forceinline__ void split_scale_state_half(uint32_t tmem, uint32_t lane_off, int cg, const float *fm,
                                                       const float *pend, int lane)
{
    uint32_t x[16];
    tmem_ld16x256_x4(tmem + kTmS + lane_off + 32 * cg, x);
    tmem_wait_ld();
    const int c0 = 32 * cg + 2 * (lane & 3);
#pragma unroll
    for (int b = 0; b < 4; b++) {
        const float2 f2 = *reinterpret_cast<const float2 *>(fm + c0 + 8 * b);
        const float2 p2 = pend ? *reinterpret_cast<const float2 *>(pend + c0 + 8 * b) : make_float2(1.f, 1.f);
        const float fv[2] = {f2.x, f2.y}, pv[2] = {p2.x, p2.y};
#pragma unroll
        for (int hr = 0; hr < 2; hr++)
#pragma unroll
            for (int e = 0; e < 2; e++) {
                float f = __uint_as_float(x[4 * b + 2 * hr + e]);
                if (pend) f = __fmul_rn(f, pv[e]);
                x[4 * b + 2 * hr + e] = __float_as_uint(__fmul_rn(f, fv[e]));
            }
    }
    uint32_t h[8];
#pragma unroll
    for (int b = 0; b < 4; b++) {
        h[2 * b] = pack_f16x2(__uint_as_float(x[4 * b]), __uint_as_float(x[4 * b + 1]));
        h[2 * b + 1] = pack_f16x2(__uint_as_float(x[4 * b + 2]), __uint_as_float(x[4 * b + 3]));
    }
    tmem_st16x256_x4(tmem + kTmS + lane_off + 32 * cg, x);
    tmem_st16x128_x4(tmem + kTmS0h + lane_off + 16 * cg, h);
}

// Chain CTA of unit uu, warp 16 (its first lane): the slot copies.  Chunk j
// goes into buffer j & 1 once the producers have published it (the flag is
// awaited ahead of time) and the chain's MMAs of chunk j - 2 are done with the
// buffer -- the part MMA1 reads as soon as MMA1 is done, the rest after MMA3;
// once chunk j has landed, its ring slot goes back to the producers.  (Done by the chain's own first
// thread, the flag round trips cost about 3.7k cycles a chunk on its path.)
template <bool kSlots, bool kHalf>
__device__ void split_loader(const TcParams &p, const SplitParams &sp, const Smem &sm, const int *order, int uu)
{
    const Unit un = get_unit<kSlots, 1>(p, order, uu);
    const int nch = un.nchunks;
    auto slot_of = [&](int j) { return uu * kRingSlots + j % kRingSlots; };
    int issued_a = 0, issued_b = 0, landed = 0;
    // part A of chunk j (k/q rows, beta*V, T16, the decay constants): what MMA-b,
    // the rescale and MMA1 read; part B (Km, tril(A_qk)^T): what MMA3 reads
    auto copy = [&](int j, uint32_t off, uint32_t bytes, uint32_t bar) {
        const uint32_t dst = sm.u32((j & 1) * kSlotBytes);
        const uint8_t *src = sp.ring + (size_t)slot_of(j) * kSlotBytes;
        for (uint32_t o = off; o < off + bytes; o += 16384)
            bulk_load(dst + o, src + o, off + bytes - o < 16384u ? off + bytes - o : 16384u, bar);
    };
    int par_next = 0;   // layout bit of the chunk whose ready flag was seen last
    auto await_ready = [&](int j) -> bool {
        int val = 0;
        KDA_PHASE(2, j, 0);
        if (!flag_wait(sp.ready + slot_of(j) * kFlagSlotStride, 2 * (j + 1), sp, sm.abort_flag(), &val)) return false;
        KDA_PHASE(2, j, 1);
        fence_proxy_async_global();
        par_next = val & 1;
        return true;
    };
    auto issue_a = [&](int j) {   // (buffer j & 1 is free: its layout bit may change now)
        sm.split_parity()[j & 1] = par_next;   // read by the chain after the part A barrier
        const uint32_t bar = sm.bar(kBarKQFull + (j & 1));
        mbar_arrive_expect_tx(bar, kOffMma3 + (kSlotBytes - kSlotT16));
        copy(j, 0, kOffMma3, bar);
        copy(j, kSlotT16, kSlotBytes - kSlotT16, bar);
        issued_a = j + 1;
    };
    auto issue_b = [&](int j) {
        const uint32_t bar = sm.bar(kBarVFull + (j & 1));
        mbar_arrive_expect_tx(bar, kSlotT16 - kOffMma3);
        copy(j, kOffMma3, kSlotT16 - kOffMma3, bar);
        issued_b = j + 1;
    };
    bool ok = true;
    for (int j = 0; ok && j < 2 && j < nch; j++) {
        ok = await_ready(j);
        if (ok) { issue_a(j); issue_b(j); }
    }
    for (int j = 0; ok && j < nch; j++) {
        const int b = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        ok = mbar_wait(sm.bar(kBarKQFull + b), ph, sm.abort_flag()) && mbar_wait(sm.bar(kBarVFull + b), ph, sm.abort_flag());
        if (!ok) break;
        KDA_PHASE(2, j, 2);
        landed = j + 1;
        // the slot may take chunk j + kRingSlots (a unit of half chains: once both
        // have counted it)
        if constexpr (kHalf) red_release_add_gpu(sp.freed + slot_of(j) * kFlagSlotStride, 1);
        else st_release_gpu(sp.freed + slot_of(j) * kFlagSlotStride, j + 1);
        if (j + 2 < nch) {
            // chunk j + 2 into buffer b: part A once MMA1 of chunk j is done with it,
            // part B once MMA3 is
            ok = await_ready(j + 2) && mbar_wait(sm.bar(kBarAFull + b), ph, sm.abort_flag());
            if (!ok) break;
            issue_a(j + 2);
            ok = mbar_wait(sm.bar(kBarKmFree + b), ph, sm.abort_flag());
            if (!ok) break;
            issue_b(j + 2);
        }
    }
    if (!ok) split_abort(p, sp, sm);
    // copies still in flight land before the CTA exits
    for (int j = landed; j < issued_a; j++) mbar_wait_drain(sm.bar(kBarKQFull + (j & 1)), (j >> 1) & 1);
    for (int j = landed; j < issued_b; j++) mbar_wait_drain(sm.bar(kBarVFull + (j & 1)), (j >> 1) & 1);
}

// The split chain's two block barriers per chunk (compute warps and the MMA
// issuer warp) and the mbarriers the issuer commits to (named barrier ids and
// mbarrier slots of the chain CTA; kBarKmFree[b] marks buffer b free).
constexpr int kBarSplitSync = 4;                       // named barrier: 16 compute warps + the issuer
constexpr int kSplitSyncThreads = kThreads + 32;
constexpr int kBarM1D = kBarMma1;                      // MMA1's Delta half done (and every MMA before it)
constexpr int kBarM3S = kBarMma3;                      // MMA3's state half done
constexpr int kBarM3O = kBarPrepDone;                  // MMA3's output half done

// Chain CTA of unit uu, warp 17: the MMA issuer (its first lane issues, the
// whole warp joins the block barriers).  Per chunk j, in this order on the
// tensor pipe: MMA-b's U half of chunk j (once the chunk has landed), then --
// after the compute warps' rescale -- MMA1's Delta half and its output half,
// then -- after their Delta conversion -- MMA3's state half and its output
// half.  The halves are the fused kernel's N = 128 MMA1 and N = 192 MMA3
// split by their B rows (K rows / Q rows; Km / tril(A_qk)^T), so that the
// compute warps can go on as soon as the half they need is done.
template <bool kSlots, bool kHalf>
__device__ void split_issuer(const TcParams &p, const Smem &sm, const int *order, int uu, int half)
{
    constexpr int M = kHalf ? 64 : 128;   // a half chain: value channels 64 half .. +63
    const int lane = threadIdx.x & 31;
    const uint32_t tmem = *sm.tmem_base();
    const Unit un = get_unit<kSlots, 1>(p, order, uu);
    const int nch = un.nchunks;
    if (nch == 0) return;
    bool ok = true;
    auto mma_b = [&](int j) {   // U^T = (beta V)^T T^T into chunk j's Delta columns
        const int b = j & 1, par = sm.split_parity()[b];
        const uint32_t buf = sm.u32(b * kSlotBytes);
        const uint32_t id = idesc_f16(M, 64, 1, 0);
#pragma unroll
        for (int ks = 0; ks < 4; ks++) {
            const uint64_t bd = smem_desc_sw128(buf + kSlotT16 + ks * 32, 16, 1024);
            const uint64_t au = smem_desc_sw128(buf + kOffV + 8192 * half + ks * 2048, 8192, 1024);
            mma_ss(tmem + tm_d(par), au, bd, id, ks > 0);
        }
    };
    if (lane == 0) {
        ok = mbar_wait(sm.bar(kBarKQFull), 0, sm.abort_flag());
        tc_fence_after();
        if (ok) mma_b(0);
    }
    for (int j = 0; j < nch; j++) {
        const int b = j & 1;
        if (role_any(!ok, kBarSplitSync, kSplitSyncThreads)) break;   // the rescale is done
        if (lane == 0) KDA_PHASE(0, j, 0);
        if (lane == 0) {
            const int par = sm.split_parity()[b];
            const uint32_t buf = sm.u32(b * kSlotBytes);
            tc_fence_after();
            const uint32_t id = idesc_f16(M, 64, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {   // U^T - S'^T W'^T: the K rows hold -W'
                const int kb = ks >> 2, kin = ks & 3;
                mma_ts(tmem + tm_d(par), tmem + kTmS0h + 8 * ks,
                       smem_desc_sw128(buf + kOffKQ + kb * 16384 + off_k(par) + kin * 32, 16, 1024), id, 1);
            }
            mma_commit(sm.bar(kBarM1D));
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {   // S'^T Qp^T: the Q rows
                const int kb = ks >> 2, kin = ks & 3;
                mma_ts(tmem + tm_o(par), tmem + kTmS0h + 8 * ks,
                       smem_desc_sw128(buf + kOffKQ + kb * 16384 + off_q(par) + kin * 32, 16, 1024), id, ks > 0);
            }
            mma_commit(sm.bar(kBarAFull + b));   // MMA-b and MMA1 are done with part A of buffer b
        }
        if (role_any(!ok, kBarSplitSync, kSplitSyncThreads)) break;   // Delta is in fp16
        if (lane == 0) KDA_PHASE(0, j, 1);
        if (lane == 0) {
            const int par = sm.split_parity()[b];
            const uint32_t buf = sm.u32(b * kSlotBytes);
            ok = mbar_wait(sm.bar(kBarVFull + b), (j >> 1) & 1, sm.abort_flag());   // part B (Km, tril(A_qk)^T)
            tc_fence_after();
            if (ok) {
#pragma unroll
            for (int ks = 0; ks < 4; ks++)     // S^T += Delta^T Km
                mma_ts(tmem + kTmS, tmem + kTmDh + 8 * ks,
                       smem_desc_sw128(buf + off_km(par) + ks * 2048, 8192, 1024), idesc_f16(M, 128, 0, 1), 1);
            }
            mma_commit(sm.bar(kBarM3S));   // (also when nothing was issued: the compute warps' wait ends)
            if (ok) {
#pragma unroll
            for (int ks = 0; ks < 4; ks++)     // O^T += Delta^T tril(A_qk)^T
                mma_ts(tmem + tm_o(par), tmem + kTmDh + 8 * ks,
                       smem_desc_sw128(buf + off_bq(par) + ks * 2048, 8192, 1024), idesc_f16(M, 64, 0, 1), 1);
            }
            mma_commit(sm.bar(kBarM3O));
            mma_commit(sm.bar(kBarKmFree + b));   // every MMA reading buffer b is done: it may take chunk j + 2
            KDA_PHASE(0, j, 2);
            if (ok && j + 1 < nch) {
                ok = mbar_wait(sm.bar(kBarKQFull + (b ^ 1)), ((j + 1) >> 1) & 1, sm.abort_flag());
                tc_fence_after();
                if (ok) mma_b(j + 1);
                KDA_PHASE(0, j, 3);
            }
        }
    }
}

// Chain CTA of unit uu (sorted order), the 16 compute warps.  Per chunk j
// (slot buffer b = j & 1; the layout bit `par` of the chunk, alternating
// from chunk to chunk, fixes where K and Q rows, Km and tril(A_qk)^T sit and
// so which TMEM columns take Delta and O):
//   the state is rescaled (S' = S pend fm, and its fp16 copy);
//   [block barrier: the issuer starts MMA1, Delta half first]
//   chunk j-1's outputs leave (O^T -> bf16 -> out), while MMA1 runs;
//   Delta^T -> fp16 once MMA1's Delta half is done;
//   [block barrier: the issuer starts MMA3, state half first]
//   the next chunk starts once MMA3's state half is done.
// The arithmetic, operand for operand, is the fused kernel's.  A half chain
// (kHalf) keeps value channels 64 half .. +63 of the unit, with M = 64 MMAs:
// row i of its accumulators in TMEM lane (i % 16) + 32 (i / 16), so warp w
// holds rows 16 (w % 4) .. +15 in lanes 0-15 of its sub-partition, and moves
// half the TMEM bytes a chunk of a whole chain.
template <bool kSlots, bool kHalf>
__device__ void split_chain(const TcParams &p, const SplitParams &sp, const Smem &sm, const int *order,
                            const Maps &maps, int uu, int half)
{
    constexpr int kRows = kHalf ? 16 : 32;                // state rows of a warp
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int q = w & 3, cg = w >> 2;
    const uint32_t tmem = *sm.tmem_base();
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const Unit un = get_unit<kSlots, 1>(p, order, uu);
    const size_t ubase = ((size_t)un.st * p.H + un.h) * kD * kD;   // used only when st >= 0
    const size_t hbase = ubase + (size_t)(kHalf ? 64 * half : 0) * kD;   // this chain's first state row
    if (un.nchunks == 0) {   // empty (or padded) sequence: its state rows pass through
        if (p.s1 && (!kSlots || un.st >= 0))
            for (int i = tid; i < 4 * kRows * kD / 4; i += kThreads)
                reinterpret_cast<float4 *>(p.s1 + hbase)[i] =
                    p.s0 ? reinterpret_cast<const float4 *>(p.s0 + hbase)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int nch = un.nchunks;
    float *pendr = sm.ptr<float>(kCPend);                     // [2][128]: pend of the last two chunks
    const size_t wrows = hbase + (size_t)(kRows * q) * kD;   // this warp's first state row
    bool ok = true;
    split_load_state<kRows>(p.s0 ? p.s0 + wrows : nullptr, tmem + kTmS + lane_off, lane, cg);
    // O^T of chunk jo (layout paro) -> bf16 tiles of 32 rows in staging buffer
    // jo & 1 (this warp: rows 16 cg .. +15, its 32 value channels; 16 in a
    // half chain, whose tiles hold its 64 channels only), stored by bulk
    // tensor copies; partial tiles row by row.  Thread 0 has made sure before
    // (bulk_wait_read1 ahead of a block barrier) that the copies of chunk
    // jo - 2 have read the buffer.  false: a thread's wait ran out.
    constexpr int kTileBytes = kHalf ? 4096 : 8192;   // one tile: 32 rows x the chain's channels
    auto outputs = [&](int jo, int paro) -> bool {
        ok = mbar_wait(sm.bar(kBarM3O), jo & 1, sm.abort_flag()) && ok;   // MMA3's output half of chunk jo
        tc_fence_after();
        const int row0 = un.bos + jo * kChunk, L = min(kChunk, un.eos - row0);
        const uint32_t ost = sm.u32(kCOut + (jo & 1) * 16384);
        constexpr int kHl = kHalf ? 1 : 2;   // 16-lane halves of the warp's lanes that hold rows
        uint32_t o[kHl][8];
        const uint32_t src = tmem + tm_o(paro) + lane_off;
#pragma unroll
        for (int hl = 0; hl < kHl; hl++) tmem_ld16x256_x2(src + ((uint32_t)(16 * hl) << 16) + 16 * cg, o[hl]);
        tmem_wait_ld();
        tc_fence_before();
        const int mi = lane >> 3, k8 = lane & 7;
        const int rl = 16 * (cg & 1) + ((mi & 2) ? 8 : 0) + k8;
#pragma unroll
        for (int hl = 0; hl < kHl; hl++) {
            const uint32_t *f = o[hl];
            const int vc = kRows * q + 16 * hl + ((mi & 1) ? 8 : 0);   // the chain's channel
            stmatrix_x4_trans(ost + (cg >> 1) * kTileBytes + (vc >> 6) * 4096 + sw128_chunk(rl, (vc & 63) >> 3),
                              pack_bf16x2(__uint_as_float(f[0]), __uint_as_float(f[1])),
                              pack_bf16x2(__uint_as_float(f[2]), __uint_as_float(f[3])),
                              pack_bf16x2(__uint_as_float(f[4]), __uint_as_float(f[5])),
                              pack_bf16x2(__uint_as_float(f[6]), __uint_as_float(f[7])));
        }
        fence_proxy_async_smem();
        if (role_any(!ok, kBarChain, kThreads)) return false;
        const int blk = kHalf ? half : 0;   // the chain's first 64-channel block
        if (tid == 0) {
            if (L >= 32) tma_store_4d(maps.o, 0, row0, blk, un.h, ost);
            if (L == kChunk) tma_store_4d(maps.o, 0, row0 + 32, blk, un.h, ost + kTileBytes);
            bulk_commit();
            KDA_PHASE(1, jo, 10);
        }
        if (L < kChunk) {
            constexpr int kPieces = kTileBytes / 512;   // 16-byte pieces of a row
            const int tile = L < 32 ? 0 : 1, nr = L - 32 * tile;
            const uint8_t *tb = sm.base + kCOut + (jo & 1) * 16384 + tile * kTileBytes;
            const size_t row_stride = (size_t)p.H * kD;
            __nv_bfloat16 *dst = p.out + ((size_t)(row0 + 32 * tile) * p.H + un.h) * kD + 64 * blk;
            for (int idx = tid; idx < nr * kPieces; idx += kThreads) {
                const int r = idx / kPieces, pc = idx % kPieces;
                *reinterpret_cast<uint4 *>(dst + (size_t)r * row_stride + 8 * pc) =
                    *reinterpret_cast<const uint4 *>(tb + (pc >> 3) * 4096 + sw128_chunk(r, pc & 7));
            }
        }
        return true;
    };
    int consumed = 0, prev_par = 0;
    bool failed = false;
    for (int j = 0; j < nch; j++) {
        const int b = j & 1;
        if (tid == 0) KDA_PHASE(1, j, 0);
        ok = ok && mbar_wait(sm.bar(kBarKQFull + b), (j >> 1) & 1, sm.abort_flag());
        tc_fence_after();
        if (tid == 0) KDA_PHASE(1, j, 1);
        const int par = sm.split_parity()[b];
        const float *hdr = sm.ptr<float>(b * kSlotBytes + kSlotHdr);
        if constexpr (kHalf)
            split_scale_state_half(tmem, lane_off, cg, hdr, j > 0 ? pendr + ((j - 1) & 1) * 128 : nullptr, lane);
        else
            split_scale_state(tmem, lane_off, cg, hdr, j > 0 ? pendr + ((j - 1) & 1) * 128 : nullptr);
        if (tid == 0) KDA_PHASE(1, j, 11);
        if (tid < 128) pendr[(j & 1) * 128 + tid] = hdr[128 + tid];
        tmem_wait_st();
        tc_fence_before();
        if (tid == 0) KDA_PHASE(1, j, 12);
        if (tid == 0) bulk_wait_read1();   // chunk j-3's output copies have read staging buffer (j-1) & 1
        if (tid == 0) KDA_PHASE(1, j, 2);
        if (role_any(!ok, kBarSplitSync, kSplitSyncThreads)) { failed = true; break; }
        consumed = j + 1;
        if (tid == 0) KDA_PHASE(1, j, 3);
        // chunk j-1's outputs, while MMA1 of chunk j runs (it writes the other
        // layout's columns); a failure there is gathered at the next barrier
        // that the issuer also joins
        if (j > 0 && !outputs(j - 1, prev_par)) ok = false;
        if (tid == 0) KDA_PHASE(1, j, 4);
        ok = mbar_wait(sm.bar(kBarM1D), j & 1, sm.abort_flag(), KDA_WAIT_LIMIT_MMA1) && ok;
        tc_fence_after();
        if (tid == 0) KDA_PHASE(1, j, 5);
        if constexpr (kHalf) {   // the same on the warp's 16 lanes (layouts as in the rescale)
            uint32_t x[8], h[4];
            tmem_ld16x256_x2(tmem + tm_d(par) + lane_off + 16 * cg, x);
            tmem_wait_ld();
#pragma unroll
            for (int b = 0; b < 2; b++) {
                h[2 * b] = pack_f16x2(__uint_as_float(x[4 * b]), __uint_as_float(x[4 * b + 1]));
                h[2 * b + 1] = pack_f16x2(__uint_as_float(x[4 * b + 2]), __uint_as_float(x[4 * b + 3]));
            }
            tmem_st16x128_x2(tmem + kTmDh + lane_off + 8 * cg, h);
        } else {   // Delta^T (fp32) -> fp16 A operand, this warp's 16 columns
            uint32_t x[16], h[8];
            tmem_ld16(tmem + tm_d(par) + lane_off + 16 * cg, x);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; i++) h[i] = pack_f16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
            tmem_st8(tmem + kTmDh + lane_off + 8 * cg, h);
        }
        tmem_wait_st();
        tc_fence_before();
        if (role_any(!ok, kBarSplitSync, kSplitSyncThreads)) { failed = true; break; }
        if (tid == 0) KDA_PHASE(1, j, 6);
        ok = mbar_wait(sm.bar(kBarM3S), j & 1, sm.abort_flag());
        tc_fence_after();
        if (tid == 0) KDA_PHASE(1, j, 7);
        prev_par = par;
    }
    // the last chunk's outputs
    if (!failed) {
        if (tid == 0) bulk_wait_read1();
        named_bar(kBarChain, kThreads);
        if (!outputs(nch - 1, prev_par)) failed = true;
    }
    const bool any_failed = role_any(!ok || failed, kBarChain, kThreads);
    const bool done = consumed == nch && !any_failed;
    if (tid == 0) {
        if (!done) split_abort(p, sp, sm);
        bulk_wait_read0();
    }
    named_bar(kBarChain, kThreads);
    // the final state = S * pend of the last chunk, straight from TMEM
    if (done && p.s1)
        split_store_state<kRows>(p.s1 + wrows, pendr + ((nch - 1) & 1) * 128, tmem + kTmS + lane_off, lane, cg);
    if (tid == 0) bulk_wait0();
}

// =============================================================================
// The split-mode kernel: a cooperative launch of one CTA per SM (every CTA
// resident at once, so that the chains and the producers can wait on one
// another); CTA b < sp.chains runs the chain of unit b (sorted order) -- with
// half chains, half b & 1 of unit b / 2 -- and the others prepare chunks.
constexpr int kSplitThreads = kThreads + 64;   // + the chain CTAs' loader warp and MMA issuer warp

template <bool kSlots, bool kHalf>
__global__ void __launch_bounds__(kSplitThreads, 1)
kda_tc_split_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                    const __grid_constant__ CUtensorMap to, TcParams p, const __grid_constant__ SplitParams sp)
{
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    sm.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool chain = (int)blockIdx.x < sp.chains;
    int *order = sm.ptr<int>(kOffOrder);
    if (tid == 0) {
        *sm.abort_flag() = 0;
        for (int i = 0; i < 2; i++) {
            mbar_init(sm.bar(kBarKQFull + i), 1);
            mbar_init(sm.bar(kBarVFull + i), 1);
            mbar_init(sm.bar(kBarPrepDone + i), 1);
            mbar_init(sm.bar(kBarAFull + i), 1);
            mbar_init(sm.bar(kBarEDone + i), kEThreads);
            mbar_init(sm.bar(kBarODone + i), 1);
            mbar_init(sm.bar(kBarFmReady + i), kGroupThreads);
            mbar_init(sm.bar(kBarKmFree + i), 1);
            mbar_init(sm.bar(kBarWReady + i), kGroupThreads);
        }
        mbar_init(sm.bar(kBarGFull), 1);
        mbar_init(sm.bar(kBarMma1), 1);
        mbar_init(sm.bar(kBarMma3), 1);
        mbar_init(sm.bar(kBarDrain), 4);   // + the chain CTAs' MMA issuer (warp 17)
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(sm.u32(kOffMisc), kTmCols);
        tmem_relinquish();
        if ((tid & 31) == 0) {
            tma_prefetch_desc(&tq); tma_prefetch_desc(&tk); tma_prefetch_desc(&tv); tma_prefetch_desc(&tg);
            tma_prefetch_desc(&to);
        }
    }
    {   // sequences sorted by length, longest first (ties: lower index), as in the fused kernel
        int *lens = sm.ptr<int>(kOffP);
        int2 *rows = reinterpret_cast<int2 *>(order + kMaxSortedSeqs);
        for (int n = tid; n < p.N; n += kSplitThreads) {
            const int cb = p.cu[n], ce = p.cu[n + 1];
            int b = min(max(cb, 0), p.T), e = min(max(ce, 0), p.T);
            if (cb < 0 || cb > p.T || ce < 0 || ce > p.T) atomicOr(p.err, kErrBadSeqlens);
            if (e < b || (kSlots && state_index<kSlots>(p, n) < 0)) e = b;
            rows[n] = make_int2(b, e);
            lens[n] = e - b;
        }
        __syncthreads();
        for (int n = tid; n < p.N; n += kSplitThreads) {
            int rank = 0;
            const int ln = lens[n];
            for (int m2 = 0; m2 < p.N; m2++) {
                const int lm = lens[m2];
                rank += (lm > ln) || (lm == ln && m2 < n);
            }
            order[rank] = n;
        }
        __syncthreads();
        if (tid == 0 && !chain) {
            // the producers' deal: claim i = chunk j of unit u, chunk index first;
            // CTA b starts with claim b - chains, the rest come from the counter
            int total = 0;
            for (int n = 0; n < p.N; n++) total += (lens[n] + kChunk - 1) / kChunk;
            total *= p.H;
            const int i0 = (int)blockIdx.x - sp.chains;
            *sm.units_nonempty() = total;
            *sm.producers() = (int)gridDim.x - sp.chains;
            ChunkDeal deal;
            const bool first = i0 < total;
            sm.sched()[0] = first ? deal.decode(order, p.N, p.H, i0) : -1;
            *sm.published() = first ? 1 : 0;
            *sm.claim_done() = first ? 0 : 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const Maps maps = {&tq, &tk, &tv, &tg, &to};
    const int cu_ = kHalf ? (int)blockIdx.x >> 1 : (int)blockIdx.x, half = kHalf ? (int)blockIdx.x & 1 : 0;
    if (warp == 16) {
        if (chain && tid == kThreads) split_loader<kSlots, kHalf>(p, sp, sm, order, cu_);
    } else if (warp == 17) {
        if (chain) split_issuer<kSlots, kHalf>(p, sm, order, cu_, half);
    } else if (chain) {
        split_chain<kSlots, kHalf>(p, sp, sm, order, maps, cu_, half);
    } else if (warp < 4) {
        ship_role<kSlots, kHalf>(p, sp, sm, order, maps);
    } else if (warp < 12) {
        const ConvParams no_conv = {};
        e_role<kSlots, kSortChunks, false>(p, no_conv, sm, order, 0, maps);
    } else {
        i_role<kSlots, kSortChunks, false>(p, nullptr, sm, order, 0);
    }
    // every MMA this CTA issued has completed before TMEM is released
    if (tid == 0 || tid == kChainThreads || tid == kChainThreads + kEThreads || tid == kThreads + 32) {
        mma_commit(sm.bar(kBarDrain));
        mbar_wait_drain(sm.bar(kBarDrain), 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(*sm.tmem_base(), kTmCols);
    // the last CTA to finish returns the deal's scratch slot to zero
    if (tid == 0 && p.sched) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

// =============================================================================
template <bool kSlots, int kSort, bool kConv>
__global__ void __launch_bounds__(kThreads, 1)
kda_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
              const __grid_constant__ CUtensorMap to, TcParams p, const __grid_constant__ ConvParams cp)
{
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    sm.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int U = p.N * p.H;
    int *order = sm.ptr<int>(kOffOrder);

    // Launched with programmatic stream serialisation, this CTA may start while
    // the kernel before it on the stream is still running: the set-up below
    // (barriers, TMEM, tensor maps) touches no global memory; griddepcontrol.wait
    // then holds every thread until that kernel has completed and its writes
    // are visible, before the first global access.  launch_dependents lets the
    // next kernel's CTAs be placed as SMs free up.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        *sm.abort_flag() = 0;
        for (int i = 0; i < 2; i++) {
            mbar_init(sm.bar(kBarKQFull + i), 1);
            mbar_init(sm.bar(kBarVFull + i), 1);
            mbar_init(sm.bar(kBarPrepDone + i), 1);
            mbar_init(sm.bar(kBarAFull + i), 1);
            mbar_init(sm.bar(kBarEDone + i), kEThreads);
            mbar_init(sm.bar(kBarODone + i), 1);
            mbar_init(sm.bar(kBarFmReady + i), kGroupThreads);
            mbar_init(sm.bar(kBarKmFree + i), 1);
            mbar_init(sm.bar(kBarWReady + i), kGroupThreads);
        }
        mbar_init(sm.bar(kBarGFull), 1);
        mbar_init(sm.bar(kBarMma1), 1);
        mbar_init(sm.bar(kBarMma3), 1);
        mbar_init(sm.bar(kBarDrain), 3);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(sm.u32(kOffMisc), kTmCols);
        tmem_relinquish();
        if ((tid & 31) == 0) {
            tma_prefetch_desc(&tq); tma_prefetch_desc(&tk); tma_prefetch_desc(&tv); tma_prefetch_desc(&tg);
            tma_prefetch_desc(&to);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // schedule: sequences sorted by length, longest first (ties: lower index), dealt
    // dynamically: CTA b starts with the b-th longest unit; the rest of the
    // nonempty units (longest first) go to whichever CTA claims them next, so
    // faster SMs take more work.  Unsorted (more sequences than are sorted here
    // and no order given): the snake deal, which needs no set-up.
    if constexpr (kSort != 0) {
        int une = 0;   // nonempty sequences x H
        if constexpr (kSort == 2) {
            // the sorted order and the row table were prepared in device memory
            if (tid == 0) une = *p.g_une;
        } else {
            int *lens = sm.ptr<int>(kOffP);
            int2 *rows = reinterpret_cast<int2 *>(order + kMaxSortedSeqs);
            for (int n = tid; n < p.N; n += kThreads) {
                const int cb = p.cu[n], ce = p.cu[n + 1];
                int b = min(max(cb, 0), p.T), e = min(max(ce, 0), p.T);
                if (cb < 0 || cb > p.T || ce < 0 || ce > p.T) atomicOr(p.err, kErrBadSeqlens);
                if (e < b || (kSlots && state_index<kSlots>(p, n) < 0)) e = b;
                rows[n] = make_int2(b, e);
                lens[n] = e - b;
            }
            __syncthreads();
            for (int n = tid; n < p.N; n += kThreads) {
                int rank = 0;
                const int ln = lens[n];
                for (int m2 = 0; m2 < p.N; m2++) {
                    const int lm = lens[m2];
                    rank += (lm > ln) || (lm == ln && m2 < n);
                }
                order[rank] = n;
            }
            __syncthreads();
            if (tid == 0) {
                for (int n = 0; n < p.N; n++) une += lens[n] > 0;
                une *= p.H;
            }
        }
        if (tid == 0) {
            const bool first = (int)blockIdx.x < une;
            *sm.units_nonempty() = une;
            sm.sched()[0] = first ? (int)blockIdx.x : -1;
            *sm.published() = first ? 1 : 0;
            *sm.claim_done() = first ? 0 : 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

#ifdef KDA_TRACE
    if (tid == 0 && blockIdx.x < 1024) g_kda_cta[blockIdx.x][0] = kda_gtimer();
#endif
    const Maps maps = {&tq, &tk, &tv, &tg, &to};
    if (warp < 4) {
        chain_role<kSlots, kSort>(p, sm, order, U, maps);
    } else if (warp < 12) {
        e_role<kSlots, kSort, kConv>(p, cp, sm, order, U, maps);
    } else {
        i_role<kSlots, kSort, kConv>(p, &cp, sm, order, U);
    }
    // every MMA this CTA issued has completed before TMEM is released
    if (tid == 0 || tid == kChainThreads || tid == kChainThreads + kEThreads) {
        mma_commit(sm.bar(kBarDrain));
        mbar_wait_drain(sm.bar(kBarDrain), 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(*sm.tmem_base(), kTmCols);
    // the last CTA to finish returns the dynamic deal's scratch slot to zero
    if (tid == 0 && p.sched) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
#ifdef KDA_TRACE
    if (tid == 0 && blockIdx.x < 1024) {
        g_kda_cta[blockIdx.x][1] = kda_gtimer();
    }
#endif
}

// ---- host side ------------------------------------------------------------------
// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised exactly once even when host threads race on the first call).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return nullptr;
    }();
    return fn;
}

// [T][H][128] viewed as 4-D {c (box_inner wide), row, channel block, head}:
// one box {box_inner, box_rows, box_blocks (default all 128/box_inner), 1} is
// [block][row][c] in shared memory -- the 128B-swizzled tiles, blocks apart.
bool make_map4(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem, int T, int H, int box_inner,
               int box_rows = kChunk, int box_blocks = 0)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const int nblk = kD / box_inner;
    cuuint64_t dims[4] = {(cuuint64_t)box_inner, (cuuint64_t)T, (cuuint64_t)nblk, (cuuint64_t)H};
    cuuint64_t strides[3] = {(cuuint64_t)H * kD * elem, (cuuint64_t)box_inner * elem, (cuuint64_t)kD * elem};
    cuuint32_t box[4] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, (cuuint32_t)(box_blocks ? box_blocks : nblk), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, dt, 4, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// one box {box_inner channels, 1 head, 64 rows}: 128B-swizzled for the MMA
// operands (k, q: box_inner 64), unswizzled for g (box_inner 128)
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem, int T, int H, int box_inner,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * elem, (cuuint64_t)H * kD * elem};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, (cuuint32_t)kChunk};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_max_sorted_seqs() { return kMaxSortedSeqs; }

// one chain CTA per unit, at least as many producer CTAs; units fit the
// producers' packed claims (8 bits) and the sequences the sorted table
bool tc_split_possible(int units, int N, int num_sms)
{
    return units >= 1 && 2 * units <= num_sms && units <= 255 && N <= kMaxSortedSeqs;
}
// half chains: two chain CTAs per unit, at least as many producers again
bool tc_split_half_possible(int units, int N, int num_sms)
{
    return tc_split_possible(units, N, num_sms) && 4 * units <= num_sms;
}
size_t tc_split_flag_bytes(int units) { return ((size_t)units * kRingSlots * kFlagSlotStride + 32) * sizeof(int); }
size_t tc_split_bytes(int units) { return (size_t)units * kRingSlots * kSlotBytes + tc_split_flag_bytes(units); }

cudaError_t launch_kda_tc_split(const KdaArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, const CUtensorMap &tg, const CUtensorMap &to)
{
    using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const CUtensorMap, TcParams, const SplitParams);
    static const Kernel kernels[4] = {kda_tc_split_kernel<false, false>, kda_tc_split_kernel<true, false>,
                                      kda_tc_split_kernel<false, true>, kda_tc_split_kernel<true, true>};
    const int variant = (a.state_slots != nullptr) + 2 * a.split_half;
    const Kernel kernel = kernels[variant];
    static std::atomic<int> attr_set[4][64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[variant][dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[variant][dev].store(1, std::memory_order_release);
    }
    const int units = a.N * a.H;
    TcParams p;
    p.cu = a.cu_seqlens;
    p.beta = a.beta;
    p.s0 = a.initial_state;
    p.out = (__nv_bfloat16 *)a.out;
    p.s1 = a.final_state;
    p.N = a.N;
    p.T = a.T;
    p.H = a.H;
    p.g_order = nullptr;
    p.g_rows = nullptr;
    p.g_une = nullptr;
    p.err = a.err_word;
    p.sched = a.sched;
    p.slots = a.state_slots;
    p.num_slots = a.num_slots;
    SplitParams sp;
    sp.ring = a.split_ring;
    int *flags = reinterpret_cast<int *>(a.split_ring + (size_t)units * kRingSlots * kSlotBytes);
    sp.ready = flags;
    sp.freed = flags + kFlagSlotStride / 2;
    sp.abort = flags + (size_t)units * kRingSlots * kFlagSlotStride;
    sp.chains = a.split_half ? 2 * units : units;
    // every CTA resident at once (one per SM): chains and producers wait on one another
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.num_sms);
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tg, to, p, sp);
}

cudaError_t launch_kda_tc_bf16_d128(const KdaArgs &a)
{
    CUtensorMap tq, tk, tv, tg, to;
    memset(&tq, 0, sizeof tq); memset(&tk, 0, sizeof tk); memset(&tv, 0, sizeof tv); memset(&tg, 0, sizeof tg);
    memset(&to, 0, sizeof to);
    if (a.T > 0) {
        if (!make_map(&tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) ||
            !make_map(&tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) ||
            !make_map4(&tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64) ||
            !make_map(&tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map4(&to, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64, 32))
            return cudaErrorInvalidValue;
    }
    if (a.split_ring) {
        if (a.conv_w || a.g_order || !a.sched || a.T == 0 || !tc_split_possible(a.N * a.H, a.N, a.num_sms) ||
            (a.split_half && !tc_split_half_possible(a.N * a.H, a.N, a.num_sms)))
            return cudaErrorInvalidValue;
        // a half chain stores the 32-row output tiles of its 64 channels
        if (a.split_half && !make_map4(&to, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, 64, 32, 1))
            return cudaErrorInvalidValue;
        return launch_kda_tc_split(a, tq, tk, tv, tg, to);
    }
    // one kernel per (slot table, sort mode): 1 sorted here (N <= kMaxSortedSeqs),
    // 2 sorted order given in g_order/g_rows, 0 unsorted; modes 1 and 2 deal
    // dynamically and need the deal's scratch words
    const int sort = a.g_order ? 2 : (a.N <= kMaxSortedSeqs ? 1 : 0);
    if (sort != 0 && !a.sched) return cudaErrorInvalidValue;
    const bool conv = a.conv_w != nullptr;
    if (conv && sort == 2) return cudaErrorInvalidValue;   // no conv build with a prepared order
    const int variant = 6 * conv + 3 * (a.state_slots != nullptr) + sort;
    using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const CUtensorMap, TcParams, const ConvParams);
    static const Kernel kernels[12] = {
        kda_tc_kernel<false, 0, false>, kda_tc_kernel<false, 1, false>, kda_tc_kernel<false, 2, false>,
        kda_tc_kernel<true, 0, false>,  kda_tc_kernel<true, 1, false>,  kda_tc_kernel<true, 2, false>,
        kda_tc_kernel<false, 0, true>,  kda_tc_kernel<false, 1, true>,  nullptr,
        kda_tc_kernel<true, 0, true>,   kda_tc_kernel<true, 1, true>,   nullptr};
    const Kernel kernel = kernels[variant];
    // the shared-memory opt-in, once per (kernel, device); setting it twice
    // (two host threads racing on a first call) is harmless
    static std::atomic<int> attr_set[12][64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[variant][dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[variant][dev].store(1, std::memory_order_release);
    }
    TcParams p;
    p.cu = a.cu_seqlens;
    p.beta = a.beta;
    p.s0 = a.initial_state;
    p.out = (__nv_bfloat16 *)a.out;
    p.s1 = a.final_state;
    p.N = a.N;
    p.T = a.T;
    p.H = a.H;
    p.g_order = a.g_order;
    p.g_rows = a.g_rows;
    p.g_une = a.g_units_nonempty;
    p.err = a.err_word;
    p.sched = a.sched;
    p.slots = a.state_slots;
    p.num_slots = a.num_slots;
    ConvParams cp;
    cp.x[0] = (const uint16_t *)a.q;
    cp.x[1] = (const uint16_t *)a.k;
    cp.x[2] = (const uint16_t *)a.v;
    cp.w = a.conv_w;
    cp.pool = a.conv_pool;
    cp.H = a.H;
    cp.act = a.conv_act;
    cp.eps = a.conv_eps;
    const int units = a.N * a.H;
    const int grid = units < a.num_sms ? units : a.num_sms;
    // one CTA per SM (shared memory), so a CTA launched early waits for an SM
    // that the previous kernel has left; its set-up overlaps that kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tg, to, p, cp);
}

}  // namespace kda
