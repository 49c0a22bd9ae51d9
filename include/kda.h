/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA chunked packed-varlen prefill.
 *
 * Kimi Delta Attention (KDA) is the gated delta rule with a per-channel decay
 * that the Kimi-K3 prefill runs in its KDA layers (kern-k3-pp-prefill README,
 * "P: the packed prefill"; the NVIDIA KDA_prefill kernels ported in SGLang
 * PR #32890, prhub report section "实现拆解", item 3).  For every packed
 * sequence n and head h, with S in R^{dk x dv}:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * computed per 64-row chunk in WY form: in-chunk cumulative log-decay G, the
 * strictly lower A_kk = beta_i (k_i * exp(G_i - G_j)) . k_j, the inverse of
 * (I + A_kk), the factors W and U, the inter-chunk state recurrence, the
 * outputs, and the fp32 final state of every sequence.  No 1/sqrt(dk) scale
 * is applied to q; token t's output includes token t's own write.
 *
 * Conventions shared by all entry points
 * --------------------------------------
 *  Pointers   all tensor pointers are DEVICE pointers; every tensor is dense
 *             and row-major (innermost index last).  The caller owns every
 *             buffer.  The library keeps no pointer after return and is
 *             reentrant across streams.  It allocates nothing per call,
 *             except in split mode (below), which takes a few MB of device
 *             memory on the call's stream from a pool of the library's own
 *             (kept for later calls) and returns them when the call ends.
 *  Async      calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *             legacy default stream).  The host never reads cu_seqlens and
 *             never synchronises.
 *  Layouts    q, k: [T][H][dk];  v, out: [T][H][dv];  g: [T][H][dk];
 *             beta: [T][H];  cu_seqlens: int32 [N+1];
 *             initial_state, final_state: [N][H][dv][dk] fp32, i.e. S^T with
 *             dk contiguous -- SGLang's recurrent-state pool layout
 *             [slot][head][v][k] f32 (kern-k3-pp-prefill README, section
 *             "D inside SGLang").
 *  Packing    sequence n occupies rows [cu_seqlens[n], cu_seqlens[n+1]);
 *             up to 16 sequences in 8192 rows is the production shape
 *             (kern-k3-pp-prefill README, "P: the packed prefill").  Chunks
 *             start at each sequence's first row and never cross a sequence;
 *             the last chunk of a sequence may be partial.  A zero-length
 *             sequence copies initial_state to final_state (zeros if NULL).
 *  cu_seqlens contract: cu[0] = 0, nondecreasing, cu[N] = T.  It is not read
 *             on the host; the kernels clamp every row index into [0, T], so
 *             a bad table never makes them access memory out of bounds.
 *  Inputs     q and k are expected L2-normalised per head by the caller.
 *  Kernels    bf16 with dk = dv = 128 runs on the tensor-core kernel; every
 *             other head size, every fp32 call and kda_chunk_prefill_fullrange
 *             run on the CUDA-core kernel (fp32 arithmetic throughout).
 *  Split      the tensor-core kernel is one CTA per SM taking whole
 *             (sequence, head) units, each unit's chunks one after another.
 *             For calls with few units (N * H at most half the SMs, T >= 1024,
 *             N <= 256) it runs in split mode instead: one SM per unit keeps
 *             that unit's state chain, and every other SM prepares chunks of
 *             any unit (the part of a chunk's work that does not depend on the
 *             state), handing them over through a ring in device memory.
 *             Where N * H is at most a fifth of the SMs, two SMs keep each
 *             unit's chain, 64 of the 128 value channels each (the value
 *             channels of the state evolve independently).  The results are
 *             the same bytes in every form.  The environment variable
 *             KDA_SPLIT, read on every call, overrides the choice: "0" never
 *             splits, "1" splits every call that allows it (T >= 1 in place
 *             of 1024), "full" and "half" do so in that form ("half" falls
 *             back to one chain SM a unit where the SMs do not allow two).
 *             A call that cannot get its ring or its cooperative launch runs
 *             unsplit.
 *  Range      the tensor-core kernel rounds its MMA operands to fp16 (fp32
 *             accumulation) and splits each in-chunk decay exp(G_i - G_j)
 *             into exp(G_i - G_m) exp(G_m - G_j) around the chunk's middle
 *             row m.  It therefore needs, per key channel and 64-row chunk,
 *             |G_r - G_m| <= 15 ln 2 (about 10.4) for every row r -- with
 *             g ~ U[-0.2, 0] the largest is about 4, with g ~ U[-0.5, 0]
 *             about 10 -- and |v|, |S| below about 6.5e4.  A chunk whose decay
 *             is outside that range sets bit 32 of the device error word
 *             (kda_device_error); the results of that call are then not to be
 *             used: run it again through kda_chunk_prefill_fullrange, which
 *             forms every decay factor directly and has no such limit.
 *  Aliasing   final_state == initial_state (the same pointer) is allowed and
 *             updates the states in place; any other overlap between an output
 *             and any other argument returns KDA_ERR_ALIAS.
 *  Errors     arguments are validated synchronously before anything is
 *             launched; a failed check returns its status and launches
 *             nothing.  A launch failure returns KDA_ERR_CUDA (the CUDA error
 *             stays readable through cudaGetLastError()).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,         /* a required pointer is NULL                    */
    KDA_ERR_SHAPE = 2,        /* N < 1, T < 0, H < 1, or a size overflows      */
    KDA_ERR_UNSUPPORTED = 3,  /* dk/dv/dtype combination or N not supported    */
    KDA_ERR_ALIGN = 4,        /* a tensor pointer is not 16-byte aligned       */
    KDA_ERR_ALIAS = 5,        /* an output overlaps another argument           */
    KDA_ERR_CUDA = 6,         /* a CUDA call failed (see cudaGetLastError)     */
    KDA_ERR_DEVICE = 7,       /* no CUDA device, or not an sm_103 device       */
    KDA_ERR_NOALLOC_LIMIT = 8 /* N above KDA_NOALLOC_MAX_SEQS (noalloc entry)  */
} kda_status;

/*
 * kda_chunk_prefill -- bf16 q/k/v in, bf16 out (round to nearest even from
 * the fp32 accumulator), fp32 g, beta and states.
 *
 *   q, k, v        bf16 bit patterns (uint16), layouts above.
 *   g              fp32 per-token log-decay log(alpha), [T][H][dk].
 *   beta           fp32 write strength, [T][H].
 *   cu_seqlens     int32 [N+1], device memory.
 *   initial_state  fp32 [N][H][dv][dk], or NULL for a zero start.
 *   out            bf16 [T][H][dv]; every row in [0, T) is written.
 *   final_state    fp32 [N][H][dv][dk], or NULL (not written).
 *   N, T, H        sequences (N >= 1), rows (T >= 0), heads (H >= 1);
 *                  N * H must fit in 31 bits.
 *   dk, dv         key and value head dims, each 64 or 128 (else
 *                  KDA_ERR_UNSUPPORTED).  dk = dv = 128 runs on the
 *                  tensor-core kernel (decay range: see "Range" above), the
 *                  other sizes on the CUDA-core kernel.
 *   stream         cudaStream_t to launch on.
 * Returns a kda_status.
 */
int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *g, const float *beta, const int32_t *cu_seqlens,
                      const float *initial_state, uint16_t *out, float *final_state,
                      int N, int T, int H, int dk, int dv, void *stream);

/*
 * kda_chunk_prefill_f32 -- the same operation with fp32 q/k/v and fp32 out,
 * on the CUDA-core kernel (fp32 arithmetic, no limit on the decay).  dk and
 * dv each 64 or 128.  All other conventions as kda_chunk_prefill.
 */
int kda_chunk_prefill_f32(const float *q, const float *k, const float *v,
                          const float *g, const float *beta, const int32_t *cu_seqlens,
                          const float *initial_state, float *out, float *final_state,
                          int N, int T, int H, int dk, int dv, void *stream);

/*
 * kda_chunk_prefill_fullrange -- kda_chunk_prefill (bf16 q/k/v/out, same
 * arguments, layouts, sizes and errors) always on the CUDA-core kernel.  It
 * computes every in-chunk decay factor exp(G_i - G_j) directly in fp32, so it
 * holds for any finite decay the recurrence itself keeps finite: strong gates
 * (alpha near 0, g of -20 and below), mixed signs and mild growth (g > 0).  It
 * never sets bit 32.  One CTA per (sequence, head), fp32 on CUDA cores: slower
 * than the tensor-core kernel, meant for inputs outside that kernel's range.
 */
int kda_chunk_prefill_fullrange(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const float *g, const float *beta, const int32_t *cu_seqlens,
                                const float *initial_state, uint16_t *out, float *final_state,
                                int N, int T, int H, int dk, int dv, void *stream);

/*
 * kda_chunk_prefill_noalloc -- kda_chunk_prefill for packed batches of up to
 * KDA_NOALLOC_MAX_SEQS sequences, for callers that cannot allocate device
 * memory per call: code inside a serving runtime whose device memory is laid
 * out in full when a model is loaded (all buffers come from a fixed pool), or
 * a layer library that is handed only its tensors.  The pages have no
 * counterpart of this entry point; it exists for those callers.
 *
 * With many sequences the work is dealt to the SMs by length from a shared
 * counter, which needs a sequence table in device memory.  That table lives in
 * a static array inside the library (about 196 KB, held by every GPU that
 * loads the library until the process exits), so the call itself allocates
 * nothing -- no cudaMalloc, cudaFree or library allocator.
 *
 * Arguments, layouts, results and errors are those of kda_chunk_prefill,
 * except 1 <= N <= KDA_NOALLOC_MAX_SEQS: the arguments are checked as there
 * first, and then a larger N returns KDA_ERR_NOALLOC_LIMIT; a failed check
 * launches nothing.  Results equal kda_chunk_prefill's bit for bit (the
 * per-sequence arithmetic does not depend on the schedule).  Head sizes other
 * than dk = dv = 128 run on the CUDA-core kernel, which needs no table.
 *
 * The first call on a device looks up the array's device address (and checks
 * the device) with that device current; make that first call before any
 * stream capture.  Every call shares the one array: the call clears the parts
 * that must start at zero, but calls whose kernels overlap on the GPU (on
 * different streams without ordering between them) race on it -- order them.
 */
#define KDA_NOALLOC_MAX_SEQS 16384
int kda_chunk_prefill_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const float *g, const float *beta, const int32_t *cu_seqlens,
                              const float *initial_state, uint16_t *out, float *final_state,
                              int N, int T, int H, int dk, int dv, void *stream);

/*
 * kda_chunk_prefill_slots -- kda_chunk_prefill with the recurrent states kept
 * in a pool that a serving engine owns and addresses by slot id (kern-k3-pp-
 * prefill README, section "D inside SGLang": a KDA layer's state lives in the
 * engine's pool laid out [slot][head][v][k] f32 and is reached through a
 * table of slot ids, where a padded entry carries slot -1 and is skipped).
 *
 *   state_slots  int32 [N], device memory: the pool entry of sequence n.
 *                -1 marks a padded sequence: nothing of it is computed, its
 *                rows of `out` are not written and the pool is not touched.
 *   state_pool   fp32 [num_slots][H][dv][dk], device memory.  Sequence n
 *                starts from state_pool[state_slots[n]] and its final state
 *                replaces that entry (in place).  Entries that no sequence
 *                names are not touched.  A sequence of zero rows leaves its
 *                entry as it was.
 *   num_slots    entries in the pool (>= 1).
 * All other arguments, layouts and limits are those of kda_chunk_prefill
 * (which takes dense [N][H][dv][dk] states instead).
 *
 * The ids are not read on the host.  Valid ids must be distinct: two
 * sequences that name one entry race on it.  An id outside [-1, num_slots)
 * is treated like -1 and sets bit 8 of the device error word
 * (kda_device_error).  Results for a sequence equal, bit for bit, those of
 * kda_chunk_prefill given the same rows and that sequence's entry as its
 * initial state.  Returns a kda_status; KDA_ERR_NULL if state_slots or
 * state_pool is NULL, KDA_ERR_SHAPE if num_slots < 1, KDA_ERR_ALIAS if the
 * pool overlaps any other argument.
 */
int kda_chunk_prefill_slots(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *g, const float *beta, const int32_t *cu_seqlens,
                            const int32_t *state_slots, float *state_pool, int num_slots,
                            uint16_t *out, int N, int T, int H, int dk, int dv, void *stream);

/*
 * kda_chunk_prefill_conv -- the short-conv + L2-norm prologue of
 * kda_short_conv fused into the tensor-core prefill, as a KDA layer runs it
 * (kern-k3-pp-prefill README: section "P: the packed prefill" runs the KDA
 * layers with per-sequence conv windows and states; section "D inside SGLang"
 * keeps both in the engine's pools, indexed by the same slot ids).  For every
 * sequence n, with e its pool entry (slots[n], or n when slots is NULL):
 *
 *     q, k, v = the conv of kda_short_conv over [window e ; the sequence's
 *               rows of xq, xk, xv] (optional SiLU; q and k scaled to unit L2
 *               norm per head with eps), rounded to bf16 as kda_short_conv's
 *               outputs are;
 *     then kda_chunk_prefill_slots on those q, k, v with the state pool entry e;
 *     the window e becomes the last three rows of [old taps ; the rows].
 *
 * q, k and v are formed in shared memory inside the kernel and never written
 * to global memory; the prologue's arithmetic is kda_short_conv's, in the same
 * order, so results and windows equal kda_short_conv followed by
 * kda_chunk_prefill_slots bit for bit.  Speed: the call saves the round trip
 * of q, k and v through global memory (402 MB for 8192 rows at H = 32), but
 * the prologue's arithmetic lengthens the prefill kernel's busiest role, and
 * on a GB300 the two calls are faster (about 239 us against 256 us at that
 * shape); use this call where memory traffic or capacity is the constraint.
 *
 *   xq, xk, xv   bf16 bits [T][H][128]: the layer's projections.
 *   conv_weight  fp32 [3][H*128][4], as for kda_short_conv.
 *   g, beta      fp32 [T][H][128], [T][H].
 *   cu_seqlens   int32 [N+1], device memory.
 *   slots        int32 [N], device memory, or NULL (entry n in both pools).
 *                -1 marks a padded sequence: nothing of it is computed or
 *                written (out rows, state, window).  An id that is not an
 *                entry of both pools is treated like -1 and sets bit 8.
 *   conv_pool    bf16 bits [conv_num_slots][3 taps][3 streams][H*128], the
 *                windows, updated in place (the layout kda_short_conv uses).
 *   state_pool   fp32 [num_slots][H][128][128], updated in place.
 *   out          bf16 bits [T][H][128].
 *   N, T, H      as for kda_chunk_prefill; with slots NULL, num_slots and
 *                conv_num_slots must be at least N.
 *   dk, dv       128 (else KDA_ERR_UNSUPPORTED).
 *   activation   0 (none) or 1 (SiLU); eps >= 0, as for kda_short_conv.
 * The decay range is that of the tensor-core kernel (bit 32, "Range" above).
 * Tensor pointers must be 16-byte aligned (beta, cu_seqlens and slots
 * 4-byte); out and the pools must not overlap an input or each other.
 * Returns a kda_status.
 */
int kda_chunk_prefill_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv,
                           const float *conv_weight, const float *g, const float *beta,
                           const int32_t *cu_seqlens, const int32_t *slots, uint16_t *conv_pool,
                           int conv_num_slots, float *state_pool, int num_slots, uint16_t *out,
                           int N, int T, int H, int dk, int dv, int activation, float eps,
                           void *stream);

/*
 * kda_decode -- one step of the recurrence for each of N sequences (one new
 * token each), the decode that runs between prefills (kern-k3-pp-prefill
 * README: the KDA step over a rank's heads on the engine's state pool, padded
 * rows skipped, section "D inside SGLang").  For sequence n and head h, with S
 * the entry state_pool[state_slots[n]][h]:
 *
 *     S <- (I - beta k k^T) Diag(exp(g)) S + beta k v^T,   out = S^T q
 *
 * which is kda_chunk_prefill_slots on cu_seqlens = {0, 1, ..., N}.
 *
 *   q, k, v      bf16 bits [N][H][dk|dv], row n = sequence n's token.
 *   g, beta      fp32 [N][H][dk], [N][H].
 *   state_slots  int32 [N], device memory, or NULL for entry n.  -1 marks a
 *                padded row: nothing of it is computed or written.  An id
 *                outside [-1, num_slots) is treated like -1 and sets bit 8 of
 *                the device error word.  Valid ids must be distinct.
 *   state_pool   fp32 [num_slots][H][dv][dk], updated in place; entries no
 *                row names are not touched.  With state_slots NULL,
 *                num_slots >= N.
 *   out          bf16 bits [N][H][dv].
 *   N, H         rows (sequences) >= 1, heads >= 1; dk = dv = 128.
 * Tensor pointers must be 16-byte aligned (beta and state_slots 4-byte); the
 * pool must not overlap any other argument and out must not overlap an
 * input.  Returns a kda_status.
 */
int kda_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
               const float *beta, const int32_t *state_slots, float *state_pool, int num_slots,
               uint16_t *out, int N, int H, int dk, int dv, void *stream);

/*
 * kda_decode_conv -- kda_decode with the short conv + L2-norm prologue of
 * kda_short_conv fused in front of it (kern-k3-pp-prefill README, section
 * "D inside SGLang": the packed decode step runs the conv on the step's rows
 * with the windows in the engine's pool, then the recurrence).  For each row n
 * (one token of sequence n) and head h, with the window of conv_slots[n]:
 *
 *     q, k, v  = the conv of kda_short_conv over [window taps 0..2 ; x_n]
 *                (optional SiLU; q and k scaled to unit L2 norm over the
 *                head's channels with eps as there), kept in fp32;
 *     then the kda_decode step on state_pool[state_slots[n]][h] with those
 *     q, k, v and g, beta, writing out[n][h];
 *     the window becomes [taps 1, 2 ; x_n].
 *
 * One kernel: one CTA per (sequence, head) computes that head's conv once,
 * steps all its value rows and rewrites its channels of the window; it is
 * faster than kda_short_conv followed by kda_decode (on a GB300, 64 sequences
 * x 32 heads: about 48 us against 58 us).  Results differ from those two
 * calls only in that q, k and v are not rounded to bf16 between them.
 *
 *   xq, xk, xv   bf16 bits [N][H][dk|dv]: the step's projections.
 *   conv_weight  fp32 [3][H*128][4], as for kda_short_conv.
 *   conv_slots   int32 [N] or NULL (entry n): the window entry of row n.
 *   conv_pool    bf16 bits [conv_num_slots][3 taps][3 streams][H*128], the
 *                layout kda_short_conv reads and writes; updated in place.
 *   g, beta, state_slots, state_pool, num_slots, out: as for kda_decode.
 *   activation, eps: as for kda_short_conv.
 *   N, H         rows (sequences) >= 1, heads >= 1; dk = dv = 128.
 * A row whose state id or window id is -1 is padding: nothing of it is
 * computed or written (neither its state, its window nor its out row).  An id
 * outside [-1, num_slots) (or [-1, conv_num_slots)) is treated like -1 and
 * sets bit 8 of the device error word.  Valid ids must be distinct within
 * each table.  Tensor pointers must be 16-byte aligned (beta and the slot
 * tables 4-byte); the pools and out must not overlap an input or each other.
 * Returns a kda_status.
 */
int kda_decode_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv,
                    const float *conv_weight, const int32_t *conv_slots, uint16_t *conv_pool,
                    int conv_num_slots, const float *g, const float *beta,
                    const int32_t *state_slots, float *state_pool, int num_slots, uint16_t *out,
                    int N, int H, int dk, int dv, int activation, float eps, void *stream);

/*
 * kda_fold_commit -- the state commit of a speculative decoding round (the
 * ReplaySSM exact fold: SGLang PR #32890, prhub report section "实现拆解",
 * item 3 and the speculative-decoding file list).  A verify pass scores W
 * draft tokens per sequence without committing states; once accepted[n] of
 * them are kept, this call folds exactly those tokens into the state:
 *
 *     for t in 0 .. accepted[n]-1:
 *         S <- (I - beta_t k_t k_t^T) Diag(exp(g_t)) S + beta_t k_t v_t^T
 *
 * with S the entry state_pool[state_slots[n]][h] for every head h.  The
 * result equals accepted[n] calls of kda_decode bit for bit (the same per-step
 * arithmetic), while reading and writing each state once.  No outputs are
 * produced (the verify pass already scored the tokens).
 *
 *   k, v         bf16 bits [N][W][H][dk|dv]: sequence n's window of W tokens.
 *   g, beta      fp32 [N][W][H][dk], [N][W][H].
 *   accepted     int32 [N], device memory, each in [0, W]; 0 leaves the state
 *                untouched.  A count outside [0, W] is clamped into it and
 *                sets bit 16 of the device error word.
 *   state_slots  int32 [N] or NULL (entry n); -1 skips the sequence; an id
 *                outside [-1, num_slots) is skipped and sets bit 8.
 *   state_pool   fp32 [num_slots][H][dv][dk], updated in place.
 *   N, W, H      sequences >= 1, window length >= 1, heads >= 1; dk = dv = 128.
 * Alignment and aliasing rules as kda_decode.  Returns a kda_status.
 */
int kda_fold_commit(const uint16_t *k, const uint16_t *v, const float *g, const float *beta,
                    const int32_t *accepted, const int32_t *state_slots, float *state_pool,
                    int num_slots, int N, int W, int H, int dk, int dv, void *stream);

/*
 * kda_short_conv -- the short-conv + L2-norm prologue that turns a KDA layer's
 * q, k, v projections into the kernel's q, k, v, with each sequence's conv
 * window carried across calls (kern-k3-pp-prefill README: section "P: the
 * packed prefill" runs the KDA layers with per-sequence conv windows and
 * states; section "D inside SGLang" keeps the window in the engine's pool laid
 * out [slot][tap][q | k | v] bf16, indexed by the same slot ids as the state).
 * For sequence n (rows t = 0 .. L-1 from cu_seqlens[n]), stream s in {q, k, v}
 * and channel c (flat over the H heads of d channels):
 *
 *     x_{-3}, x_{-2}, x_{-1}   the window's taps 0, 1, 2 (oldest first)
 *     y_t[c] = sum_{j=0..3} conv_weight[s][c][j] * x_{t-3+j}[c]
 *     y_t    = y_t, or SiLU(y_t) = y_t / (1 + exp(-y_t)) with activation 1
 *     q_t = y_t / sqrt(|y_t|^2 + eps) over each head's d channels; k_t likewise;
 *     v_t = y_t
 *
 * after which the window holds the last three rows of [old taps ; the L rows].
 * The pages fix the window layout; the kernel size (four taps: the three
 * carried rows and the row itself) is read off the window, and the weights,
 * the activation and eps are the caller's.
 *
 *   xq, xk, xv   bf16 bits [T][H][d], the projections of the packed rows.
 *   conv_weight  fp32 [3][H*d][4]: stream (q, k, v), channel, tap; tap 3
 *                weighs the row itself.
 *   cu_seqlens   int32 [N+1], as for kda_chunk_prefill.
 *   conv_slots   int32 [N], device memory, or NULL for entry n: the pool entry
 *                of sequence n.  -1 marks a padded sequence: its rows of the
 *                outputs are not written and its entry is not touched.  An id
 *                outside [-1, num_slots) is treated like -1 and sets bit 8 of
 *                the device error word.  Valid ids must be distinct.
 *   conv_pool    bf16 bits [num_slots][3 taps][3 streams][H*d], updated in
 *                place; a sequence of zero rows leaves its entry as it was.
 *   q_out, k_out, v_out  bf16 bits [T][H][d] (rows of no sequence and of
 *                padded sequences are not written).
 *   activation   0 (none) or 1 (SiLU); eps >= 0 (an all-zero row with eps 0
 *                gives NaN, as the formula does).
 *   N >= 1, T >= 0, H >= 1; d = 128.
 * Tensor pointers must be 16-byte aligned (cu_seqlens and conv_slots 4-byte).
 * The outputs must not overlap an input, the pool or each other; the pool must
 * not overlap an input.  One kernel runs on `stream`; the warp that holds a
 * sequence's first row alone reads its window and then rewrites it.  Returns
 * a kda_status.
 */
int kda_short_conv(const uint16_t *xq, const uint16_t *xk, const uint16_t *xv,
                   const float *conv_weight, const int32_t *cu_seqlens,
                   const int32_t *conv_slots, uint16_t *conv_pool, int num_slots,
                   uint16_t *q_out, uint16_t *k_out, uint16_t *v_out, int N, int T, int H, int d,
                   int activation, float eps, void *stream);

/* Human-readable name of a kda_status value (static string, never NULL). */
const char *kda_status_string(int status);

/*
 * kda_device_error -- read the library's sticky device error word on the
 * current device.  Every wait inside the kernels is bounded; a wait that runs
 * out sets bit 1 here and the kernel returns early (outputs are then
 * undefined).  Bit 2: a cu_seqlens entry broke its contract (indices were
 * clamped).  Bit 8: a state slot id was outside [-1, num_slots) (that
 * sequence was skipped).  Bit 16: an accepted count of kda_fold_commit was
 * outside [0, W] (clamped).  Bit 32: the tensor-core prefill met a chunk whose
 * decay is outside its fp16 operand range (see "Range" above; use
 * kda_chunk_prefill_fullrange for such inputs).  0 means no kernel of this
 * library has reported an error.
 * Synchronises the current device.  If `reset` is nonzero the word is
 * cleared after reading.  Returns KDA_OK or KDA_ERR_CUDA.
 */
int kda_device_error(int *word, int reset);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
