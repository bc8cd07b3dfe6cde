/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification step.
 *
 * The operation (one verification round, after the target model's single
 * forward over the drafted tokens) is the modified rejection sampler that all
 * of these pages state:
 *   [P1] "Speculative Decoding" (atonlee.tistory.com/330), ch.2 (one round:
 *        accept in order, cut at the first rejection, k accepted + 1 token)
 *        and ch.3 (accept test r < min(1, p(x)/q(x)), residual
 *        norm(max(0, p - q)), greedy rule at temperature 0);
 *   [P2] "Speculative Decoding으로 LLM 추론 속도 높이기" (donmain.dev), section
 *        "품질은 rejection sampling이 지킨다";
 *   [P3] "Fast Inference from Transformers via Speculative Decoding" notes
 *        (obsidian-dorae222.pages.dev), method details, steps 2-3 (gamma+1
 *        target distributions from one forward, accept probability, residual
 *        sample, bonus token from p at row gamma when every draft passes);
 *   [P4] "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가" (ailab.paldyn.com),
 *        section on why the output does not change (greedy: draft == argmax).
 *
 * For each sequence b with g = num_draft[b] drafts and temperature T = temperature[b]:
 *   T > 0:  p_i = softmax(target_logits[b, i, :] / T) for i <= g,
 *           q_i = softmax(draft_logits[b, i, :] / T) for i < g.
 *           Position i < g accepts draft x_i = draft_tokens[b, i] iff
 *           uniforms[b, i] * q_i(x_i) < p_i(x_i); n = first rejected i, or g.
 *           One more token y is drawn by inverse CDF with u = uniforms[b, gamma_max]
 *           from max(0, p_n - q_n) (n < g) or from p_g (n == g): y is the
 *           smallest id j with u * S < C_j, C_j the running sum of the weights
 *           in id order and S their total.  The weights are integers on a
 *           2^-60 grid, each within about 2^-36 of its exact value where it
 *           matters (ids whose weight is within a factor 2^15 of the row's
 *           largest; float32, to about 2^-22, for the rest), so every sum is
 *           exact and y differs from the float64 definition only when u lies
 *           within ~1e-9 of a boundary C_j / S (rows whose
 *           |logit| * log2(e) / T passes 2^21 keep float32 weights throughout).
 *   T == 0: greedy; a_i = argmax of the raw target logits of row i (lowest id
 *           on ties); position i accepts iff x_i == a_i; y = a_n.  No draft row
 *           and no uniform is read.
 *   Output: out_tokens[b, 0..n-1] = x_0..x_{n-1}, out_tokens[b, n] = y,
 *           out_tokens[b, n+1..gamma_max] = -1, out_num_accepted[b] = n.
 * Point-mass proposals (draft_logits == NULL; a deterministic proposer such as
 * prompt lookup, "Speculative Decoding" ch.5): q_i is 1 at x_i, so position i
 * accepts iff uniforms[b, i] < p_i(x_i) and a rejection samples p_n with x_n
 * removed (max(0, p - q) for that q).  No draft row is read.
 * The full sweep (options.kernel 2) also reads the rows after the cut; the
 * early exit (kernel 3, the automatic choice for large batches and tiny rows)
 * reads none.  Rows i > g (target) and i >= g (draft), and every draft row of
 * a greedy sequence, are never read.
 *
 * Layout.  All arrays are dense, row-major, and readable by the device of the
 * calling thread's current CUDA context:
 *   target_logits  [B, gamma_max + 1, V]   dtype (SPEC_F32 or SPEC_BF16)
 *   draft_logits   [B, gamma_max, V]       dtype, or NULL for point-mass proposals
 *   draft_tokens   [B, gamma_max]          int32
 *   num_draft      [B]                     int32
 *   uniforms       [B, gamma_max + 1]      float32 in [0, 1)
 *   temperature    [B]                     float32
 *   out_tokens     [B, gamma_max + 1]      int32 (written)
 *   out_num_accepted [B]                   int32 (written)
 * Logit pointers must be aligned to their element size; the fast path is
 * taken when both are 16-byte aligned and V * element size is a multiple of
 * 16 bytes, a scalar-load path otherwise.  int32/float32 arrays must be
 * 4-byte aligned.  Outputs must not overlap inputs.
 * Where the inputs live.  Arrays the kernels only read (logits, tokens,
 * num_draft, uniforms, temperature) may be device memory or page-locked host
 * memory mapped into the device's address space (cudaHostAlloc, or
 * cudaHostRegister with cudaHostRegisterMapped); pass the address that
 * spec_device_pointer returns for it.  The kernels then read those bytes over
 * the host link while they run ("zero copy"): no staging copy is made, and the
 * early-exit kernel (options.kernel 3) moves only the rows it needs across
 * the link, each once where two row slices fit in shared memory (it keeps the
 * decided rows there for the final sample; host memory is not cached in L2).
 * The kernels read such memory after the call has returned, so the caller
 * keeps it allocated and unchanged until the stream has passed the call (for
 * example until an event recorded after the call completes).  Everything the
 * kernels write (outputs, status, counters, diagnostics) must be device
 * memory.
 *
 * Ownership and execution.  The caller owns every buffer.  The call enqueues
 * one kernel on 'stream' (a cudaStream_t; NULL = legacy default stream) and
 * returns without synchronising; it allocates no memory.  It is reentrant:
 * the only process-wide state is a per-device cache of kernel attributes.
 *
 * Errors.  Argument problems found on the host return an error code before
 * anything is enqueued.  Problems in the data never trap: a sequence with
 * num_draft outside [0, gamma_max], a temperature that is negative, NaN,
 * infinite or positive but below FLT_MIN, a drafted id outside [0, V) at a
 * position it uses, or a sampled row it uses whose logits have no finite
 * softmax normaliser (all -inf, any +inf or NaN) gets out_tokens[b, :] = -1
 * and out_num_accepted[b] = 0, and its SPEC_STATUS_* bit is OR-ed into
 * *status when status is not NULL (the caller zeroes it).  The kernels wait only
 * at hardware barriers that every thread of the CTA or cluster reaches.  NaN
 * logits in greedy rows give unspecified (in-range) tokens.
 *
 * Limits: 0 <= B <= SPEC_MAX_BATCH (B == 0 is a no-op), 0 <= gamma_max <=
 * SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_VOCAB.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_MAX_GAMMA 16
#define SPEC_MAX_VOCAB (1 << 24)
#define SPEC_MAX_BATCH (1 << 26)
#define SPEC_MAX_TREE_NODES 256

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* null pointer, size out of range, misaligned pointer */
    SPEC_ERR_UNSUPPORTED = 2, /* unknown dtype, or no usable launch shape on this device */
    SPEC_ERR_CUDA = 3         /* a CUDA runtime call or the launch failed */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Per-sequence data problems (bits OR-ed into *status). */
#define SPEC_STATUS_BAD_TOKEN 1u
#define SPEC_STATUS_BAD_TEMPERATURE 2u
#define SPEC_STATUS_BAD_NUM_DRAFT 4u
#define SPEC_STATUS_BAD_LOGITS 8u
/* spec_tree_verify: a node's parent is not an earlier node. */
#define SPEC_STATUS_BAD_TREE 32u

/* One verification round for B independent sequences (see the top of this
 * file for the operation, layout, ownership and errors).
 * status: optional device word (may be NULL) receiving SPEC_STATUS_* bits. */
spec_status spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                        const int32_t *num_draft, const float *uniforms, const float *temperature,
                        int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                        spec_dtype dtype, uint32_t *status, void *stream);

/* Launch options (tuning, A/B measurement and the early-exit variant).  They
 * change no decision except one that lies very close to its boundary: the
 * normalisers are merged from per-CTA partials, so the split of a row (the
 * cluster size) and the kernel variant move p-hat and q-hat by about 1e-7
 * relative, and an accept test that close to its threshold (or a final draw
 * within ~1e-9 of a CDF boundary) may come out differently.  Greedy (T == 0)
 * results never change. */
typedef struct spec_verify_options {
    int cluster_size; /* CTAs sharing one sequence's rows: 0 = automatic, else 1 to 16 */
    int kernel;       /* 0 = automatic: the early exit (3) when the full sweep's grid would
                             fill more than half of the device's resident CTA slots or the
                             rows are tiny (V * element size <= 8 KB), else the full sweep (2);
                         1 = not a kernel (SPEC_ERR_INVALID_ARG);
                         2 = full sweep, register loads;
                         3 = row-ordered early exit: position i's rows are read, reduced
                             and tested before position i+1's, and no row after the first
                             rejection is read (n+1 target and min(n+1, g) draft rows per
                             sequence; the method needs nothing after the cut, "Speculative
                             Decoding" ch.2).  Diagnostics then cover the rows read only. */
    uint64_t *counters; /* optional device array [3] (8-byte aligned), accumulated with atomics:
                           += drafted ids, += accepted ids, += verified sequences (valid ones).
                           Their ratio is the acceptance rate; accepted / sequences + 1 the mean
                           tokens per round (the counts a serving engine exports, per
                           "Speculative Decoding으로 LLM 추론 속도 높이기", vLLM section).  NULL: none. */
    uint64_t *accept_hist; /* optional device array [SPEC_MAX_GAMMA + 1] (8-byte aligned): += 1 at
                              index n (accepted count; min(n, SPEC_MAX_GAMMA) for trees) for each
                              verified sequence, the distribution behind the mean.  NULL: none. */
} spec_verify_options;

/* Same round, plus optional float32 diagnostics for tests (any may be NULL):
 *   p_hat [B, gamma_max]     p_i(x_i) for i < g of sampled sequences, NaN elsewhere
 *   q_hat [B, gamma_max]     q_i(x_i), same positions
 *   logz_t [B, gamma_max+1]  natural-log normaliser log sum_j exp(l_j / T) of
 *                            target rows i <= g of sampled sequences, NaN elsewhere
 *   logz_d [B, gamma_max]    same for draft rows i < g
 *   resid_mass [B]           total weight S of the decided row of a sampled
 *                            sequence (residual mass, or ~1 for a bonus row)
 *   seq_status [B]           SPEC_STATUS_* bits of each sequence (0 = valid)
 * The diagnostic rows are computed for every i <= g, also after the cut (with
 * the full-sweep kernels; options.kernel 0 takes the full sweep here).  A sequence with a data problem (seq_status != 0)
 * may carry partial diagnostics: the rows swept before the problem was found.
 * options: as for spec_verify_ex (NULL = automatic). */
spec_status spec_verify_debug(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                              const int32_t *num_draft, const float *uniforms, const float *temperature,
                              int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                              spec_dtype dtype, uint32_t *status, void *stream, float *p_hat, float *q_hat,
                              float *logz_t, float *logz_d, float *resid_mass, int32_t *seq_status,
                              const spec_verify_options *options);

/* spec_verify with explicit launch options (NULL = automatic).  Returns
 * SPEC_ERR_UNSUPPORTED if the device cannot co-schedule the requested shape. */
spec_status spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                           const int32_t *num_draft, const float *uniforms, const float *temperature,
                           int32_t *out_tokens, int32_t *out_num_accepted, int B, int gamma_max, int V,
                           spec_dtype dtype, uint32_t *status, void *stream, const spec_verify_options *options);

/* Sampling from one distribution per sequence: y_b ~ softmax(logits[b, :] / T_b)
 * by inverse CDF with u = uniforms[b] (the smallest id j with u * S < C_j), or
 * y_b = argmax logits[b, :] (lowest id on ties) when T_b == 0.  This is the
 * verification round with no drafts: the draft-side sampling of a proposer
 * ("Fast Inference from Transformers via Speculative Decoding" notes, method
 * details step 1: x ~ q) and target-only decoding, with the same kernels.
 *   logits [B, V] dtype; uniforms [B] float32 in [0, 1); temperature [B];
 *   out_tokens [B] int32 (-1 for a sequence with an invalid temperature or a
 *   sampled row without a finite normaliser; its bit goes to *status).
 * options: as for spec_verify_ex.
 * Same ownership, stream and error rules as spec_verify. */
spec_status spec_sample(const void *logits, const float *uniforms, const float *temperature, int32_t *out_tokens,
                        int B, int V, spec_dtype dtype, uint32_t *status, void *stream,
                        const spec_verify_options *options);

/* Prompt-lookup (n-gram) proposer: drafts without a model.  "Speculative
 * Decoding" (atonlee.tistory.com/330) ch.5: find the current suffix earlier in
 * the context and propose the tokens that followed it; the vLLM section of
 * "Speculative Decoding으로 LLM 추론 속도 높이기" sets the n-gram lengths with
 * prompt_lookup_min / prompt_lookup_max.  For each sequence b, with
 * L = context_len[b] tokens in context[b * context_stride, +L): the longest
 * n in [min_n, max_n] whose last-n-token suffix also occurs at an earlier start
 * j < L - n wins, and among its occurrences the most recent one; the proposal
 * is the min(gamma_max, L - (j + n)) tokens after it.  No occurrence: no
 * drafts.
 *   context        int32, row b starts at b * context_stride (device memory,
 *                  or mapped host memory as for spec_verify)
 *   context_len    [B] int32, clamped to [0, context_stride]
 *   draft_tokens   [B, gamma_max] int32 (written; -1 after the proposal)
 *   num_draft      [B] int32 (written)
 * Limits: 1 <= min_n <= max_n <= 64, 0 <= gamma_max <= SPEC_MAX_GAMMA.  One
 * kernel on 'stream'; allocates nothing.  The proposals feed spec_verify with
 * draft_logits == NULL (point-mass proposals). */
spec_status spec_ngram_propose(const int32_t *context, int64_t context_stride, const int32_t *context_len, int B,
                               int min_n, int max_n, int gamma_max, int32_t *draft_tokens, int32_t *num_draft,
                               void *stream);

/* Candidate-tree verification: one round in which the target checked a tree
 * of candidates in one forward ("Speculative Decoding" (atonlee.tistory.com/
 * 330) ch.5: Medusa heads propose their top few tokens per position, the
 * combinations form a tree checked through a tree attention mask; the EAGLE
 * paragraph of "Speculative Decoding으로 LLM 추론 속도 높이기": EAGLE-2 drafts
 * a tree).  For each sequence b with nn = num_nodes[b] nodes:
 *   node 0 is the root (the last emitted token); node k in [1, nn) carries the
 *   candidate id tokens[b, k] and hangs under parent[b, k] in [0, k);
 *   target_logits[b, k, :] is the target's next-token logits after the path
 *   root..k (row 0: after the root).
 * The candidates are deterministic (a proposer's top tokens), i.e. point
 * masses.  Walking from the root, the children of the current node are tried
 * in index order with the single-candidate rule ("Speculative Decoding"
 * ch.3) applied to p without the ids already rejected there (R): child c is
 * accepted iff uniforms[b, c] * (1 - p(R)) < p(tokens[b, c]), p = softmax(row /
 * T_b); the first accepted child becomes the current node.  When none is (or
 * the node is a leaf), one token is sampled from p without R, renormalised,
 * by inverse CDF with uniforms[b, 0] (smallest j with u*S < C_j on the exact
 * fixed-point grid), which keeps the target's law at every step; with one
 * child per node this is spec_verify with point-mass drafts.  T_b == 0: the
 * accepted child is the first whose id is the argmax of the node's raw
 * logits (lowest id on ties), and the walk ends by emitting that argmax.
 * Only the rows on the accepted path are read.
 *   target_logits  [B, max_nodes, V] dtype; rows of nodes >= nn are never read
 *   parent, tokens [B, max_nodes] int32 (entries 0 and >= nn ignored)
 *   num_nodes      [B] int32 in [1, max_nodes]
 *   uniforms       [B, max_nodes] float32 in [0, 1): column c tests node c,
 *                  column 0 drives the final sample
 *   temperature    [B] float32 (0: greedy)
 *   out_tokens     [B, max_nodes] int32: the n accepted ids, then the sampled
 *                  (or argmax) id, then -1
 *   out_num_accepted [B] int32: n, the accepted path length
 *   out_path       [B, max_nodes] int32 or NULL: the accepted node indices,
 *                  then -1 (for keeping their cache entries)
 * Invalid data (num_nodes outside [1, max_nodes], a parent outside [0, k), a
 * candidate id outside [0, V), a bad temperature, a sampled row on the path
 * without a finite normaliser) gives -1 tokens, n = 0 and a status bit
 * (SPEC_STATUS_BAD_NUM_DRAFT for num_nodes, SPEC_STATUS_BAD_TREE, ...).
 * options: cluster_size and counters as for spec_verify_ex (counters add
 * nn - 1 candidates, n accepted, 1 sequence); kernel must be 0.  Limits:
 * 1 <= max_nodes <= SPEC_MAX_TREE_NODES, 1 <= V <= SPEC_MAX_VOCAB.  Same
 * ownership, stream and error rules as spec_verify; allocates nothing. */
spec_status spec_tree_verify(const void *target_logits, const int32_t *parent, const int32_t *tokens,
                             const int32_t *num_nodes, const float *uniforms, const float *temperature,
                             int32_t *out_tokens, int32_t *out_num_accepted, int32_t *out_path, int B,
                             int max_nodes, int V, spec_dtype dtype, uint32_t *status, void *stream,
                             const spec_verify_options *options);

/* Launch shape spec_verify would use on the current device for these sizes
 * (device-memory rows): cluster size (CTAs per sequence), total CTAs, threads
 * per CTA and the kernel the automatic choice takes (2 = full sweep, 3 = early
 * exit; see spec_verify_options.kernel).  Any output pointer may be NULL.
 * Touches the device (attribute queries) but enqueues nothing. */
spec_status spec_verify_launch_shape(int B, int gamma_max, int V, spec_dtype dtype, int *cluster_size,
                                     int *num_ctas, int *threads_per_cta, int *kernel);

/* The address the kernels use for ptr: ptr itself for this device's memory,
 * the device alias for page-locked host memory mapped into the device's
 * address space (with unified addressing, the same value).  Returns
 * SPEC_ERR_INVALID_ARG (and leaves *device_ptr unchanged) for pageable or
 * unregistered host memory, another device's memory or a NULL argument, and
 * SPEC_ERR_CUDA if the runtime query fails.  Enqueues nothing. */
spec_status spec_device_pointer(const void *ptr, const void **device_ptr);

/* Static description of a status code. */
const char *spec_status_string(spec_status s);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
