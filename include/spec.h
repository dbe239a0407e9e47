/*
 * spec.h - C ABI of the GB300 (sm_103a) block-speculative-decoding hot path.
 *
 * Three operations on vocabulary-wide logit rows, each one or two CUDA kernels:
 *
 *   spec_draft_block  DSpark low-rank Markov logit bias + softmax + argmax/sample
 *                     over a parallel drafter's gamma positions.
 *   spec_verify       target verification of gamma draft tokens against gamma+1
 *                     target rows: accepted length, committed tokens, bonus token.
 *   spec_e2etv        SpecOPD E2E-TV surrogate: overlap 1-TV, prefix survival,
 *                     mean loss and its gradient w.r.t. the draft logits.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every array argument is a DEVICE pointer owned by the caller.  The
 *           library allocates nothing and keeps no per-call global state.
 *           Scratch lives in a caller-supplied workspace (see below).
 * Layout.   Row-major, contiguous.  A "row" is V consecutive elements.
 * Dtypes.   Logits are float32 or bfloat16 (stored as raw 16-bit words); every
 *           reduction accumulates in float32.  Tokens are int32 in [0, V).
 * Align.    Every logits/weights base pointer must be 16-byte aligned (rejected
 *           with SPEC_ERR_ALIGN otherwise).  V need not be a multiple of anything:
 *           rows whose byte length is not a multiple of 16 take a scalar path.
 * Streams.  Calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *           stream) and never synchronise the host.
 * Errors.   Argument errors are returned synchronously before anything is
 *           enqueued.  A failed CUDA launch returns SPEC_ERR_CUDA.  Conditions met
 *           on the device (a non-finite row, a token out of range, a bounded wait
 *           that ran out) are OR-ed as flags into a status word inside the
 *           workspace; read them with spec_get_device_status.  Affected requests
 *           also get -1 outputs (see each call).
 * Invalid rows.  A logit of -inf is a token of probability zero.  A row that holds
 *           NaN or +inf, or no finite entry, has no distribution: the request that
 *           reads it is reported with -1 tokens and the SPEC_DEV_NONFINITE flag.
 * Workspace.  Query the size with spec_workspace_bytes, allocate it on the device,
 *           and zero it ONCE with spec_workspace_init before its first use.  Every
 *           call returns the counters, keys and flags it relies on to zero (its
 *           other contents are scratch that the call writes before it reads them),
 *           so later calls of the SAME operation and shape reuse it as it is, on
 *           the same stream.  Before a call with another operation or shape, run
 *           spec_workspace_init again (or use a separate workspace): its counters
 *           sit where the earlier call left scratch.  Calls that run concurrently
 *           need separate workspaces.  After a SPEC_DEV_TIMEOUT flag, run
 *           spec_workspace_init again before reusing it.
 * Randomness.  T=1 draws use Philox4x64-10 (Salmon et al., SC'11) with key
 *           (seed_b, 0) and counter (b, j, stream, 0); the uniform is
 *           (word0 >> 40) * 2^-24.  Streams: 0 draft sample, 1 accept test,
 *           2 residual draw, 3 bonus draw.  Any call replays bit for bit.
 * Sampling.  Single-uniform inverse CDF in vocabulary order: the smallest v with
 *           C_v > u * Z (C_v running sum of the weights, Z their total).  Argmax
 *           ties go to the lowest index.
 */
#ifndef SPEC_GB300_SPEC_H
#define SPEC_GB300_SPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (CUDA declares it as struct CUstream_st *). */
struct CUstream_st;
typedef struct CUstream_st *spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* null pointer, bad temperature, bad op code        */
    SPEC_ERR_SHAPE = 2,       /* a size outside the supported range               */
    SPEC_ERR_DTYPE = 3,       /* unknown dtype code                               */
    SPEC_ERR_ALIGN = 4,       /* a base pointer that is not 16-byte aligned       */
    SPEC_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed             */
    SPEC_ERR_TIMEOUT = 6,     /* device: a bounded wait gave up                   */
    SPEC_ERR_NONFINITE = 7,   /* device: a row with NaN/+inf or no finite entry   */
    SPEC_ERR_TOKEN = 8,       /* device: a token outside [0, V)                   */
    SPEC_ERR_WORKSPACE = 9    /* workspace null or smaller than required          */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
    SPEC_OP_DRAFT = 0,
    SPEC_OP_VERIFY = 1,
    SPEC_OP_E2ETV = 2,
    SPEC_OP_DRAFT_VERIFY = 3,
    SPEC_OP_BRANCH_PLAN = 4,
    SPEC_OP_VERIFY_TOPK = 5,
    SPEC_OP_TREE_VERIFY = 6,
    SPEC_OP_DRAFT_TOPK = 7
} spec_op;

/* Device status flags (OR-ed into the workspace status word). */
#define SPEC_DEV_TIMEOUT 1u
#define SPEC_DEV_NONFINITE 2u
#define SPEC_DEV_TOKEN 4u

/* Supported ranges. */
#define SPEC_MAX_GAMMA 64      /* draft positions per request                      */
#define SPEC_MAX_RANK 256      /* Markov rank r                                    */
#define SPEC_MAX_V (1 << 26)   /* vocabulary size                                  */
#define SPEC_MAX_DRAFT_ROWS (1 << 20)   /* spec_draft_block: B * gamma             */
#define SPEC_MAX_TRUNK 16384   /* spec_branch_plan: tokens of one reference        */
#define SPEC_MAX_TOP_K 32      /* spec_verify_topk: largest top_k                  */
#define SPEC_MAX_V_DRAFT_TOPK (1 << 19)   /* spec_draft_block_topk: vocabulary size */
#define SPEC_MAX_TREE_NODES 1024  /* spec_tree_select / spec_tree_verify: nodes per tree */

/*
 * spec_workspace_bytes - workspace size for one operation (host only, pure).
 *   op     SPEC_OP_DRAFT / SPEC_OP_VERIFY / SPEC_OP_DRAFT_VERIFY: B requests, gamma
 *          positions, V, r.
 *          SPEC_OP_E2ETV: B = number of branches, gamma = branch length Wb, r unused.
 *          SPEC_OP_BRANCH_PLAN: the status word only (pass B = references, gamma =
 *          W, V = Lmax, r = 0).
 *          SPEC_OP_VERIFY_TOPK: B requests, gamma positions (V and r unused).
 *          SPEC_OP_TREE_VERIFY: B = trees, gamma = nodes per tree (0 allowed, up to
 *          SPEC_MAX_TREE_NODES), V, r unused.
 *          SPEC_OP_DRAFT_TOPK: B requests, V entries (gamma and r unused).
 *          For SPEC_OP_DRAFT the size covers one launch's slice of requests, which
 *          spec_draft_block reuses across the slices of a larger batch.
 * Returns 0 for arguments outside the supported ranges.
 */
size_t spec_workspace_bytes(spec_op op, int B, int gamma, int V, int r);

/* spec_workspace_init - zero `bytes` of workspace on `stream` (asynchronous). */
spec_status spec_workspace_init(void *workspace, size_t bytes, spec_stream_t stream);

/*
 * spec_get_device_status - synchronise `stream`, read the workspace status word.
 * Writes the raw SPEC_DEV_* flags to *flags_out (nullable) and returns SPEC_OK when
 * no flag is set, else the status of the most severe flag (TIMEOUT, then TOKEN,
 * then NONFINITE).  Flags stay set until spec_workspace_init.
 */
spec_status spec_get_device_status(const void *workspace, spec_stream_t stream,
                                   uint32_t *flags_out);

/* spec_status_string - static description of a status code. */
const char *spec_status_string(spec_status status);

/*
 * spec_last_cuda_error - the CUDA runtime error code behind the most recent
 * SPEC_ERR_CUDA returned on the calling host thread (0 if none), and its message.
 * Kept per host thread, like errno; no other call state is kept.
 */
int spec_last_cuda_error(void);
const char *spec_last_cuda_error_string(void);

/*
 * spec_draft_block - DSpark block draft with the rank-r Markov logit bias.
 *
 * Defines ("Speculative Decoding Part 2", VESSL AI, DSpark section, bias equation;
 * "Solar Open2 DSpark", sionic.ai, section 2): for request b and positions
 * j = 1..gamma, with x_0 = anchor[b],
 *     z_j = l_j + W_1[x_{j-1}] W_2          (W_1 = U [V, r], W_2 = Wt^T)
 *     m = max z_j,  Z = sum_v exp(z_j,v - m),  c_j = 1/Z  (the max probability)
 *     T=0: x_j = lowest index attaining m
 *     T=1: x_j = inverse-CDF draw from softmax(z_j), u = Philox(seed_b; b, j, 0)
 *     q_j(x_j) = exp(z_j,x_j - m) / Z
 * computed exactly as this sequential recurrence defines it (the library solves it
 * by fixed-point passes over all positions at once; the result is the sequential
 * one).
 *
 *   draft_logits  [B, gamma, V], dtype logits_dtype; row (b, j-1) is l_j.
 *   anchor        [B] int32, x_0 of each request.
 *   U, Wt         [V, r] each, dtype w_dtype (both the same).  U row x is W_1[x];
 *                 Wt row v is column v of W_2 (the nn.Linear(r, V) weight layout).
 *                 r = 0 means no bias; U and Wt may then be NULL.
 *   temperature   0 (argmax) or 1 (sample at temperature 1).
 *   seeds         [B] uint64 Philox keys; required when temperature == 1.
 *   tokens_out    [B, gamma] int32.
 *   conf_out      [B, gamma] float32, c_j.
 *   qtok_out      [B, gamma] float32, q_j(x_j) (nullable).
 *   qlogits_out   [B, gamma, V] float32, the biased logits z_j the draws used
 *                 (nullable; pass it to spec_verify as the T=1 draft rows).
 *   passes_out    [1] int32 (nullable): biased fixed-point passes, up to the first
 *                 that changes no token, at most gamma (at T=1 a pass recomputes only
 *                 the rows whose predecessor changed in the pass before, and a pass
 *                 with no such row is counted without being run); gamma when the
 *                 chain is walked position by position.
 * A request whose anchor lies outside [0, V), or whose row j is invalid, gets
 * tokens -1 and NaN statistics from that position on (flags TOKEN / NONFINITE).
 * More than 256 rows with bf16 logits and weights, r a multiple of 64, V a multiple
 * of 8 and no qlogits_out: the chain is walked position by position on the tensor
 * cores, each position reading its rows and W once, in slices of up to 1024
 * requests.  Otherwise a batch larger than one launch takes (256 rows on the
 * tensor-core path: bf16 weights with r a multiple of 64; 4096 rows otherwise) runs
 * as consecutive launches over slices of requests on `stream`, and passes_out is the
 * largest over the slices.  Either way the results are those of one call (the Philox
 * request index b is the request's index in the whole batch).
 * Limits: 1 <= gamma <= SPEC_MAX_GAMMA, 0 <= r <= SPEC_MAX_RANK, 1 <= V <= SPEC_MAX_V,
 * 1 <= B*gamma <= SPEC_MAX_DRAFT_ROWS.
 */
spec_status spec_draft_block(const void *draft_logits, spec_dtype logits_dtype,
                             const int32_t *anchor, const void *U, const void *Wt,
                             spec_dtype w_dtype, int r, int B, int gamma, int V,
                             int temperature, const uint64_t *seeds, int32_t *tokens_out,
                             float *conf_out, float *qtok_out, float *qlogits_out,
                             int32_t *passes_out, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/*
 * spec_verify - verify gamma draft tokens against gamma+1 target rows.
 *
 * Defines ("Solar Open2 DSpark", sionic.ai, sections 1 and 6: one target forward
 * over gamma+1 positions checks the drafts and commits the agreeing prefix;
 * "Speculative Decoding Part 2", VESSL AI, blockwise decoding section: the longest
 * matching prefix is accepted).  Target row i is the distribution of position i+1.
 *     T=0: n = largest k with x_j == argmax(target row j-1) for all j <= k;
 *          y = argmax(target row n).
 *     T=1: for j = 1..gamma: accept iff u_j * q_j(x_j) < p_j(x_j), u_j =
 *          Philox(seed_b; b, j, 1); at the first rejection k, y is drawn from
 *          max(0, p_k - q_k) normalised (from p_k if that is all zero) with
 *          Philox(seed_b; b, k, 2); if all are accepted, y is drawn from
 *          p_{gamma+1} with Philox(seed_b; b, gamma+1, 3).  p = softmax(target
 *          row), q = softmax(draft row), both at temperature 1.
 *   target_logits   [B, gamma+1, V], dtype target_dtype.
 *   draft_logits    [B, gamma, V], dtype draft_dtype (may be the float32
 *                   qlogits_out of spec_draft_block); ignored and nullable at T=0.
 *   draft_tokens    [B, gamma] int32.
 *   seeds           [B] uint64, required at T=1.
 *   n_accepted_out  [B] int32 in [0, gamma]; the acceptance length as the pages
 *                   count it (with the bonus) is n + 1.
 *   committed_out   [B, gamma+1] int32: x_1..x_n, y, then -1.
 *   bonus_out       [B] int32: y.
 *   near_tie_out    [B] int32 (nullable): 1 when some draw of the request landed
 *                   within 1e-6 (relative) of its decision threshold, where float32
 *                   and exact arithmetic may legitimately decide differently.
 * An invalid request (a token outside [0, V) or an invalid row it reads) gets
 * n = -1, committed all -1 and bonus -1.
 * Limits: 1 <= gamma <= SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_V, 1 <= B <= 65535.
 */
spec_status spec_verify(const void *target_logits, spec_dtype target_dtype,
                        const void *draft_logits, spec_dtype draft_dtype,
                        const int32_t *draft_tokens, int B, int gamma, int V, int temperature,
                        const uint64_t *seeds, int32_t *n_accepted_out, int32_t *committed_out,
                        int32_t *bonus_out, int32_t *near_tie_out, void *workspace,
                        size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_draft_verify - one greedy (T=0) block step: spec_draft_block followed by
 * spec_verify of its tokens against the target rows, in one call.
 *
 * Defines: the draft-then-verify cycle ("Solar Open2 DSpark", sionic.ai, sections 1
 * and 6: the drafter proposes a block, one target forward over gamma+1 positions
 * commits the agreeing prefix and the target's next token), with each half defined
 * as in spec_draft_block (temperature 0) and spec_verify (temperature 0).  The
 * outputs equal those of the two calls made in sequence, bit for bit: tokens_out,
 * conf_out, qtok_out and passes_out as spec_draft_block writes them; n_accepted_out,
 * committed_out and bonus_out as spec_verify writes them for those tokens.
 *
 * It runs the draft kernel and, as its programmatic dependent, the verify kernel:
 * one workspace and one call for the common greedy step.
 *
 *   draft_logits .. V   as spec_draft_block.
 *   target_logits       [B, gamma+1, V], dtype target_dtype; target row i is the
 *                       distribution of position i+1.
 *   tokens_out, conf_out  [B, gamma]; qtok_out [B, gamma] (nullable); passes_out [1]
 *                       (nullable).
 *   n_accepted_out [B], committed_out [B, gamma+1], bonus_out [B]  as spec_verify.
 *   workspace           spec_workspace_bytes(SPEC_OP_DRAFT_VERIFY, B, gamma, V, r).
 * Limits: those of spec_draft_block.  Device conditions of either half set the same
 * status flags in this one workspace.
 */
spec_status spec_draft_verify(const void *draft_logits, spec_dtype logits_dtype,
                              const int32_t *anchor, const void *U, const void *Wt,
                              spec_dtype w_dtype, int r, int B, int gamma, int V,
                              const void *target_logits, spec_dtype target_dtype,
                              int32_t *tokens_out, float *conf_out, float *qtok_out,
                              int32_t *passes_out, int32_t *n_accepted_out,
                              int32_t *committed_out, int32_t *bonus_out, void *workspace,
                              size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_noalloc - spec_verify without a caller-supplied workspace.
 *
 * No counterpart in the pages: it exists for callers that cannot allocate device
 * memory, such as a plugin running inside a host program whose own allocator owns
 * the GPU's memory and lends none of it out, or a serving process that has given
 * nearly all device memory to a caching pool (where one more cudaMalloc fails, and
 * synchronises the device on a latency-critical path even when it succeeds).  It
 * computes exactly what spec_verify computes, with the same arguments and outputs
 * minus `workspace` and `workspace_bytes`, and calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Scratch.  The workspace lives in a static device array of
 * SPEC_NOALLOC_SCRATCH_BYTES that the library holds on every GPU that loads it, until
 * the process exits.  A problem whose spec_workspace_bytes(SPEC_OP_VERIFY, B, gamma,
 * V, 0) exceeds that size is rejected with SPEC_ERR_SHAPE before anything is
 * enqueued (B = 32, gamma = 7, V = 248,320 needs about 1.05 MB).
 * Sharing.  Every call on a device uses the same array, which keeps the previous
 * call's contents: each call first clears the bytes it needs (an asynchronous memset
 * on `stream`).  Calls whose work overlaps on the GPU (issued on different streams,
 * or from several host threads without ordering) race on the array and give wrong
 * results; order them on one stream.
 * Set-up.  The first call made with a given device current looks up the array's
 * device address (cudaGetSymbolAddress) and keeps it; make that first call before
 * any stream capture begins.
 * Device conditions (a non-finite row, a token out of range, a bounded wait that
 * ran out) show only as the -1 outputs of the requests concerned: the status word
 * is inside the array and is cleared by the next call.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (4u << 20)   /* 4 MiB */
spec_status spec_verify_noalloc(const void *target_logits, spec_dtype target_dtype,
                                const void *draft_logits, spec_dtype draft_dtype,
                                const int32_t *draft_tokens, int B, int gamma, int V,
                                int temperature, const uint64_t *seeds,
                                int32_t *n_accepted_out, int32_t *committed_out,
                                int32_t *bonus_out, int32_t *near_tie_out,
                                spec_stream_t stream);

/*
 * spec_verify_budget - how many draft positions of each request to verify.
 *
 * Defines: "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL
 * AI), DSpark section, the paragraphs after the bias equation.  The confidence of a
 * position (spec_draft_block's conf_out) is the probability that it passes given that
 * every earlier position passed; the scheduler multiplies these into expected lengths
 * and gives the verification budget to the most likely positions across the batch,
 * maximising throughput against a measured cost curve.  The pages give no formula;
 * the reading is:
 *   P[b][j] = prod_{i <= j} c[b][i], each c clamped to [0, 1] and NaN read as 0,
 *   computed in float64 in position order;
 *   candidates (b, j) ordered by P descending, ties by b * gamma + j ascending (the
 *   first k candidates hold a prefix of every request's positions);
 *   E(k) = B + sum of the first k P: expected committed tokens with k positions
 *   verified in all (each request commits its accepted drafts plus one token);
 *   k* = the k in 0..budget with the largest E(k) / cost_us[k], the smallest on ties,
 *   an entry that is not positive and finite left out (no usable entry: k* = 0); with
 *   cost_us NULL, k* = budget;
 *   gamma_out[b] = request b's positions among the first k*.
 *
 *   conf          float32 device [B, gamma].
 *   budget        0 <= budget <= B * gamma: most positions verified in all.
 *   cost_us       float32 device [budget + 1] or NULL: time to verify k positions.
 *   gamma_out     int32 device [B].
 *   expected_out  float32 device [1] or NULL: E(k*).
 * Limits: 1 <= gamma <= SPEC_MAX_GAMMA, 1 <= B * gamma <= SPEC_MAX_BUDGET_CANDIDATES.
 * Arguments are checked before anything is enqueued; one CTA does the work (no
 * workspace, nothing allocated).
 */
#define SPEC_MAX_BUDGET_CANDIDATES 8192
spec_status spec_verify_budget(const float *conf, int B, int gamma, int budget, const float *cost_us,
                               int32_t *gamma_out, float *expected_out, spec_stream_t stream);

/*
 * spec_e2etv - SpecOPD E2E-TV surrogate and its gradient.
 *
 * Defines ("SpecOPD" paper summary, onedev.kr, section "how to use it"; VESSL AI
 * "Speculative Decoding Part 2", DSpark section: alpha = 1 - D_TV).  Rows are
 * branch-major: row n*Wb + i is position i of branch n.  p = softmax(target row),
 * q = softmax(draft row):
 *     a_{n,i} = sum_v min(p_v, q_v),   s_{n,i} = sum_{q_v < p_v} q_v
 *     S_{n,j} = prod_{i<=j} a_{n,i},   loss = 1 - mean_{n,j} S_{n,j}
 *     grad_{n,i,v} = dloss/dz_{n,i,v} = -kappa_{n,i} q_v (1[q_v < p_v] - s_{n,i}),
 *     kappa_{n,i} = (1/(N*Wb)) sum_{j>=i} prod_{k<=j, k!=i} a_{n,k}
 * The target is held fixed (no gradient w.r.t. the target logits).
 *   target_logits, draft_logits  bf16 [N*Wb, V].
 *   a_out, surv_out              [N*Wb] float32: a and S.
 *   loss_out                     [1] float32.
 *   grad_out                     bf16 [N*Wb, V], rounded once from float32 (RNE).
 * A branch with an invalid row gets NaN a/surv, a zero gradient, and makes the
 * loss NaN (flag NONFINITE).
 * Limits: 1 <= Wb <= SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_V, 1 <= N*Wb <= 2^24.
 */
spec_status spec_e2etv(const uint16_t *target_logits, const uint16_t *draft_logits,
                       int n_branches, int Wb, int V, float *a_out, float *surv_out,
                       float *loss_out, uint16_t *grad_out, void *workspace,
                       size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_e2etv_shard - spec_e2etv on one shard of a batch split across processes (one
 * per GPU), for the same definitions over the whole batch of total_branches branches.
 * The rows are this shard's n_branches branches; every branch is independent, so a
 * shard needs nothing from the others except the loss's count: kappa and the gradient
 * use 1/(total_branches*Wb), and
 *   msum_out  [1] float32: this shard's part of the mean survival,
 *             sum over its branches and positions of S / (total_branches * Wb).
 * The loss of the whole batch is 1 - (the sum of msum_out over the shards): one scalar
 * all-reduce, left to the caller.  A shard with an invalid branch writes NaN.
 * Limits: those of spec_e2etv, and n_branches <= total_branches.  The workspace is
 * spec_workspace_bytes(SPEC_OP_E2ETV, n_branches, Wb, V, 0).
 */
spec_status spec_e2etv_shard(const uint16_t *target_logits, const uint16_t *draft_logits,
                             int n_branches, int Wb, int V, int total_branches, float *a_out,
                             float *surv_out, float *msum_out, uint16_t *grad_out,
                             void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_draft_block_topk - spec_draft_block at T=1 with top-k / top-p filtered draws.
 *
 * Defines ("Speculative Decoding Part 2", VESSL AI, DSpark section, bias equation; "DSpine
 * card numbers and public file headers", aiwithghost.com, section on raising the
 * temperature: sampling at T=1 with top_p 0.95 and top_k 20).  For request b and
 * j = 1..gamma, with x_0 = anchor[b]:
 *     z_j = l_j + W_1[x_{j-1}] W_2                     (as spec_draft_block)
 *     filter(z_j): spec_verify_topk's reading (the top_k largest logits renormalised,
 *     the shortest prefix in descending order reaching top_p, renormalised again)
 *     x_j = inverse-CDF draw from filter(z_j) in vocabulary-index order,
 *           u = Philox(seed_b; b, j, 0)
 *     c_j = 1/Z of the unfiltered softmax(z_j) (its largest probability)
 *     q_j(x_j) = filter(z_j)(x_j)
 *   draft_logits  [B, gamma, V], dtype logits_dtype.
 *   anchor        [B] int32.
 *   U, Wt         bf16 [V, r] (the layout of spec_draft_block), r a multiple of 16 up to
 *                 SPEC_MAX_RANK; r = 0 means no bias (U, Wt may then be NULL).
 *   top_k, top_p  1 <= top_k <= SPEC_MAX_TOP_K, 0 < top_p <= 1.
 *   seeds         [B] uint64.
 *   tokens_out    [B, gamma] int32; conf_out [B, gamma] float32; qtok_out [B, gamma]
 *                 float32 (nullable).
 *   workspace     spec_workspace_bytes(SPEC_OP_DRAFT_TOPK, B, gamma, V, r): about
 *                 B * V * 4 bytes (each position's biased logits are kept there for the
 *                 draw), 32 MB at B = 32, V = 248,320.
 * A request whose anchor lies outside [0, V) (flag TOKEN), or whose row j holds NaN or
 * +inf or no finite entry (flag NONFINITE), gets tokens -1 and NaN statistics from that
 * position on.  The chain is walked position by position (2 * gamma launches); the
 * weights are read once per position for every 32 requests.
 * Limits: 1 <= gamma <= SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_V_DRAFT_TOPK, 1 <= B <= 65535.
 */
spec_status spec_draft_block_topk(const void *draft_logits, spec_dtype logits_dtype, const int32_t *anchor,
                                  const void *U, const void *Wt, spec_dtype w_dtype, int r, int B, int gamma,
                                  int V, int top_k, double top_p, const uint64_t *seeds, int32_t *tokens_out,
                                  float *conf_out, float *qtok_out, void *workspace, size_t workspace_bytes,
                                  spec_stream_t stream);

/*
 * spec_verify_topk - spec_verify at T=1 against top-k / top-p filtered rows.
 *
 * Defines ("DSpine card numbers and public file headers", aiwithghost.com, section on
 * raising the temperature: sampling at T=1 with top_p 0.95 and top_k 20; the rejection
 * rule as for spec_verify).  The page names only the setting; the reading is:
 *   filter(row): the top_k largest logits (ties to the lowest index), renormalised over
 *   them; the kept set is the shortest prefix, in descending order, whose running sum
 *   reaches top_p (at least one entry); p_f is p on the kept set, renormalised.
 *   For j = 1..gamma: accept iff u_j * q_f(x_j) < p_f(x_j), u_j = Philox(seed_b; b, j, 1),
 *   with p_f from target row j-1 and q_f from draft row j-1; at the first rejection k,
 *   y is drawn from max(0, p_f - q_f) normalised (from p_f if that is all zero) with
 *   Philox(seed_b; b, k, 2); if all are accepted, y is drawn from the filtered target
 *   row gamma with Philox(seed_b; b, gamma+1, 3).  Draws are the inverse CDF in
 *   vocabulary-index order.
 *   target_logits, draft_logits, draft_tokens, seeds, outputs: as spec_verify at T=1.
 *   top_k   1 <= top_k <= SPEC_MAX_TOP_K.
 *   top_p   0 < top_p <= 1 (a double, so the cut-off is the caller's exact value).
 *   workspace  spec_workspace_bytes(SPEC_OP_VERIFY_TOPK, B, gamma, V, 0).
 * A request with a token outside [0, V) or a row without a distribution (NaN, +inf or
 * no finite entry) among its 2*gamma+1 rows gets n = -1, committed and bonus -1 (flag
 * TOKEN).  Limits: 1 <= B <= 65535, 1 <= gamma <= SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_V.
 */
spec_status spec_verify_topk(const void *target_logits, spec_dtype target_dtype,
                             const void *draft_logits, spec_dtype draft_dtype,
                             const int32_t *draft_tokens, int B, int gamma, int V, int top_k,
                             double top_p, const uint64_t *seeds, int32_t *n_accepted_out,
                             int32_t *committed_out, int32_t *bonus_out, int32_t *near_tie_out,
                             void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_branch_plan - SpecOPD anchor-branch plan: anchors on each reference response,
 * and the metadata that packs the branches drafted from them into one proposal tree.
 *
 * Defines ("SpecOPD" paper summary, onedev.kr, section "how it works": n anchors
 * picked at random on the reference, a branch of W tokens drafted from each,
 * independently; section "how it differs": the branches packed into a proposal tree,
 * each node seeing its own reference prefix and branch history through a parent map,
 * with rotary positions from semantic positions).  The pages give no formula; the
 * reading is:
 *   anchors of reference r (length L_r): the n distinct positions of 0..L_r-1 with
 *   the smallest (key, position), key = word0 >> 40 of Philox4x64-10 with key
 *   (seed, 0) and counter (r, i, 4, 0); every n-subset is equally likely; listed in
 *   ascending position;
 *   packing of reference r: trunk tokens are nodes 0..L_r-1 (node i's parent is
 *   i-1); branch k, step t = 1..W is node L_r + k*W + t-1, its parent a_k when t = 1
 *   and the node before otherwise, its semantic position a_k + t.
 * The branch tokens come from spec_draft_block with B = n_refs * n_anchors,
 * gamma = W, anchor = anchor_tok_out and the drafter's logits for each anchor.
 *
 *   trunk_tokens    int32 device [n_refs, Lmax].
 *   lengths         int32 device [n_refs], L_r.
 *   anchors_out     int32 device [n_refs, n_anchors]: a_k.
 *   anchor_tok_out  int32 device [n_refs, n_anchors]: trunk token at a_k (x_0).
 *   parent_out      int32 device [n_refs, n_anchors * W]: parent node of each branch
 *                   node, (k, t) at k*W + t-1.
 *   position_out    int32 device [n_refs, n_anchors * W]: semantic positions.
 *   workspace       spec_workspace_bytes(SPEC_OP_BRANCH_PLAN, ...) (the status word).
 * A reference with L_r < n_anchors or L_r > Lmax gets -1 everywhere (flag TOKEN).
 * Limits: 1 <= n_refs <= 65535, 1 <= n_anchors <= Lmax <= SPEC_MAX_TRUNK,
 * 1 <= W <= SPEC_MAX_GAMMA.
 */
spec_status spec_branch_plan(const int32_t *trunk_tokens, const int32_t *lengths, int n_refs,
                             int Lmax, int n_anchors, int W, uint64_t seed, int32_t *anchors_out,
                             int32_t *anchor_tok_out, int32_t *parent_out, int32_t *position_out,
                             void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_tree_select - EAGLE-2 top-m selection of draft-tree nodes by path product.
 *
 * Defines ("Speculative Decoding Part 2: the evolution of drafter architectures", VESSL
 * AI, EAGLE section: EAGLE-2 scores each branch of a dynamic draft tree by the product
 * of the confidences from the root and keeps the highest-scored nodes; a parent scores
 * at least as high as its children, so the kept set holds every kept node's parent).
 * The page gives no formula; the reading is:
 *   nodes 0..n-1 of a tree in topological order: parent[i] is -1 (the root, the last
 *   committed token) or an earlier node;
 *   score[i] = c[i] * score[parent[i]] (1 at the root), c = conf clamped to [0, 1] with
 *   NaN read as 0, in float64;
 *   the m nodes with the largest scores are kept, ties to the lower index.
 *
 *   parent        int32 device [n_trees, n_nodes].
 *   conf          float32 device [n_trees, n_nodes]: the drafter's confidence of each
 *                 node given its parent (e.g. spec_draft_block's conf_out).
 *   m             nodes kept per tree, 0 <= m (all nodes when m >= n_nodes).
 *   score_out     float64 device [n_trees, n_nodes] (nullable): the scores.
 *   keep_out      int32 device [n_trees, n_nodes]: 1 for a kept node, else 0.
 *   selected_out  int32 device [n_trees, m] (nullable): the kept nodes in ascending
 *                 index order, then -1.
 * A tree with a parent outside [-1, i) gets NaN scores, no kept node and -1 in
 * selected_out (there is no workspace and no status word).
 * Limits: 1 <= n_trees <= 65535, 1 <= n_nodes <= SPEC_MAX_TREE_NODES.  One CTA per
 * tree; nothing is allocated.
 */
spec_status spec_tree_select(const int32_t *parent, const float *conf, int n_trees, int n_nodes, int m,
                             double *score_out, int32_t *keep_out, int32_t *selected_out,
                             spec_stream_t stream);

/*
 * spec_tree_verify - T=0 verification of draft trees.
 *
 * Defines ("Speculative Decoding Part 2", VESSL AI, EAGLE section: verification of an
 * EAGLE-2 draft tree; "Solar Open2 DSpark", sionic.ai, sections 1 and 6: the target
 * commits the longest agreeing prefix and its next token).  The reading is:
 *   the target row of the root is row 0 of the tree and that of node i is row 1 + i
 *   (the distribution of the position after the node's token);
 *   from the root, move to the kept child whose token is the argmax of the current
 *   node's row (the lowest index among such children; argmax ties to the lowest
 *   vocabulary index), and stop when there is none;
 *   n = nodes passed; committed = their tokens in path order, then y = argmax of the
 *   last node's row (the bonus).
 * A chain (parent[i] = i - 1) is exactly spec_verify at T=0.
 *
 *   target_logits   [n_trees, n_nodes + 1, V], dtype target_dtype; the rows of nodes
 *                   that are not kept are never read.
 *   parent, token   int32 device [n_trees, n_nodes] (NULL allowed when n_nodes == 0).
 *   keep            int32 device [n_trees, n_nodes] (nullable: every node kept); e.g.
 *                   spec_tree_select's keep_out.
 *   n_accepted_out  int32 device [n_trees].
 *   path_out        int32 device [n_trees, n_nodes]: the accepted nodes, then -1.
 *   committed_out   int32 device [n_trees, n_nodes + 1]: their tokens, y, then -1.
 *   bonus_out       int32 device [n_trees]: y.
 *   workspace       spec_workspace_bytes(SPEC_OP_TREE_VERIFY, n_trees, n_nodes, V, 0).
 * A tree with a parent outside [-1, i) (flag TOKEN), or whose walk reaches a row without
 * a distribution (NaN, +inf or no finite entry; flag NONFINITE), gets n = -1 and -1
 * everywhere.  A token outside [0, V) never matches.
 * Limits: 1 <= n_trees <= 65535, 0 <= n_nodes <= SPEC_MAX_TREE_NODES,
 * 1 <= V <= SPEC_MAX_V.
 */
spec_status spec_tree_verify(const void *target_logits, spec_dtype target_dtype, const int32_t *parent,
                             const int32_t *token, const int32_t *keep, int n_trees, int n_nodes, int V,
                             int32_t *n_accepted_out, int32_t *path_out, int32_t *committed_out,
                             int32_t *bonus_out, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_GB300_SPEC_H */
