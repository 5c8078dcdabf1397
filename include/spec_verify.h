/*
 * spec_verify.h -- C ABI of the GB300 speculative-decoding verify library (libspec_verify.so).
 *
 * The operation. Speculative decoding lets a cheap draft model propose gamma tokens and has the
 * large target model score all of them in one parallel pass; a rejection-sampling test on the
 * target's own probabilities accepts the longest passing prefix and a distribution-preserving
 * correction makes every emitted token an exact sample of the target ("Fast Inference from
 * Transformers via Speculative Decoding", Leviathan, Kalman, Matias; pith.science review,
 * sections "The pith", "Core claim", "What carries the argument", "Desk Editor's Note",
 * "Circularity Check"). Falcon verifies a tree of drafts in one pass under greedy decoding
 * ("Falcon: Faster and Parallel Inference of Large Language Models through Enhanced
 * Semi-Autoregressive Drafting and Custom-Designed Decoding Tree", pith.science review,
 * "What carries the argument", Figure 3, Figure 4). This library is that verify step and
 * nothing else: the draft and target models are the caller's.
 *
 * Common rules for every entry point
 *   - All pointers except `stream` and `workspace`'s host-side size are DEVICE pointers on the
 *     current CUDA device. The caller owns every buffer; the library allocates nothing, frees
 *     nothing and keeps no state except cached device attributes.
 *   - Logits are row-major, contiguous, fp32 (SPEC_F32) or bf16 (SPEC_BF16) whose base address
 *     is aligned to the element size. Rows need not be 16-byte aligned (an unaligned row is read
 *     with scalar loads at its ends).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are stream-ordered and
 *     asynchronous: they enqueue work and return; nothing synchronises with the host.
 *   - Return value: SPEC_OK, or a negative SPEC_ERR_* code found on the host before anything
 *     was enqueued (SPEC_ERR_LAUNCH: the launch itself failed, cudaGetLastError).
 *   - Device-side problems found in the data (a non-finite logit row, a token outside [0, V),
 *     a bad tree parent) never trap: the affected batch row reports accept_len = -1 with all
 *     its output tokens -1, and *status receives the first such code (atomic compare-and-swap
 *     from 0). *status is never cleared by the library: zero it before a call whose errors you
 *     want to see.
 *   - A logits row is valid when it holds no NaN and no +inf and at least one finite value;
 *     -inf entries (masked tokens) are allowed and get probability 0.
 *   - Workspace: a caller-owned device buffer of at least spec_workspace_bytes(...) bytes,
 *     16-byte aligned. It is scratch: every call overwrites the parts it uses before reading
 *     them, so it needs no initialisation and holds nothing between calls. Calls on one
 *     stream may share a workspace; two calls that may run at the same time need two.
 *   - Results are deterministic: the same inputs give bit-identical outputs on the same GPU.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* host-side return codes */
#define SPEC_OK 0
#define SPEC_ERR_NULL (-1)      /* a required pointer is NULL                                */
#define SPEC_ERR_SHAPE (-2)     /* B, gamma, N, V or rows out of range (see limits below)     */
#define SPEC_ERR_TEMP (-3)      /* temperature not 0 and not in [FLT_MIN, FLT_MAX]             */
#define SPEC_ERR_DTYPE (-4)     /* dtype not SPEC_F32 / SPEC_BF16                             */
#define SPEC_ERR_WORKSPACE (-5) /* workspace smaller than spec_workspace_bytes(...)            */
#define SPEC_ERR_ALIGN (-6)     /* a pointer is not aligned to its element size (16 for the
                                   workspace)                                                */
#define SPEC_ERR_LAUNCH (-7)    /* the kernel launch failed (e.g. no sm_103a device)          */
/* device-side codes, written to *status */
#define SPEC_ERR_NONFINITE (-20) /* a logits row has NaN or +inf, or no finite entry          */
#define SPEC_ERR_TOKEN (-21)     /* a draft / node token is outside [0, V)                    */
#define SPEC_ERR_PARENT (-22)    /* parents[b,0] != -1 or parents[b,i] not in [0, i)          */
#define SPEC_ERR_TIMEOUT (-23)   /* a bounded wait inside a kernel gave up (an on-chip copy or
                                    tensor-core result did not arrive within 2 s)             */
#define SPEC_ERR_CHECK (-24)     /* checked build only (libspec_verify_checked.so): an index the
                                    kernels computed fell outside its buffer; the access was
                                    skipped. Never seen from a correct library.               */

/* limits */
#define SPEC_MAX_V (1 << 20)   /* vocabulary size                                            */
#define SPEC_LMHEAD_MAX_V (1 << 19)   /* vocabulary size of spec_verify_chain_lmhead          */
#define SPEC_MAX_GAMMA 255     /* draft length of the chain                                  */
#define SPEC_MAX_NODES 1024    /* nodes per candidate tree                                   */

/*
 * Bytes of workspace needed by a call over B batch rows of `rows_per_b` logits rows of V
 * elements: rows_per_b = 2*gamma+1 for spec_verify_chain (any temperature), N for
 * spec_verify_tree, 2*N for spec_verify_tree_sample at T > 0, 1 for spec_probs and spec_sample
 * (with B = rows), k for spec_topk (with B = rows). Returns 0 for invalid arguments.
 */
size_t spec_workspace_bytes(int B, int rows_per_b, int V, int dtype);

/* Zero-fills a workspace on `stream` (a cudaMemsetAsync). Optional: no call requires it. */
int spec_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Chain verification (rejection sampling), batched over B independent steps.
 *
 *   p_i = softmax(target_logits[b, i, :] / T)   for i = 0..gamma
 *   q_i = softmax(draft_logits[b, i, :] / T)    for i = 0..gamma-1
 *   x_i = draft_tokens[b, i]; draft x_i is accepted while u_i <= p_i(x_i) / q_i(x_i)
 *         (u_i = uniforms[b, i]); q_i(x_i) = 0 counts as +inf if p_i(x_i) > 0, else as 0.
 *   n   = index of the first rejection, or gamma if all pass.
 *   The emitted token at position n is drawn with u = uniforms[b, gamma] by inverse CDF
 *   (the first k whose running sum strictly exceeds u * S) from
 *     r = max(0, p_n - q_n)   if n < gamma (r = p_n if that sums to 0), or
 *     r = p_gamma             if n == gamma (the bonus token).
 *   T == 0 is greedy decoding: x_i is accepted iff it is the lowest-index argmax of target
 *   row i, and the emitted token is the argmax of target row n; draft_logits is not read
 *   (may be NULL) and neither is uniforms (may be NULL).
 *
 *   target_logits [B, gamma+1, V]   dtype
 *   draft_logits  [B, gamma, V]     dtype (unused at T == 0)
 *   draft_tokens  [B, gamma]        int32 (may be NULL when gamma == 0)
 *   uniforms      [B, gamma+1]      fp32 in (0, 1) (unused at T == 0)
 *   accept_len    [B]               int32 out: n, or -1 for an invalid batch row
 *   out_tokens    [B, gamma+1]      int32 out: x_0..x_{n-1}, the drawn token, then -1
 *   status        [1]               int32 device word, see the common rules
 * Limits: 1 <= V <= SPEC_MAX_V, 0 <= gamma <= SPEC_MAX_GAMMA, B >= 0 (B == 0 does nothing),
 * temperature == 0 or FLT_MIN <= temperature <= FLT_MAX.
 */
int spec_verify_chain(const void *target_logits, const void *draft_logits, int dtype,
                      const int32_t *draft_tokens, const float *uniforms, int B, int gamma, int V,
                      float temperature, int32_t *accept_len, int32_t *out_tokens,
                      int32_t *status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Greedy tree verification, batched over B candidate trees of N nodes.
 *
 *   g_j = lowest-index argmax of target_logits[b, j, :]
 *   node 0 is the committed root and is accepted; node i > 0 is accepted iff its parent is
 *   accepted and node_tokens[b, i] == g_{parents[b, i]}.
 *   d* = the deepest accepted node (the smallest index among equally deep ones).
 *
 *   target_logits [B, N, V]   dtype
 *   parents       [B, N]      int32, parents[b, 0] = -1, 0 <= parents[b, i] < i
 *   node_tokens   [B, N]      int32 (node 0's entry is not read)
 *   accept_len    [B]         int32 out: depth of d* (accepted draft tokens), or -1
 *   path_nodes    [B, N]      int32 out: root .. d* (depth+1 entries), then -1
 *   out_tokens    [B, N]      int32 out: tokens of path nodes 1..depth, then g_{d*} (the bonus
 *                             token), then -1
 * Limits: 1 <= N <= SPEC_MAX_NODES, 1 <= V <= SPEC_MAX_V, B >= 0.
 */
int spec_verify_tree(const void *target_logits, int dtype, const int32_t *parents,
                     const int32_t *node_tokens, int B, int N, int V, int32_t *accept_len,
                     int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Chain verification (T > 0) fused with its logit producer: the target's and the drafter's LM
 * heads evaluated on the 5th-generation tensor cores, logits = hidden states x head^T (bf16
 * inputs, fp32 accumulation, logits stored as bf16), with the softmax reduction that verification
 * starts with computed from the accumulators in the GEMM's epilogue, so that no pass reads the
 * logits back for it. The target scores every drafted position in one parallel pass ("Fast
 * Inference from Transformers via Speculative Decoding", pith.science review, "The pith"); this
 * is that pass's last layer with verification's first step fused in. The verification itself is
 * spec_verify_chain's, on the stored logits:
 *   logits_t[b*(gamma+1) + i, :] = bf16(hidden_t[b*(gamma+1) + i, :] . head_t^T)  (i = 0 .. gamma)
 *   logits_d[b*gamma + i, :]     = bf16(hidden_d[b*gamma + i, :] . head_d^T)      (i < gamma)
 * (dot products accumulated in fp32, rounded to nearest-even bf16)
 * then accept_len / out_tokens exactly as spec_verify_chain(logits_t, logits_d, ...) defines them.
 *
 *   hidden_t  [B*(gamma+1), Ht] bf16       hidden_d [B*gamma, Hd] bf16 (the positions' final
 *                                          hidden states, row-major; Ht = hidden_t_size, Hd =
 *                                          hidden_d_size: the drafter may be a smaller model)
 *   head_t [V, Ht] bf16, head_d [V, Hd]    the two LM heads (row-major: one row per token)
 *   logits_t  [B*(gamma+1), V] bf16 out    logits_d [B*gamma, V] bf16 out (also read back by
 *                                          the draw)
 *   draft_tokens, uniforms, accept_len, out_tokens, status: as for spec_verify_chain
 *   workspace  at least spec_lmhead_workspace_bytes(B, gamma, V) bytes (scratch)
 * Limits: 1 <= gamma <= SPEC_MAX_GAMMA, V a multiple of 256 in [256, SPEC_LMHEAD_MAX_V], Ht and Hd
 * positive multiples of 64, temperature in [FLT_MIN, FLT_MAX] (the greedy case is not offered here: use
 * spec_verify_chain at T = 0 on the logits); every matrix 16-byte aligned. A non-finite hidden
 * state or head row makes its logits rows non-finite: the batch row reports -1. A wait inside
 * the GEMM that gives up (after 2 s) sets *status to SPEC_ERR_TIMEOUT.
 */
size_t spec_lmhead_workspace_bytes(int B, int gamma, int V);
int spec_verify_chain_lmhead(const void *hidden_t, const void *head_t, int hidden_t_size,
                             const void *hidden_d, const void *head_d, int hidden_d_size,
                             const int32_t *draft_tokens,
                             const float *uniforms, int B, int gamma, int V, float temperature,
                             void *logits_t, void *logits_d, int32_t *accept_len,
                             int32_t *out_tokens, int32_t *status, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * Stochastic (T > 0) tree verification, batched over B candidate trees of N nodes: the walk of
 * each tree by sequential per-sibling rejection sampling. The pages verify Falcon's tree only
 * greedily ("Falcon: ...", pith.science review, Figure 4, "greedy (temperature=0)"); for sampling
 * this library applies chain verification's rule ("Fast Inference from Transformers via
 * Speculative Decoding", pith.science review, "The pith", "Desk Editor's Note": accept while
 * u <= p/q, correct a rejection from norm(max(0, p - q))) to the siblings of a node in turn:
 *
 *   p_j = softmax(target_logits[b, j, :] / T), q_j = softmax(draft_logits[b, j, :] / T)
 *   (q_j: the distribution node j's children were drafted from). From the root: r = p_cur; for
 *   each child c of the current node, in increasing index, with x = node_tokens[b, c]:
 *   accepted if uniforms[b, c] <= r(x) / q_cur(x) (q(x) = 0: +inf if r(x) > 0, else 0), and the
 *   walk moves to c; else r = norm(max(0, r - q_cur)) (unchanged if that sums to 0). When every
 *   child is rejected, or the node has none, the last token is drawn from r with
 *   u = uniforms[b, 0] (inverse CDF: the first k whose running sum strictly exceeds u * S).
 *   When every node's children were drafted independently from q at that node, each emitted
 *   token is an exact sample of the target given the tokens before it.
 *
 *   target_logits, draft_logits [B, N, V]  dtype
 *   parents, node_tokens       [B, N]      int32, as for spec_verify_tree
 *   uniforms                   [B, N]      fp32 in (0, 1): [b, 0] the final draw, [b, i] node
 *                                          i's acceptance test (i >= 1)
 *   accept_len, path_nodes, out_tokens     as for spec_verify_tree: the accepted nodes' depth,
 *                                          root .. last accepted node, their tokens then the
 *                                          drawn token, then -1
 *   workspace  at least spec_workspace_bytes(B, 2 * N, V, dtype) bytes (scratch)
 * T == 0 is spec_verify_tree (greedy; draft_logits and uniforms are not read, may be NULL; a
 * workspace of spec_workspace_bytes(B, N, V, dtype) suffices). A node with many rejected
 * children costs one pass over its two rows per rejection. Invalid trees (a bad parent, a
 * token outside [0, V), a non-finite target or draft row) report accept_len = -1, all -1, and
 * *status.
 * Limits: 1 <= N <= SPEC_MAX_NODES, 1 <= V <= SPEC_MAX_V, B >= 0, temperature as for
 * spec_verify_chain.
 */
int spec_verify_tree_sample(const void *target_logits, const void *draft_logits, int dtype,
                            const int32_t *parents, const int32_t *node_tokens,
                            const float *uniforms, int B, int N, int V, float temperature,
                            int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens,
                            int32_t *status, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Temperature softmax of `rows` logits rows into fp32 probabilities: the target and draft
 * distributions p and q that the verification step compares ("Fast Inference from Transformers
 * via Speculative Decoding", pith.science review, "The pith" and "What carries the argument":
 * the step works on the target's own output distribution; at temperature 0 the distribution is
 * the greedy one-hot, as in Falcon's Figure 4):
 *   out_probs[r, k] = exp((l[r,k] - max_k l[r,k]) / T) / sum_j exp((l[r,j] - max l[r]) / T)
 * T == 0 gives the one-hot vector at the lowest-index argmax. An invalid row is written as NaN
 * and reported through *status (SPEC_ERR_NONFINITE). Besides the logits, T and the output, the
 * call takes a status word (so that invalid rows are reported as in the verify calls) and a
 * workspace (rows too long to be held on chip take the stream kernel, whose unit partials live
 * there).
 *
 *   logits    [rows, V]   dtype
 *   out_probs [rows, V]   fp32 out (4-byte aligned)
 * Limits: 1 <= V <= SPEC_MAX_V, rows >= 0, temperature as for spec_verify_chain.
 */
int spec_probs(const void *logits, int dtype, int rows, int V, float temperature,
               float *out_probs, int32_t *status, void *workspace, size_t workspace_bytes,
               void *stream);

/*
 * Drafter-side sampling, the step before verification: each row's token drawn from
 * softmax(logits[r, :] / T) by inverse CDF with uniform u = uniforms[r] (the first k whose running
 * sum strictly exceeds u * S), exactly as spec_verify_chain draws its bonus token; T == 0 gives
 * the lowest-index argmax (uniforms not read, may be NULL). An invalid row gets token -1 and sets
 * *status (SPEC_ERR_NONFINITE).
 *   logits     [rows, V]   dtype
 *   uniforms   [rows]      fp32 in (0, 1)
 *   out_tokens [rows]      int32 out
 *   workspace  at least spec_workspace_bytes(rows, 1, V, dtype) bytes (scratch)
 * Limits: 1 <= V <= SPEC_MAX_V, rows >= 0, temperature as for spec_verify_chain.
 */
int spec_sample(const void *logits, int dtype, int rows, int V, float temperature,
                const float *uniforms, int32_t *out_tokens, int32_t *status, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Top-n candidates per row, for expanding a draft tree with the drafter's most likely tokens at
 * each node (Falcon, pith.science review, "What carries the argument"): out_idx[r, 0..k) = the
 * indices of the k largest logits of row r, largest first, equal values by increasing index.
 * An invalid row (NaN, +inf, or no finite value) gets -1 everywhere and sets *status
 * (SPEC_ERR_NONFINITE).
 *   logits    [rows, V]  dtype
 *   out_idx   [rows, k]  int32 out
 *   workspace at least spec_workspace_bytes(rows, k, V, dtype) bytes (scratch)
 * Limits: 1 <= k <= min(V, SPEC_MAX_TOPK), 1 <= V <= SPEC_MAX_V, rows >= 0.
 */
#define SPEC_MAX_TOPK 16
int spec_topk(const void *logits, int dtype, int rows, int V, int k, int32_t *out_idx,
              int32_t *status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Tree-attention mask of B candidate trees (Falcon review, Figure 3, "SAR decoding tree
 * attention": every node attends to itself and its ancestors): with W = ceil(N / 32), bit j % 32
 * of mask_words[b, i, j / 32] is set iff node j is node i or an ancestor of node i. Parents as
 * for spec_verify_tree; an invalid tree gets an all-zero mask and sets *status
 * (SPEC_ERR_PARENT). No workspace.
 *   parents    [B, N]     int32
 *   mask_words [B, N, W]  uint32 out
 * Limits: 1 <= N <= SPEC_MAX_NODES, B >= 0.
 */
int spec_tree_mask(const int32_t *parents, int B, int N, uint32_t *mask_words, int32_t *status,
                   void *stream);

/* Static text for any SPEC_* code ("unknown status" otherwise). */
const char *spec_status_string(int code);

/*
 * The CUDA runtime error (a cudaError_t value) behind the most recent SPEC_ERR_LAUNCH that a call
 * of this library returned on the calling thread, 0 if there was none; and its text. Lets a
 * caller tell a missing device, a launch the device cannot fit and an earlier sticky fault
 * apart. Thread-local; never reset by a successful call.
 */
int spec_last_cuda_error(void);
const char *spec_cuda_error_string(int cuda_error);

/*
 * Self-check of the bounded waits (not an operation of the method). The LM-head GEMM's roles
 * wait on shared-memory barriers (copy completion, MMA completion, the other CTA's epilogue);
 * each wait gives up after a limit (2 s in the kernels), writes SPEC_ERR_TIMEOUT to *status and
 * lets the kernel finish, so that a lost arrival ends the call with an error instead of hanging
 * the GPU. This call launches one cluster of two CTAs that waits, through the same wait
 * routines, on barriers nothing ever arrives on, with the given limit: a CTA-scope wait in each
 * CTA and a cluster-scope wait in the even one.
 *   status         [1] int32 device word; receives SPEC_ERR_TIMEOUT when the waits give up (the
 *                  caller zeroes it first; the first nonzero code written is kept)
 *   limit_seconds  how long each wait tries, 1e-6 .. 10
 * Returns SPEC_OK once enqueued (the kernel then runs for about two limits), or
 * SPEC_ERR_NULL / ALIGN / SHAPE (limit out of range) / LAUNCH.
 */
int spec_selftest_bounded_wait(int32_t *status, double limit_seconds, void *stream);

/*
 * The kernel launches a call of the given shape makes on the current device; it enqueues
 * nothing and touches no memory (for tests and profiling; the pages have no counterpart).
 *   kind        SPEC_CALL_CHAIN (rows_per_b = 2*gamma+1, any temperature), SPEC_CALL_TREE
 *               (rows_per_b = N) or SPEC_CALL_PROBS (B = rows, rows_per_b = 1)
 *   kernels[0]  kernel launches per call: 1 when one kernel holds every row in registers
 *               (spec_probs with rows of at most 8 x 64 KB of logits), else 2 (a stream kernel
 *               over every row, then the finishing kernel, launched as its programmatic
 *               dependent)
 *   grid[0]     CTAs of the launch that finishes the call
 *   cluster[0]  its thread-block cluster size (1 = no cluster)
 * Returns SPEC_OK or SPEC_ERR_NULL / SHAPE / DTYPE / TEMP. The shape depends on the device's
 * multiprocessor count.
 */
#define SPEC_CALL_CHAIN 0
#define SPEC_CALL_TREE 1
#define SPEC_CALL_PROBS 2
int spec_launch_shape(int kind, int B, int rows_per_b, int V, int dtype, float temperature,
                      int *kernels, int *grid, int *cluster);

/*
 * spec_verify_chain without a workspace argument; the pages have no counterpart. It is for
 * callers that cannot hand the library device memory of their own: a process whose device
 * memory is all owned by another framework's caching allocator, or a per-step decode path that
 * must not allocate (an allocation can synchronise the device and fragments memory over a long
 * run). The scratch is instead a file-scope device array of SPEC_STATIC_SCRATCH_BYTES inside the
 * library, one per device, reserved when the library's device code is loaded; the call itself
 * allocates and frees nothing.
 *   - Nothing in the array needs to start at any particular value.
 *   - A call whose spec_workspace_bytes(B, 2*gamma+1, V, dtype) exceeds the array returns
 *     SPEC_ERR_WORKSPACE before anything is enqueued.
 *   - The array's device address is looked up (cudaGetSymbolAddress) on the first call made on
 *     each device, with that device current, and cached (for device ordinals below 64; a
 *     device with a higher ordinal repeats the lookup on every call); make that first call
 *     before any stream capture begins. SPEC_ERR_LAUNCH here means that the lookup failed
 *     (no usable device).
 *   - Every call on a device shares the one array: two calls that may run at the same time (on
 *     different streams, or from different host threads without ordering) race on it and give
 *     undefined results. Calls ordered on one stream are fine.
 * Arguments, results and every other rule are those of spec_verify_chain.
 */
#define SPEC_STATIC_SCRATCH_BYTES (4u << 20)
int spec_verify_chain_static(const void *target_logits, const void *draft_logits, int dtype,
                             const int32_t *draft_tokens, const float *uniforms, int B, int gamma,
                             int V, float temperature, int32_t *accept_len, int32_t *out_tokens,
                             int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
