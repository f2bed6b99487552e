/*
 * ps.h -- C ABI of libps: scoring one prefetched subtree batch of PreSTO-style
 * Metropolis-Hastings power sampling, and walking it, on one NVIDIA GB300 GPU.
 *
 * Method: "PreSTO: Predictive Subtree Prefetching for Fast LLM Power Sampling"
 * (arXiv 2610.13171).  One prefetch round issues the feasible suffix-resampling
 * requests of a subtree in a single batched call, scores them, and follows the
 * realised accept/reject path (section 3.2, steps (2) and (3); Algorithm 2,
 * PrefetchAndScore and MHTransition).
 *
 * Vocabulary of this header
 *   position t      1..T; x_{0:c} is the prompt plus tokens 1..c, and a suffix
 *                   resampled at cut c covers positions c+1..T (eq. (5)).
 *   row             one scored position of one sequence: a row of V logits
 *                   (the next-token distribution given tokens < t) and the
 *                   token at t.
 *   segment         the rows of one sequence's scored suffix.  Segment s covers
 *                   positions seg_cut[s]+1..T in order, rows seg_row0[s] ..
 *                   seg_row0[s+1]-1.  The first segment of every chain is the
 *                   chain's current state x (its "root"); every other segment
 *                   is one feasible request (v_i, c_i) with cut c_i = seg_cut[i].
 *   src             for a request i, the segment whose proposal the state at the
 *                   decision node came from: the nearest accepted request above
 *                   the node, or the chain root.  Under Condition 1 that state
 *                   is x_{0:c_src} followed by src's rows, so the x suffix of
 *                   request i reads root rows for positions c_i+1..c_src and
 *                   then all of src's rows (c_src = T for the root).
 *   chain           one independent subtree.  Chains share nothing.
 *
 * Ownership: every pointer passed to the GPU calls is device memory owned by
 * the caller, including the workspace.  The library allocates no device
 * memory, keeps no per-call state and is safe to call from several host
 * threads on different streams, each call with its own workspace and outputs
 * (calls that share a workspace must be ordered on one stream: they use it as
 * scratch, and its counters start from zero at each call).  Calls are
 * asynchronous on the given stream (a cudaStream_t passed as void*, NULL =
 * the legacy default stream), with plain stream order: each call sees
 * everything enqueued on the stream before it, including the caller's own
 * kernels that write its inputs.  (Some kernels
 * are launched so that they may start while the previous kernel finishes;
 * they read nothing until that kernel's writes are visible, except the second
 * kernel of ps_score_walk_subtree, which reads the segment arrays, the tree
 * and the uniforms early: those were complete before that call's own first
 * kernel began.)
 *
 * Errors: the returned ps_status reports what the host can check without
 * reading device memory (sizes, null pointers, alignment, launch failures).
 * What only the device can see is reported as bits OR-ed into the caller's
 * device int32 status word (PS_DEV_*); read it after synchronising.  The
 * kernels never trap: a row or request that fails a device check gets NaN
 * outputs and the walk treats a NaN log A as a rejection.
 */
#ifndef PS_H
#define PS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PS_OK = 0,
    PS_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, bad parameter */
    PS_ERR_INFEASIBLE = 2,    /* a request violates Condition 1 (c_i > c_src) */
    PS_ERR_BAD_TREE = 3,      /* tree arrays inconsistent (child/segment ids, cycles) */
    PS_ERR_UNSUPPORTED = 4,   /* dtype, device or temperature set not supported */
    PS_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    PS_ERR_TIMEOUT = 6,       /* reserved: device waits report PS_DEV_TIMEOUT */
    PS_ERR_WORKSPACE = 7      /* workspace null, misaligned or too small */
} ps_status;

typedef enum { PS_BF16 = 0, PS_F32 = 1 } ps_dtype;

/* Device status bits (OR-ed into the caller's int32 status word). */
#define PS_DEV_BAD_TOKEN     0x01  /* a token id outside [0, V) */
#define PS_DEV_NONFINITE     0x02  /* a NaN or +inf logit (row result is NaN) */
#define PS_DEV_INFEASIBLE    0x04  /* c_i > c_src, or c_i below the root's first row */
#define PS_DEV_BAD_TREE      0x08  /* walk: bad child/segment id, or a path longer than the tree */
#define PS_DEV_BAD_LAYOUT    0x10  /* segment sizes, row ranges or src ids inconsistent */
#define PS_DEV_TIMEOUT       0x20  /* a bounded wait on a bulk copy gave up */
#define PS_DEV_BAD_ROW_INDEX 0x40  /* row_index outside [0, n_logit_rows) */
#define PS_DEV_BAD_UNIFORM   0x80  /* walk: an acceptance uniform outside (0, 1] */

/* Request codes of a tree node's `req` entry. */
#define PS_NODE_LEAF     (-1)     /* not expanded: the walk stops here */
#define PS_NODE_DEFERRED (-2)     /* its request was deferred: the walk stops here */

/*
 * Batch hints.  PS_FLAG_MASKED_LOGITS: the logits may hold many -inf entries
 * (a masked vocabulary).  Results are the same with or without it.  Without
 * it the entropy variant's fast path assumes finite logits, and a chunk with a
 * -inf input is summed again on its slow path (about 2x the time on a mostly
 * masked row).  With it the fast path clamps -inf itself, which costs
 * ordinary rows about 3%.
 */
#define PS_FLAG_MASKED_LOGITS 0x1

/*
 * One subtree batch to score (section 3.2 step (2); eq. (6)).
 *
 * logits       [n_logit_rows][ld] row-major, dtype; base 16-byte aligned and
 *              ld * element size a multiple of 16 bytes with
 *              ld * element size >= V * element size rounded up to 16.
 *              Elements V..ld-1 of a row are ignored.  -inf is a valid logit
 *              (a masked token); NaN and +inf are reported as PS_DEV_NONFINITE.
 *              A row holds at most 2^30 bytes (V <= 2^29 for bf16, 2^28 for
 *              float32); larger V returns PS_ERR_INVALID_ARG.
 * row_index    [n_rows] int64 or NULL: scored row r reads logits row
 *              row_index[r]; NULL means row r reads logits row r (then
 *              n_logit_rows >= n_rows).
 * tokens       [n_rows] int32: the token at the row's position.
 * chain_seg0   [n_chains+1] CSR offsets into segments; chain c owns segments
 *              chain_seg0[c] .. chain_seg0[c+1]-1 and the first is its root.
 * seg_row0     [n_seg+1] int64 CSR offsets into rows, seg_row0[n_seg] == n_rows,
 *              seg_row0[s+1] - seg_row0[s] == T - seg_cut[s].
 * seg_cut      [n_seg]: requests 0 <= c_i <= T-1 and c_i >= the chain root's
 *              cut; a root's cut is the position before its first row (0..T).
 * seg_src      [n_seg]: -1 for a chain root; for request i a segment of the
 *              same chain other than i (the chain root's id when the decision
 *              node holds the current state); c_i <= c_src (Condition 1).
 * alpha, tau   power exponent (finite) and proposal temperature (> 0).
 * eps          epsilon of the epsilon-certainty classes (section 3.3), in
 *              (0, 1/2); read only when ps_score_out.eps_class is requested.
 * root_lp0, root_lq  optional [n_chains][T] float64 (position t at t-1): the
 *              current state's token log-probabilities retained from the
 *              previous round (ps_carry_state).  When given, positions up to a
 *              chain root's cut take these values instead of rows, and a
 *              request's cut may lie below the root's cut; a root cut of T
 *              means the current state needs no scored rows at all.  When NULL,
 *              every request's cut must be >= its root's cut.
 */
typedef struct {
    int32_t V;
    int32_t T;
    int32_t dtype;          /* ps_dtype */
    int32_t n_chains;
    int32_t n_seg;
    int32_t flags;          /* PS_FLAG_* hints; other bits must be 0 */
    int64_t n_rows;
    int64_t ld;
    int64_t n_logit_rows;
    double alpha;
    double tau;
    double eps;
    const int32_t *chain_seg0;
    const int64_t *seg_row0;
    const int32_t *seg_cut;
    const int32_t *seg_src;
    const void *logits;
    const int64_t *row_index;
    const int32_t *tokens;
    const double *root_lp0;
    const double *root_lq;
} ps_subtree_batch;

/*
 * Outputs of ps_score_subtree (all device memory, float64).  Entries of chain
 * roots are set to NaN.
 * lp0, lq      [n_rows] optional (NULL = not returned): log p0(token) and
 *              log q_tau(token) of every row (Appendix B.1; Appendix D.3).
 * lp_y, lq_y   [n_seg] optional: log p0 / log q_tau of the proposal suffix
 *              y_{c_i+1:T} given x_{0:c_i}.
 * lp_x, lq_x   [n_seg] optional: the same for the current suffix x_{c_i+1:T}.
 * log_ratio    [n_seg] optional: r_i = (lq_x - lq_y) + alpha (lp_y - lp_x).
 * log_accept   [n_seg] required: log A_i = min{0, r_i} (eq. (6)).
 * status       device int32 word, required; the caller zeroes it.
 * entropy      [n_rows] optional: full-vocabulary entropy of p0 of every row,
 *              in nats (Appendix D.3, quantity (iii)), from the same pass.
 * eps_class    [n_seg] optional int8: 0 if A_i <= eps (epsilon-certain
 *              reject), 2 if A_i >= 1 - eps (epsilon-certain accept), 1
 *              otherwise; -1 for chain roots and NaN entries (section 3.3).
 */
typedef struct {
    double *lp0;
    double *lq;
    double *lp_y;
    double *lq_y;
    double *lp_x;
    double *lq_x;
    double *log_ratio;
    double *log_accept;
    int32_t *status;
    double *entropy;
    int8_t *eps_class;
} ps_score_out;

/*
 * Bytes of device workspace the scoring calls need for this batch (depends
 * only on n_rows and n_chains).  The workspace is scratch: per-row results
 * when lp0/lq are not requested, partial sums of rows that are split across
 * the scoring kernel's chunk ranges, their arrival counters, the counter of
 * the tail blocks that warps take at run time, and one arrival counter per
 * chain for ps_score_walk_subtree.  Returns 0 if batch is NULL.
 */
size_t ps_score_workspace_bytes(const ps_subtree_batch *batch);

/*
 * Score one subtree batch (section 3.2 step (2); eq. (6); Appendix B.1).
 *
 * For every row: log p0 and log q_tau of its token from the same logits, at
 * temperature 1 and tau, in one pass over the row.  For every request i:
 * suffix sums over its own rows (y) and over the rows of its from-state
 * x_{0:c_src} + src (x), then r_i and log A_i = min{0, r_i}.
 *
 * workspace    device memory, 256-byte aligned, >= ps_score_workspace_bytes().
 * cuda_stream  cudaStream_t or NULL.
 * Returns PS_OK once the work is enqueued; see the header comment for errors.
 */
ps_status ps_score_subtree(const ps_subtree_batch *batch, const ps_score_out *out,
                           void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * The two halves of ps_score_subtree, for callers that want per-token scores
 * only or time the halves separately.
 *
 * ps_score_rows: log p0 and log q_tau of every row's token (Appendix B.1;
 * Appendix D.3).  Reads only V, dtype, tau, n_rows, ld, n_logit_rows, logits,
 * row_index and tokens of the batch.  lp0, lq: [n_rows] device float64,
 * required.  entropy: [n_rows] device float64 or NULL (then not computed).
 * status: device int32 word, required.  workspace as for ps_score_subtree
 * (its per-row area is unused here).
 *
 * ps_assemble_subtree: suffix sums and log A of every request from per-row
 * values lp0 / lq already computed for the batch's rows (eq. (6)).  Reads the
 * segment arrays, T, alpha and n_rows of the batch; out->lp0 and out->lq are
 * ignored.
 */
ps_status ps_score_rows(const ps_subtree_batch *batch, double *lp0, double *lq, double *entropy,
                        int32_t *status, void *workspace, size_t workspace_bytes,
                        void *cuda_stream);
ps_status ps_assemble_subtree(const ps_subtree_batch *batch, const double *lp0,
                              const double *lq, const ps_score_out *out, void *cuda_stream);

/*
 * Multi-temperature row scoring (MultiTryMH, as the PreSTO pages describe it
 * in section 5.1 and Appendix D.4, Table 6(a): each candidate suffix is drawn
 * at a temperature from {0.25, 0.5, 1.0}, and the sequential sampler rescores
 * every candidate at all of them).  One pass over each row gives log p0 of the
 * row's token and log q_tau of it for every tau in taus[0..n_taus-1]:
 *     lq[k * n_rows + r] = log softmax(l_r / taus[k])[tok_r].
 * The multiple-try Metropolis update itself is not part of this library.
 *
 * taus      host array of n_taus temperatures, 1 <= n_taus <= 4, each with 1/tau
 *           exactly 1, 2, 4 or 8 (0.25, 0.5 and 1.0 qualify); anything else
 *           returns PS_ERR_UNSUPPORTED (use ps_score_rows once per tau).
 * lp0       [n_rows] device float64, required.
 * lq        [n_taus][n_rows] device float64, required.
 * entropy   [n_rows] device float64 or NULL, as for ps_score_rows.
 * The batch is read as by ps_score_rows except that batch->tau is ignored
 * (it must still be a positive finite number).  status, workspace and stream
 * as for ps_score_rows; errors and device status bits are the same.
 */
ps_status ps_score_rows_multi(const ps_subtree_batch *batch, const double *taus,
                              int32_t n_taus, double *lp0, double *lq, double *entropy,
                              int32_t *status, void *workspace, size_t workspace_bytes,
                              void *cuda_stream);

/*
 * Round carry-over (section 3.2 step (3): after the walk the sampler keeps the
 * reached state's token-level log-probabilities for the next round's
 * acceptance computations).  For every chain, the reached state
 * x_Delta = x_{0:c*} + y^{s*} (s* = state_seg, c* its cut; x itself when s* is
 * the root) gives per-position values for positions 1..T: the previous
 * round's values up to the root's cut, root rows up to c*, then the rows of
 * s*.  Optionally also eq. (21) (length-normalised log-likelihood, the mean of
 * lp0 over positions 1..T) and eq. (22) (confidence, minus the mean entropy).
 *
 * state_seg        [n_chains] int32, from ps_walk_subtree.
 * row_lp0, row_lq  [n_rows] per-row values of this batch (ps_score_rows);
 * row_entropy      [n_rows] optional.
 * prev_lp0, prev_lq, prev_entropy   [n_chains][T] the current state's values;
 *                  read only at positions up to a root's cut (may be NULL when
 *                  every root cut is 0, or equal to the batch's root_lp0/lq).
 * next_lp0, next_lq  [n_chains][T] out, required; next_entropy optional (needs
 *                  row_entropy, and prev_entropy when a root cut is > 0).
 * loglik, confidence  [n_chains] optional (confidence needs next_entropy).
 * status           device int32 word, required (PS_DEV_BAD_LAYOUT when a needed
 *                  input is missing or state_seg is not a segment of its chain;
 *                  that chain's outputs are NaN).
 */
typedef struct {
    const int32_t *state_seg;
    const double *row_lp0;
    const double *row_lq;
    const double *row_entropy;
    const double *prev_lp0;
    const double *prev_lq;
    const double *prev_entropy;
    double *next_lp0;
    double *next_lq;
    double *next_entropy;
    double *loglik;
    double *confidence;
    int32_t *status;
} ps_carry_io;

ps_status ps_carry_state(const ps_subtree_batch *batch, const ps_carry_io *io,
                         void *cuda_stream);

/*
 * ps_score_subtree_noalloc: the same scoring as ps_score_subtree, for callers
 * that cannot allocate device memory and so cannot provide a workspace.  The
 * pages have no counterpart of this entry point; it exists for embedding.
 * Examples of such callers: a sampler hook running inside another engine whose
 * device memory is owned by that engine's pool, code executing in a region
 * where a cudaMalloc would stall or is forbidden (it synchronises the device),
 * or a host program that only receives device pointers from elsewhere.
 *
 * Instead of a caller workspace it uses one static device array compiled into
 * libps (about 4.5 MB, held on every GPU that loads the library until the
 * process exits).  It never calls cudaMalloc, cudaFree or any allocating
 * routine.  Inputs and outputs are the caller's, exactly as in
 * ps_score_subtree.
 *
 * Limit: a per-row array the caller leaves NULL (out->lp0, out->lq, or both)
 * is kept in the static array instead, which holds at most 262144 rows of
 * each; a larger batch then returns PS_ERR_WORKSPACE without launching
 * anything.  Whichever of lp0 and lq the caller supplies is written, as in
 * ps_score_subtree; with both supplied there is no row limit.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.
 * Sharing: every call uses the same array, which keeps the previous call's
 * contents (the arrival counters are zeroed on the stream at each call).  Calls
 * whose work overlaps on the GPU (different streams, or different host threads,
 * without ordering between them) race on it and give wrong results; order them.
 */
ps_status ps_score_subtree_noalloc(const ps_subtree_batch *batch, const ps_score_out *out,
                                   void *cuda_stream);

/*
 * The prefetched subtree of every chain, for the walk (section 3.2 step (3)).
 * Node ids and segment ids are global (the same numbering as the batch).
 * chain_node0  [n_chains+1] CSR offsets into nodes; the first node of a chain
 *              is its root v0.
 * chain_seg0   [n_chains+1] as in ps_subtree_batch (the root segment of chain c
 *              is chain_seg0[c]).
 * acc, rej     [n_nodes] acceptance / rejection child node id, or -1.
 * req          [n_nodes] the request whose proposal the decision at the node
 *              uses (a segment id of the chain), PS_NODE_LEAF or
 *              PS_NODE_DEFERRED.
 * u            [n_seg] acceptance uniform of each request, in (0, 1]; deferred
 *              requests keep theirs for a later round, so none is consumed.
 * max_steps    K - k: at most this many transitions (>= 0).
 */
typedef struct {
    int32_t n_chains;
    int32_t n_nodes;
    int32_t n_seg;
    int32_t max_steps;
    const int32_t *chain_node0;
    const int32_t *chain_seg0;
    const int32_t *acc;
    const int32_t *rej;
    const int32_t *req;
    const double *u;
} ps_tree;

/*
 * Outputs of ps_walk_subtree (device int32 arrays, [n_chains] each).
 * state_seg    segment of the reached state: the last accepted request, or
 *              the chain root when nothing was accepted (x_Delta).
 * end_node     node where the walk stopped.
 * k_delta      transitions completed (every visited scored decision counts,
 *              accepted or rejected; Definition 1).
 * path         optional [n_chains][max_steps+1]: node ids visited, root first,
 *              then -1 padding.
 * status       device int32 word, required; the caller zeroes it.
 */
typedef struct {
    int32_t *state_seg;
    int32_t *end_node;
    int32_t *k_delta;
    int32_t *path;
    int32_t *status;
} ps_walk_out;

/*
 * Walk every chain's subtree from its root (section 3.2 step (3); Example 5;
 * Algorithm 2 MHTransition).  At a node whose request was scored, one
 * transition: move to the acceptance child if log u <= log A (u <= A,
 * the accept test of Algorithm 1), else to the rejection child.  Stop at a leaf, at a node
 * whose request was deferred, or after max_steps transitions.
 * log_accept   [n_seg] device float64, as written by ps_score_subtree.
 */
ps_status ps_walk_subtree(const ps_tree *tree, const double *log_accept,
                          const ps_walk_out *out, void *cuda_stream);

/*
 * One whole round in one call: ps_score_subtree, then ps_walk_subtree
 * (section 3.2 steps (2)-(3); Algorithm 2, PrefetchAndScore then
 * MHTransition).  Outputs are those of the two calls, bit for bit; the suffix
 * sums and the walk run in one kernel, in which the last block of each chain
 * to write its log A walks that chain, so the round takes two kernel launches
 * instead of three.
 *
 * batch, out   as for ps_score_subtree.
 * tree, wout   as for ps_walk_subtree; tree->n_chains and tree->n_seg must
 *              equal the batch's (else PS_ERR_INVALID_ARG); the walk reads
 *              out->log_accept.
 * workspace    device memory, 256-byte aligned, >= ps_score_workspace_bytes().
 * Device status bits go to out->status (scoring, suffix sums) and
 * wout->status (walk), as in the two calls.  A chain whose chain_seg0
 * bounds fail the device checks (PS_DEV_BAD_LAYOUT) is not walked: its walk
 * outputs are left unwritten.  Other layout failures give the request NaN
 * outputs, and the walk treats it as rejected.
 */
ps_status ps_score_walk_subtree(const ps_subtree_batch *batch, const ps_tree *tree,
                                const ps_score_out *out, const ps_walk_out *wout,
                                void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Full structural check of a batch and its tree in HOST memory (synchronous;
 * reads no logits).  Either argument may be NULL to skip it.  When both are
 * given, also checks that each request's src is the state of its decision
 * node.  Writes a one-line reason into msg (if msg_len > 0) on failure.
 * Returns PS_OK, PS_ERR_INVALID_ARG, PS_ERR_INFEASIBLE or PS_ERR_BAD_TREE.
 */
ps_status ps_validate_subtree(const ps_subtree_batch *batch, const ps_tree *tree,
                              char *msg, size_t msg_len);

/*
 * Host-side tree construction (synchronous; all pointers are host memory).
 *
 * ps_build_bfs_tree: BFS request collection for one chain (section 3.2 step
 * (1), Example 2).  From the root (cut T) nodes are expanded in breadth-first
 * order; expansion k uses cuts[k] (the random cut of that decision, drawn by
 * the caller: Proposition 1, (A2)).  The acceptance child gets the cut, the
 * rejection child keeps its parent's cut and state; a request is feasible when
 * its cut is <= the node's cut (Condition 1), else it is deferred (req =
 * PS_NODE_DEFERRED, deferred_cut = its cut) and its acceptance child is not
 * expanded; the rejection child is enqueued either way.  Stops at n_pf
 * feasible requests, an empty queue, or when the cuts run out.  depth_cap < 0
 * means no cap (else nodes at depth >= depth_cap are not expanded: the K - k
 * cap of Appendix C.1).
 * Outputs (capacities max_nodes >= 1 + 2 n_cuts, max_seg >= n_pf + 1): acc,
 * rej, req, node_cut, deferred_cut per node; seg_cut, seg_src per segment
 * (segment 0 is the root: its cut is the smallest request cut, or T);
 * n_nodes, n_seg, and the number of cuts used.  Returns PS_ERR_INVALID_ARG for
 * a cut outside [0, T-1] or too small a capacity.
 */
ps_status ps_build_bfs_tree(int32_t T, int32_t n_pf, int32_t depth_cap, const int32_t *cuts,
                            int32_t n_cuts, int32_t max_nodes, int32_t max_seg, int32_t *acc,
                            int32_t *rej, int32_t *req, int32_t *node_cut,
                            int32_t *deferred_cut, int32_t *seg_cut, int32_t *seg_src,
                            int32_t *n_nodes, int32_t *n_seg, int32_t *n_cuts_used);

/*
 * ps_predictive_allocation: the selection of at most `budget` candidate nodes,
 * ancestor-closed, that maximises the predicted number of completed
 * transitions (eq. (17)), by the dynamic program of eq. (19) (Proposition 2).
 * The caller gives a finite tree rooted at node 0 (acc, rej: child ids or -1),
 * which nodes are candidates (expandable with all strict ancestors expandable,
 * Appendix C.1) and each node's predicted acceptance-branch probability h_acc
 * in [0, 1] (e.g. from class probabilities by eq. (14)).  Outputs V(v0,
 * budget) and selected[v] = 1 for the chosen nodes (smallest m on ties).
 * Host memory O(n_nodes * budget).  PS_ERR_BAD_TREE for an inconsistent tree.
 */
ps_status ps_predictive_allocation(int32_t n_nodes, const int32_t *acc, const int32_t *rej,
                                   const uint8_t *candidate, const double *h_acc,
                                   int32_t budget, double *value, uint8_t *selected);

/* eq. (14): h(v+) = (1 + P(certain accept) - P(certain reject)) / 2 (Lemma 3). */
double ps_midpoint_branch_probability(double p_accept, double p_reject);

/*
 * Diagnostic with no counterpart in the PreSTO pages: checks on the device the
 * bounded wait that every bulk-copy wait of the scoring kernel uses.  One warp
 * waits on a shared-memory mbarrier that nothing completes; after limit_ns of
 * wall time (or a fixed poll count) the wait gives up and PS_DEV_TIMEOUT is
 * OR-ed into *status, and the kernel returns, leaving the context usable.
 * This lets a caller or a test see the timeout path work without faulting or
 * hanging the GPU.
 *
 * limit_ns  1,000 .. 2,000,000,000 (1 us .. 2 s), else PS_ERR_INVALID_ARG.
 * status    device int32 word, required.
 */
ps_status ps_selftest_wait_timeout(uint64_t limit_ns, int32_t *status, void *cuda_stream);

/*
 * Diagnostic with no counterpart in the PreSTO pages: reads `bytes` of device
 * memory at `data` once, with 16-byte streaming loads spread over every SM,
 * and folds the words into *sink with XOR.  Timing it gives the plain read
 * rate of the device, to which the scoring kernel's rate can be compared.
 *
 * data    device memory, 16-byte aligned.
 * bytes   a multiple of 16 (else PS_ERR_INVALID_ARG); 0 launches nothing.
 * sink    device uint32 word; its value is meaningless beyond keeping the
 *         loads.
 */
ps_status ps_selftest_read(const void *data, size_t bytes, uint32_t *sink, void *cuda_stream);

/* Static text for a status code. */
const char *ps_status_string(ps_status status);

/* Library version string. */
const char *ps_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PS_H */
