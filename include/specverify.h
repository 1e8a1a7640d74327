/*
 * specverify.h — C ABI of libspecverify: batched speculative-decoding verification on one GPU.
 *
 * The library implements the verification step of speculative decoding over the vocabulary,
 * plus the draft-side pieces of the SSD / Saguaro method and a Mirror-SD style branch check:
 *
 *   sv_verify          accept draft token s_i with probability min(1, q_i(s_i)/p_i(s_i)), stop at
 *                      the first rejection, then draw the bonus token from (q - p)_+ / sum (q - p)_+
 *                      at that position, or from q_{K+1} when all K are accepted.
 *                      ["Speculative Speculative Decoding" notes, §2.2 steps ①-④;
 *                       "Accelerating LLM Decoding with Speculative Sampling (2023)" notes, §1, §3]
 *   sv_saguaro_sample  draft sampling under sigma_{F,C}: the top-F draft probabilities are
 *                      multiplied by C and the row is renormalised.
 *                      [SSD notes §4.4, Theorems 15 and 19; SSD abstract page, "Method"]
 *   sv_fanout          Theorem 12 geometric fan-out F_k.            [SSD abstract page, "Method"]
 *   sv_cache_keys      top-F_k draft tokens per depth, excluding the proposed token.
 *                                                                    [SSD notes §5.1]
 *   sv_cache_lookup    hit iff the verification outcome (k, t*) is a key.
 *                                                                    [SSD abstract page, "Method"]
 *   sv_topk_rows       top-kappa ids and log-probabilities of logit rows (early-exit roots).
 *                                                                    [Mirror-SD notes §3.1]
 *   sv_mirror_reuse    does the committed prefix (accepted..., correction) match a branch?
 *                                                                    [Mirror-SD notes §3.2]
 *
 * Notation: q is the target distribution, p the draft distribution (SpS notes §1).  B sequences,
 * K draft tokens per sequence, vocabulary V.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Logits are row-major: row r of a logit tensor starts at element r * row_pitch of the base
 *    pointer (row_pitch >= V, in elements).  For per-sequence tensors, row (b, j) is row
 *    b * rows_per_seq + j.  dtype SV_F32 (IEEE float) or SV_BF16 (bfloat16 bit patterns).
 *    Rows are moved with 16-byte bulk copies, so base pointers must be 16-byte aligned and
 *    row_pitch * elem_size a multiple of 16 (else SV_ERR_INVALID_ARG); V itself is free.
 *  - Pointers marked "dev" are device memory the caller owns; "host" are host memory.  The
 *    library allocates nothing: calls that need scratch take a caller-owned device workspace
 *    whose size comes from the matching *_workspace_size() function.  A workspace may be reused
 *    by consecutive calls on one stream; concurrent calls need distinct workspaces.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *    Every call works on the current device (cudaGetDevice): the stream and the device arrays
 *    it names (the logits; for the integer calls their outputs) must belong to it, else the
 *    call returns SV_ERR_INVALID_ARG after the size and workspace checks, before any launch.
 *    The check is skipped while `stream` is being captured into a CUDA graph.
 *    Argument errors are returned synchronously, before anything is launched.  Conditions only
 *    the GPU can see (non-finite logits, out-of-range tokens, a wait that timed out) are written
 *    to the optional device-side sv_stats block, which the caller reads after synchronising.
 *  - Ranking ties (argmax, top-F, top-kappa, nucleus order) go to the lowest token id.
 *  - Temperature 0 marks a greedy sequence: q and p are one-hot at the first argmax.
 *  - Randomness is an input: uniforms are doubles in [0, 1).  An accept test accepts iff
 *    u < min(1, q/p).  A draw with weights w returns the smallest id v with
 *    w_0 + ... + w_v > u * (w_0 + ... + w_{V-1}) (token-id order).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *sv_stream_t;

typedef enum sv_status {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,  /* bad size, null pointer, misaligned base, unsupported value */
    SV_ERR_CUDA = 2,         /* a CUDA runtime call failed (launch, memset, device query) */
    SV_ERR_NONFINITE = 3,    /* device: a row holds NaN, or its maximum is not finite */
    SV_ERR_TIMEOUT = 4,      /* device: a bounded wait on a shared-memory copy gave up */
    SV_ERR_WORKSPACE = 5,    /* workspace pointer null/misaligned or smaller than required */
    SV_ERR_BAD_TOKEN = 6     /* device: a token id outside [0, V) */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/*
 * Device-written status and counters.  Each call that takes a stats pointer overwrites the
 * block (it is cleared on the call's stream before any kernel of the call writes to it).  status holds the first
 * device-detected error and error_index the row (or sequence) it concerns, -1 if none.
 *
 * Decisions (accept tests and draws) are first taken in float32 with a proven error bound.
 * Those the bound cannot settle are recomputed in a float-float tier (about 44 significant
 * bits) and counted in `reresolved`; those within 2e-11 relative of the boundary even there
 * are counted in `unresolved`.  `near_boundary` counts decisions whose uniform lies within
 * 1e-6 of a ratio or a normalised CDF boundary (a property of the data, reported for context).
 */
typedef struct sv_stats {
    int32_t status;
    int32_t error_index;
    int64_t rows;           /* logit rows streamed by the statistics pass */
    int64_t accept_tests;   /* ratio tests performed (sampled sequences) */
    int64_t draws;          /* inverse-CDF draws (residual, bonus or draft) */
    int64_t reresolved;
    int64_t near_boundary;
    int64_t unresolved;
} sv_stats;

/* Per-position debug values written by sv_verify when `debug` is not NULL:
 * debug[(b * (K + 1) + j) * SV_DEBUG_FIELDS + field], float64, NaN where undefined.
 *   LSE_Q    log sum_v exp(x_v / T) of target row j (j = 0..K)
 *   LSE_P    the same for draft row j (j < K)
 *   Q_S, P_S q_j(s_j) and p_j(s_j) after temperature, top-k, top-p and sigma_{F,C} (j < K)
 *   RATIO    q_j(s_j) / p_j(s_j), unclipped (j < K)
 *   MASS_Q   mass of target row j that the top-k / top-p filters keep (1 without filters)
 *   MASS_P   the same for draft row j
 *   R        (j == 0 only) sum of the weights of the residual / bonus draw   */
#define SV_DEBUG_FIELDS 8
enum {
    SV_DBG_LSE_Q = 0, SV_DBG_LSE_P = 1, SV_DBG_Q_S = 2, SV_DBG_P_S = 3,
    SV_DBG_RATIO = 4, SV_DBG_MASS_Q = 5, SV_DBG_MASS_P = 6, SV_DBG_R = 7
};

/* Largest K accepted by sv_verify / sv_cache_keys (draft tokens per sequence). */
#define SV_MAX_K 32

/* Most drafted nodes in one tree of sv_tree_verify. */
#define SV_MAX_TREE 128

/* Library utilities (no counterpart on the pages): the text of a status code (a static string,
 * never freed), and the version as major * 10000 + minor * 100 + patch. */
const char *sv_status_string(sv_status s);
int sv_version(void);

/* ----------------------------------------------------------------------------------------
 * sv_verify — modified rejection sampling over the vocabulary for B sequences.
 * [SSD notes §2.2; SpS notes §3 (rule, mass identities), §6 (filters act before the ratio);
 *  Mirror-SD notes §2 step 3 (greedy: longest prefix equal to the target argmax)]
 *
 *  target_logits  dev, rows (b, j) for j = 0..K at b*(K+1)+j, pitch t_row_pitch: the target
 *                 scores for positions 1..K+1.
 *  draft_logits   dev, rows (b, j) at b*d_rows_per_seq+j (d_rows_per_seq >= K), pitch
 *                 d_row_pitch; rows j < K are the draft distributions that proposed s_1..s_K.
 *                 Never read for greedy sequences.
 *  draft_tokens   dev int32 [B][K], each in [0, V) (else SV_ERR_BAD_TOKEN in stats).
 *  uniforms       dev float64 [B][K+1]: u[b][i] (i < K) the accept test of position i+1,
 *                 u[b][K] the residual / bonus draw.  Greedy sequences consume none.
 *  temperature    dev float [B]: T in [1e-3, 1e3] sampled, T == 0 greedy (anything else is
 *                 reported in stats as SV_ERR_INVALID_ARG).  Applied to both q and p.
 *  top_p          dev float [B] or NULL (no nucleus filter).  top_p >= 1 disables the filter
 *                 for that sequence; otherwise the shortest prefix of tokens in (probability
 *                 desc, id asc) order whose mass reaches top_p is kept, on q and on p.
 *  top_k          dev int32 [B] or NULL (no top-k filter).  k <= 0 or k >= V disables the
 *                 filter for that sequence; otherwise the first k tokens in (probability desc,
 *                 id asc) order are kept, on q and on p.  With both filters on, top-k acts
 *                 first and the nucleus is that of the renormalised top-k distribution (the
 *                 pages fix no order between the two; this is the common sampler order).
 *  saguaro_F, saguaro_C  the draft-side sigma_{F,C} transform applied to every draft row
 *                 before the ratio and the residual (F = 0 or C = 1: none; 0 <= C <= 1).
 *  accept_len     dev int32 [B]: k, the number of accepted draft tokens (0..K).
 *  out_tokens     dev int32 [B][K+1]: s_1..s_k, then t*, then -1 padding.
 *  debug          dev float64 [B][K+1][SV_DEBUG_FIELDS] or NULL.
 *  stats          dev sv_stats or NULL.
 *  workspace      dev, >= sv_verify_workspace_size(B, K, V) bytes, 256-byte aligned.
 * Returns SV_ERR_INVALID_ARG for B < 1, K < 0, K > SV_MAX_K, V < 1, a pitch < V, a null
 * required pointer, d_rows_per_seq < K, F < 0, C outside [0, 1] or a misaligned base.
 * -------------------------------------------------------------------------------------- */
size_t sv_verify_workspace_size(int B, int K, int V);

sv_status sv_verify(const void *target_logits, int64_t t_row_pitch,
                    const void *draft_logits, int64_t d_row_pitch, int d_rows_per_seq,
                    sv_dtype dtype,
                    const int32_t *draft_tokens, const double *uniforms,
                    int B, int K, int V,
                    const float *temperature, const float *top_p, const int32_t *top_k,
                    int saguaro_F, float saguaro_C,
                    int32_t *accept_len, int32_t *out_tokens,
                    double *debug, sv_stats *stats,
                    void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_verify_host — sv_verify on inputs in host memory, outputs to host memory.
 * [the same rule as sv_verify; the transfer is part of the call]
 *
 * The arguments mean what sv_verify's do, with these pointers in HOST memory (pinned memory,
 * e.g. from cudaHostAlloc, makes the copies asynchronous and full-speed; pageable memory
 * works through the driver's staging):
 *   target_logits, draft_logits, draft_tokens, uniforms, temperature, top_p (or NULL),
 *   top_k (or NULL), accept_len (written), out_tokens (written).
 * stats and workspace stay in device memory; debug output is not offered.
 *
 * Copies: the call enqueues host-to-device copies, then the verification, then the
 * device-to-host copies of accept_len and out_tokens, all on `stream`.
 * - Inputs copied: every target row, and the draft rows j < K of each sequence with a nonzero
 *   temperature (a greedy sequence's draft rows are never read, so they are not copied), plus
 *   the tokens, uniforms, temperatures and filters.  The host reads the temperatures itself
 *   to choose the rows.
 * - Staging: the inputs land in device buffers carved from the workspace (rows padded to 16
 *   bytes).  Copies are pitched, one per run of consecutive rows.
 * - Completion: the host outputs are valid, and the host inputs may change, once the stream
 *   has synchronised.
 * - h2d_bytes: (host, may be NULL) receives the bytes copied to the device.
 *
 *  workspace  dev, >= sv_verify_host_workspace_size(B, K, V, dtype) bytes, 256-byte aligned.
 * Returns sv_verify's argument errors, SV_ERR_WORKSPACE for a short workspace, SV_ERR_CUDA if
 * a copy cannot be enqueued.
 * -------------------------------------------------------------------------------------- */
size_t sv_verify_host_workspace_size(int B, int K, int V, sv_dtype dtype);

sv_status sv_verify_host(const void *target_logits, int64_t t_row_pitch,
                         const void *draft_logits, int64_t d_row_pitch, int d_rows_per_seq,
                         sv_dtype dtype,
                         const int32_t *draft_tokens, const double *uniforms,
                         int B, int K, int V,
                         const float *temperature, const float *top_p, const int32_t *top_k,
                         int saguaro_F, float saguaro_C,
                         int32_t *accept_len, int32_t *out_tokens,
                         sv_stats *stats, void *workspace, size_t workspace_bytes,
                         size_t *h2d_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_verify_lazy — sv_verify that reads each sequence's rows position by position and stops at
 * its first rejection.
 * [SpS notes §3: after the first rejection the draft tokens to its right are discarded, so
 *  their rows decide nothing]
 *
 * Arguments, workspace (sv_verify_workspace_size) and outputs are those of sv_verify, and the
 * outputs are identical.  Rows after a sequence's first rejection (after its first greedy
 * mismatch) are never read: their debug fields stay NaN, they do not count in stats.rows, and
 * non-finite values in them raise no error.  The bytes read fall with the acceptance rate
 * (about 30% of sv_verify's at the large-batch workload).  Calls with top_p, top_k or an active
 * sigma_{F,C} (saguaro_F > 0 and saguaro_C != 1) run the sv_verify pipeline unchanged.  One
 * kernel of the call waits on work that other blocks of the same launch queue; it is
 * launched cooperatively, so SV_ERR_CUDA results if the device cannot hold all its blocks.
 * -------------------------------------------------------------------------------------- */
sv_status sv_verify_lazy(const void *target_logits, int64_t t_row_pitch,
                         const void *draft_logits, int64_t d_row_pitch, int d_rows_per_seq,
                         sv_dtype dtype,
                         const int32_t *draft_tokens, const double *uniforms,
                         int B, int K, int V,
                         const float *temperature, const float *top_p, const int32_t *top_k,
                         int saguaro_F, float saguaro_C,
                         int32_t *accept_len, int32_t *out_tokens,
                         double *debug, sv_stats *stats,
                         void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_verify_static — sv_verify for callers that cannot allocate device memory.  The paper
 * has no counterpart: this is a deployment convenience, not a step of the method.
 *
 * Who needs it: a serving engine that hands (nearly) all free HBM to its KV-cache pool when
 * it starts, so that a cudaMalloc later, in the decode loop, would fail or eat into that
 * pool; and a host program that loads this library as a plug-in and owns every device
 * allocation in its process.  Neither can give sv_verify a workspace of its own.
 *
 * The arguments and results are those of sv_verify without workspace/workspace_bytes.  The
 * scratch lives in one fixed device array of SV_STATIC_SCRATCH_BYTES (32 MiB) inside the
 * library, which every GPU that loads the library holds until the process exits.  The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 *  - Limit: a call whose scratch need for (B, K, V, dtype) exceeds SV_STATIC_SCRATCH_BYTES
 *    returns SV_ERR_WORKSPACE before any device work (B = 512, K = 5, V = 128256 needs about
 *    23.9 MiB and fits).  sv_verify_workspace_size(B, K, V) bounds the need from above.
 *  - Set-up: the first call on a device, with that device current, looks up the array's
 *    device address (cudaGetSymbolAddress) and caches it for that device; a failure there
 *    returns SV_ERR_CUDA.  Make that first call before any stream capture.  The cached
 *    address belongs to the device's context at that time: after cudaDeviceReset, or after
 *    the primary context is released and created again, it is stale, so a process that
 *    resets a device must not call sv_verify_static on it afterwards.
 *  - Contents: every call shares the array, and it keeps the last call's contents.  Nothing
 *    in it has to start at zero: each call's first kernel clears its counters (queued draws,
 *    queued float-float items, grid-barrier count, next unit of the statistics pass) on its
 *    stream once the stream's previous kernel has finished, and every other byte is written
 *    before it is read within the same call.
 *  - Races: calls whose kernels overlap on the GPU (other streams, other host threads on the
 *    same device) use the same scratch and race.  Order them, e.g. on one stream.
 * -------------------------------------------------------------------------------------- */
#define SV_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

sv_status sv_verify_static(const void *target_logits, int64_t t_row_pitch,
                           const void *draft_logits, int64_t d_row_pitch, int d_rows_per_seq,
                           sv_dtype dtype,
                           const int32_t *draft_tokens, const double *uniforms,
                           int B, int K, int V,
                           const float *temperature, const float *top_p, const int32_t *top_k,
                           int saguaro_F, float saguaro_C,
                           int32_t *accept_len, int32_t *out_tokens,
                           double *debug, sv_stats *stats, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_fuzzy_verify — one verification stage of three-model speculative decoding: a verifier
 * (the qualifier checking the draft model, or the target checking the qualifier) accepts a
 * drafter's tokens position by position.
 * [PyramidSD notes, "Method": fuzzy acceptance Div(P_verifier, P_drafter) <= tau (PSDF) and
 *  assisted acceptance (PSDA); SpS notes §3 for the test the assisted mode keeps]
 *
 *  mode SV_ACCEPT_DIVERGENCE  position i+1 passes while the Jensen-Shannon divergence (bits,
 *                  in [0, 1]) of the verifier's and the drafter's distributions at that
 *                  position is <= tau, whatever the drafted token; uniforms[b][i < K] unused.
 *  mode SV_ACCEPT_ASSISTED    position i+1 passes iff u[b][i] < min(1, q(s)/p(s)) (greedy: s ==
 *                  argmax q), as in sv_verify; tau unused.
 *  In both modes the first failing position takes a token drawn from the verifier's
 *  distribution there (inverse CDF in id order at u[b][K]; greedy: its argmax), and when all K
 *  pass the verifier's row K+1 gives the bonus token.  The divergence is certified: a value
 *  the float32 bound cannot place on one side of tau is recomputed in float-float.
 *
 *  verifier_logits  dev, rows (b, j), j = 0..K, pitch v_row_pitch (as sv_verify's target).
 *  drafter_logits   dev, rows (b, j) at b*d_rows_per_seq+j, j < K.  Read for every sequence.
 *  temperature      dev float [B]: 0 greedy (one-hot rows: Div is 0 or 1), else [1e-3, 1e3].
 *  divergence       dev float64 [B][K] or NULL (must be NULL in the assisted mode): Div of every
 *                   position (certified to the float32 bound, or float-float where that bound
 *                   could not place it on one side of tau).
 *  accept_len, out_tokens, stats, workspace as sv_verify (workspace: sv_fuzzy_verify_workspace_size).
 * Returns SV_ERR_INVALID_ARG for a bad mode, a non-finite tau, or the conditions of sv_verify.
 * -------------------------------------------------------------------------------------- */
typedef enum { SV_ACCEPT_DIVERGENCE = 0, SV_ACCEPT_ASSISTED = 1 } sv_accept_mode;

size_t sv_fuzzy_verify_workspace_size(int B, int K, int V);

sv_status sv_fuzzy_verify(const void *verifier_logits, int64_t v_row_pitch,
                          const void *drafter_logits, int64_t d_row_pitch, int d_rows_per_seq,
                          sv_dtype dtype,
                          const int32_t *draft_tokens, const double *uniforms,
                          int B, int K, int V,
                          const float *temperature, float tau, int mode,
                          int32_t *accept_len, int32_t *out_tokens,
                          double *divergence, sv_stats *stats,
                          void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_tree_verify — verify a tree of drafted tokens per sequence in one pass.
 * [Mirror-SD notes §1.1 (tree drafts verified at once), §3.1 (branch-complete trees); SpS notes
 *  §3 (the accept test and the residual, applied again after each rejection)]
 *
 * Node i (1..N) holds tokens[b][i-1] below node parents[b][i-1] in [0, i-1]; node 0 is the
 * committed context.  Row i of target_logits / draft_logits is the distribution that follows node
 * i; a node's children are drafted from its draft row.
 *  Greedy (T == 0): from node 0, move to the first child (lowest index) holding the target argmax;
 *    the target argmax where no child matches is the correction.
 *  Sampled: the children of the current node are tested in index order; child i passes iff
 *    u[b][i] < min(1, (q(t) - c_i p(t))+ / (R(c_i) p(t))), R(c) = sum_v (q_v - c p_v)+, c_1 = 0,
 *    c_(i+1) = c_i + R(c_i) (SpS's residual applied again after each rejection: lossless).  A
 *    passing child becomes the current node; when every child fails (or there is none) t* is
 *    drawn from (q - c p)+ by the inverse CDF in id order at u[b][0].
 *  Decisions are certified in float32 and redone in float-float where the margin is too thin.
 *
 *  target_logits, draft_logits  dev, rows (b, i) at b*(N+1)+i, i = 0..N, pitches in elements.
 *                 Draft rows of greedy sequences are not read; draft rows of leaves are read
 *                 by the statistics pass but not used (they must be finite).
 *  parents, tokens  dev int32 [B][N]; uniforms dev float64 [B][N+1]; temperature dev float [B].
 *  accept_len     dev int32 [B]: the number of accepted nodes k (the depth reached).
 *  out_tokens     dev int32 [B][N+1]: the k accepted tokens, t*, then -1.
 *  path           dev int32 [B][N] or NULL: the accepted node ids, then -1.
 * Errors (stats): SV_ERR_INVALID_ARG for a parent outside [0, i-1] or a bad temperature,
 * SV_ERR_BAD_TOKEN for a token outside [0, V), SV_ERR_NONFINITE for a non-finite row used.
 * -------------------------------------------------------------------------------------- */
size_t sv_tree_verify_workspace_size(int B, int N, int V);

sv_status sv_tree_verify(const void *target_logits, int64_t t_row_pitch,
                         const void *draft_logits, int64_t d_row_pitch, sv_dtype dtype,
                         const int32_t *parents, const int32_t *tokens, const double *uniforms,
                         int B, int N, int V, const float *temperature,
                         int32_t *accept_len, int32_t *out_tokens, int32_t *path,
                         sv_stats *stats, void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_tree_reuse — does the committed prefix spell a path of a drafted tree?
 * [Mirror-SD notes §3.2-§3.3: reuse when (accepted tokens, correction) is a path of the
 *  branch-complete tree, a depth-2 node with several branches included]
 *  parents, tokens  dev int32 [B][N] (as sv_tree_verify); accept_len dev int32 [B];
 *  out_tokens       dev int32 [B][K+1] (k accepted tokens then the correction);
 *  reuse_node       dev int32 [B] (output): the node where the path ends (1..N), or -1.
 * At each depth the first child (lowest index) holding the committed token is followed.
 * -------------------------------------------------------------------------------------- */
sv_status sv_tree_reuse(const int32_t *parents, const int32_t *tokens, int N,
                        const int32_t *accept_len, const int32_t *out_tokens, int K, int B,
                        int32_t *reuse_node, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_saguaro_sample — draw one token from each of the first n_rows rows of every sequence's
 * draft distribution p' = sigma_{F,C}(p): p after temperature, top-k and top-p, the top-F tokens
 * (ranked by draft logit) scaled by C, renormalised.  F = 0 or C = 1 is a plain draft sampler.
 * [SSD notes §4.4 Theorem 15 (scaling the cached tokens' draft mass raises the hit rate),
 *  Theorem 19 (worked example); SSD abstract page, "Method" (sigma_{F,C})]
 *
 *  draft_logits  dev, rows (b, j) at b*rows_per_seq+j, pitch row_pitch; rows j < n_rows used.
 *  temperature   dev float [B] (0: argmax), top_p dev float [B] or NULL, top_k dev int32 [B]
 *                or NULL (both as in sv_verify).
 *  uniforms      dev float64 [B][n_rows].
 *  tokens        dev int32 [B][n_rows] (output).
 *  debug         dev float64 [B][n_rows][4] or NULL: LSE, P_D (top-F mass before scaling),
 *                Z' (normaliser after scaling), mass kept by the top-k / top-p filters.
 * A row where C = 0 and all of p's mass lies in the top-F set has no defined transform and
 * is sampled from p unchanged.
 * -------------------------------------------------------------------------------------- */
size_t sv_saguaro_sample_workspace_size(int B, int n_rows, int V);

sv_status sv_saguaro_sample(const void *draft_logits, int64_t row_pitch, int rows_per_seq,
                            sv_dtype dtype, int B, int n_rows, int V,
                            const float *temperature, const float *top_p, const int32_t *top_k,
                            int F, float C, const double *uniforms,
                            int32_t *tokens, double *debug, sv_stats *stats,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_fanout — Theorem 12 fan-out, host only.  [SSD abstract page, "Method"; SSD notes §4.3]
 *   F_k = F_0 a^(k/(1+r)) for k < K,  F_K = F_0 a^(K/(1+r)) (1-a)^(-1/(1+r)),  sum_k F_k = budget.
 *  F_real  host float64 [K+1] (output), summing to budget.
 *  F_int   host int32 [K+1] (output): floor(F_real) plus one for the largest fractional parts
 *          (ties to the smaller k) until the sum is floor(budget).
 * Requires 0 < a < 1, r > -1, budget >= 0 (finite, < 2^31), 0 <= K <= SV_MAX_K.
 * -------------------------------------------------------------------------------------- */
sv_status sv_fanout(double budget, double a, double r, int K, double *F_real, int32_t *F_int);

/* ----------------------------------------------------------------------------------------
 * sv_cache_keys — the speculation cache's key set.  [SSD notes §5.1; SSD abstract page]
 * For depth k < K: the top-F_k tokens of draft row k (the row that proposed s_{k+1}), ranked by
 * raw logit, after removing s_{k+1}; for depth K: the top-F_K tokens of draft row K.
 *  draft_logits  dev, rows (b, j) at b*rows_per_seq+j, j = 0..K used (rows_per_seq >= K+1).
 *  draft_tokens  dev int32 [B][K].
 *  F_int         host int32 [K+1], 0 <= F_k <= V-1 (k < K), 0 <= F_K <= V.
 *  keys          dev int32 [B][sum F_k], depth-major: depth k occupies
 *                [sum_{i<k} F_i, sum_{i<=k} F_i).
 * -------------------------------------------------------------------------------------- */
size_t sv_cache_keys_workspace_size(int B, int K, int V);

sv_status sv_cache_keys(const void *draft_logits, int64_t row_pitch, int rows_per_seq,
                        sv_dtype dtype, const int32_t *draft_tokens, const int32_t *F_int,
                        int B, int K, int V, int32_t *keys, sv_stats *stats,
                        void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_cache_lookup — hit[b] = 1 iff t* = out_tokens[b][k] is among the depth-k keys of sequence
 * b, with k = accept_len[b].  [SSD abstract page, "Method": cache lookup on (k, t*)]
 *  accept_len dev int32 [B]; out_tokens dev int32 [B][K+1]; keys dev int32 [B][sum F_int];
 *  F_int host int32 [K+1]; hit dev uint8 [B] (output).
 * A corrupt accept_len (outside [0, K]) yields hit 0.
 * -------------------------------------------------------------------------------------- */
sv_status sv_cache_lookup(const int32_t *accept_len, const int32_t *out_tokens,
                          const int32_t *keys, const int32_t *F_int, int B, int K,
                          uint8_t *hit, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_topk_rows — top-kappa token ids of each logit row (logit desc, id asc) and their
 * log-probabilities log softmax(x / T).  [Mirror-SD notes §3.1: the early-exit head's top-kappa
 * (token, log-prob) pairs become the branch roots]
 *  logits       dev, n_rows rows with pitch row_pitch.
 *  temperature  dev float [n_rows] (> 0) or NULL for T = 1.
 *  ids          dev int32 [n_rows][kappa]; logprobs dev float64 [n_rows][kappa] (may be NULL).
 * Requires 1 <= kappa <= min(V, 1024).  A row with T outside [1e-3, 1e3] is reported in stats.
 * -------------------------------------------------------------------------------------- */
size_t sv_topk_rows_workspace_size(int n_rows, int V);

sv_status sv_topk_rows(const void *logits, int64_t row_pitch, sv_dtype dtype, int n_rows,
                       int V, int kappa, const float *temperature, int32_t *ids,
                       double *logprobs, sv_stats *stats, void *workspace,
                       size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_mirror_reuse — reuse[b] = 1 iff k = accept_len[b] < gamma and the committed prefix
 * (s_1..s_k, t*) = out_tokens[b][0..k] equals the first k+1 tokens of some branch.
 * [Mirror-SD notes §3.2: reuse vs. fallback]
 *  branches dev int32 [B][kappa][gamma]; accept_len dev int32 [B];
 *  out_tokens dev int32 [B][gamma+1]; reuse dev uint8 [B] (output).
 * -------------------------------------------------------------------------------------- */
sv_status sv_mirror_reuse(const int32_t *branches, const int32_t *accept_len,
                          const int32_t *out_tokens, int B, int kappa, int gamma,
                          uint8_t *reuse, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * sv_set_profile_events — measurement hook (no counterpart on the pages).  begin and end are
 * cudaEvent_t handles (or NULL to disable).  While set, every call made from this host thread
 * records `begin` on its stream just before its statistics pass (the one streaming read of the
 * logit rows, the call's dominant kernel) and `end` just after it, so the caller can time that
 * kernel with cudaEventElapsedTime.  The setting is thread-local and persists until changed.
 * -------------------------------------------------------------------------------------- */
void sv_set_profile_events(void *begin, void *end);

/* ----------------------------------------------------------------------------------------
 * Self-tests of the device error paths (no counterpart on the pages).
 *
 * sv_selftest_timeout: one block waits on a shared-memory barrier that nothing completes,
 * gives up after `limit_cycles` SM clock cycles, and reports SV_ERR_TIMEOUT in stats.  It
 * shows that the library's bounded waits return an error instead of hanging; no copy is in
 * flight and nothing faults.
 *
 * sv_selftest_exp2: evaluates the library's fast base-2 exponential (the float32 tier) and
 * its float-float exponential on n inputs spread over [lo, hi] and writes their largest
 * relative errors against CUDA's double-precision exp2 to out[0] (fast) and out[1]
 * (float-float).  The bounds that certify float32 decisions rest on these errors.
 * -------------------------------------------------------------------------------------- */
sv_status sv_selftest_timeout(int64_t limit_cycles, sv_stats *stats, sv_stream_t stream);
sv_status sv_selftest_exp2(double lo, double hi, int64_t n, double *out, sv_stream_t stream);

/* sv_selftest_exp2_all: the same two errors over EVERY float32 input in [lo, hi] (lo >= -125,
 * hi <= 100) whose exact result is above 2^-125; out[0] fast, out[1] float-float, out[2] the
 * number of inputs evaluated (a double).  Over [-125, 1] this is an exhaustive proof of the
 * fast exponential's error bound on the GPU it runs on (about 2.2e9 inputs). */
sv_status sv_selftest_exp2_all(float lo, float hi, double *out, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
