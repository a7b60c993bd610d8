/*
 * specverify.h — C ABI of the batched speculative-decoding verifier
 * (rejection sampler) for NVIDIA GB300 (sm_103a).
 *
 * What it computes. For every request b the caller has K_b draft tokens
 * d_1..d_K, the target model's logits for the K_b+1 positions that one
 * verification pass scores (p_1..p_{K+1}, each conditioned on the drafts
 * before it) and the draft's law q_1..q_K. The verifier commits the accepted
 * prefix of the drafts and one more token:
 *
 *   - lossless rule: accept d_i with probability min(1, p_i(d_i)/q_i(d_i))
 *     (outright when q <= p), stop at the first rejection, draw the
 *     replacement from norm(max(0, p - q)); when all K are accepted draw a
 *     bonus token from p_{K+1}.
 *       Sources: "Acceptance Is Not Speed (arXiv:2610.23818)", §1 and §6;
 *       "RheoSampling 2026", §4 "RheoVerification"; nalar.dev "Speculative
 *       decoding: memverifikasi token draft sebelum diterima", sections
 *       "Draft mengubah tebakan serial menjadi batch verifikasi",
 *       "Semantik penerimaan" and "Penolakan memendekkan pekerjaan
 *       speculative".
 *   - greedy (T < 0.05, or rule SPEC_RULE_GREEDY): accept while d_i equals
 *     argmax p_i (lowest id on ties); the target's argmax replaces the first
 *     mismatch, or is the bonus token. (nalar.dev, "Semantik penerimaan".)
 *   - p = softmax(z_t / T), q = softmax(z_d / T) with the request's
 *     temperature T ("RheoSampling 2026", §1 and §7).
 *   - top-128 draft truncation: the draft logits keep their 128 largest
 *     entries (ties to the lower id), the rest is -inf, then the softmax
 *     ("RheoSampling 2026", §3).
 *   - tree verification by recursive rejection sampling without replacement
 *     over siblings ("RheoSampling 2026", §4).
 *   - relaxed (lossy) CACTUS rule: accept d_i with probability
 *     min(1, gamma/q_i(d_i)), gamma = min(p + sqrt(2 alpha p (1 - p)), 1) at
 *     p = p_i(d_i), after a low-support guard that rejects outright a draft
 *     whose target rank exceeds k or whose p is below a floor ("Acceptance
 *     Is Not Speed (arXiv:2610.23818)", §2, §6 rules 1-3 and §7 item 3). The
 *     page's residual for this rule is lost; the library draws the
 *     replacement from norm(max(0, p - q)) as in the lossless rule.
 *
 * Random numbers. Every uniform is u = (splitmix64(seed ^ splitmix64(key))
 * >> 40) * 2^-24 with key = (b << 32) | (pos << 8) | stream, where
 * splitmix64(x) is the SplitMix64 output function (Steele, Lea & Flood 2014)
 * of x + 0x9E3779B97F4A7C15. stream 0 = acceptance coin, 1 = residual draw,
 * 2 = bonus draw. Linear: pos = 1-based position (coin of d_i at i, final
 * draw at n+1). Tree: the coin of child c at pos = c (local node id), the
 * final draw at node v at pos = v + 1. A draw at u picks the smallest token
 * x (ascending id) with u * Z < C_x, C the inclusive prefix sum of the
 * weights and Z their total.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller unless stated; the
 *     library allocates nothing and keeps no state between calls. Logit and
 *     probability buffers must be 16-byte aligned; rows are contiguous with
 *     a row stride of V elements.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *   - A negative return value is a host-detected error; nothing was
 *     launched. SPEC_OK means the work was enqueued.
 *   - Errors found on the device (bad offsets, tokens out of range, a
 *     temperature that is negative or NaN, a malformed tree, a bounded wait
 *     that ran out) are written to a status word in the workspace; read it
 *     with spec_get_status(). Outputs of the affected requests are then
 *     unspecified.
 *   - Logits must be finite or -inf; NaN is undefined behaviour. Each row
 *     needs at least one finite logit.
 *   - Deterministic: the same inputs and seed give the same bits.
 *   - Calls that share a workspace must not overlap on the device.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st *spec_stream_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = -1, /* bad pointer, size, enum or input value      */
  SPEC_ERR_UNSUPPORTED = -2, /* valid but outside this build's limits        */
  SPEC_ERR_WORKSPACE = -3,   /* workspace NULL, misaligned or too small      */
  SPEC_ERR_CUDA = -4,        /* a CUDA runtime call failed                   */
  SPEC_ERR_TIMEOUT = -5,     /* a bounded device-side wait ran out           */
  SPEC_ERR_BOUNDS = -6       /* checked build only: an access outside the
                                call's buffers (detail: its source line)     */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
  SPEC_DRAFT_LOGITS = 0,    /* draft [R_d, V] logits; q = softmax(z/T)       */
  SPEC_DRAFT_PROBS = 1,     /* draft [R_d, V] probabilities, used as given   */
  SPEC_DRAFT_SPARSE128 = 2  /* draft [R_d, 128] f32 probs + draft_idx ids    */
} spec_draft_kind;

typedef enum {
  SPEC_RULE_STRICT = 0,       /* lossless; requests with T < 0.05 greedy     */
  SPEC_RULE_GREEDY = 1,       /* every request greedy                        */
  SPEC_RULE_STRICT_TOP128 = 2, /* lossless, dense draft logits cut to top-128 */
  SPEC_RULE_CACTUS = 3         /* relaxed rule + guard; needs spec_linear_ext */
} spec_rule;

#define SPEC_TOPK 128
#define SPEC_MAX_K 256          /* drafts per request                        */
#define SPEC_MAX_V (1 << 24)    /* vocabulary size                           */
#define SPEC_MAX_TREE_NODES 4096 /* nodes per tree                           */
#define SPEC_MAX_TREE_DEPTH 64
#define SPEC_MAX_TREE_BRANCH 64
#define SPEC_GREEDY_T 0.05f

/* Human-readable name of a spec_status value (static string). */
const char *spec_status_string(int status);

/* Bytes of workspace spec_verify_linear needs for at most B requests of at
 * most max_k drafts each over a vocabulary of V (0 on invalid sizes). */
size_t spec_verify_linear_workspace(int B, int max_k, int V, int rule);

/*
 * Linear verification of B requests.
 *
 *   target       [R_t, V] logits (tdt), R_t = cu_draft[B] + B. Request b's
 *                rows p_1..p_{K+1} start at row cu_draft[b] + b.
 *   draft        dk == LOGITS: [R_d, V] logits (ddt); PROBS: [R_d, V]
 *                probabilities (ddt), no temperature applied; SPARSE128:
 *                [R_d, 128] f32 probabilities (ddt must be SPEC_F32).
 *                R_d = cu_draft[B]; request b's rows start at cu_draft[b].
 *                May be NULL when every request is greedy.
 *   draft_idx    SPARSE128 only: [R_d, 128] int32 token ids (-1 = empty
 *                slot, any order, no duplicates); NULL otherwise.
 *   draft_tokens [R_d] int32 in [0, V).
 *   cu_draft     [B+1] int32, cu_draft[0] = 0, 0 <= K_b <= max_k.
 *   temperature  [B] f32, >= 0; T < 0.05 makes the request greedy.
 *   rule         spec_rule. SPEC_RULE_STRICT_TOP128 needs dk == LOGITS.
 *   out_tokens   [B, max_k+1] int32: d_1..d_n, the final token, then -1.
 *   out_accepted [B] int32: n, the number of accepted drafts.
 *   out_pq       optional [R_d, 2] f32 {p_i(d_i), q_i(d_i)} for every draft
 *                position (also after the first rejection); greedy
 *                requests give {1 if d_i == argmax p_i else 0, -1}. NULL to
 *                skip.
 *   workspace    device scratch, >= spec_verify_linear_workspace(...) bytes,
 *                256-byte aligned, contents need no initialisation.
 * Schedule: small calls run as one fused kernel (spec_set_fused_limit). Any
 * other call with out_pq NULL, draft logits, bf16 target and draft
 * rows, V a multiple of 8 and rule SPEC_RULE_STRICT or SPEC_RULE_GREEDY
 * runs the position-lazy streaming schedule (SPEC_EXT_LAZY below): a
 * request's rows after its first rejection are not used, so a row there
 * without a finite logit is not reported. Other calls read every row (the
 * eager schedule); spec_verify_linear_ext with SPEC_EXT_EAGER forces it.
 * Both give the same tokens and counts up to the rounding of the row sums.
 * Returns SPEC_OK or a negative spec_status.
 */
int spec_verify_linear(const void *target, int tdt, const void *draft, int ddt,
                       int dk, const int32_t *draft_idx,
                       const int32_t *draft_tokens, const int32_t *cu_draft,
                       const float *temperature, int B, int V, int max_k,
                       uint64_t seed, int rule, int32_t *out_tokens,
                       int32_t *out_accepted, float *out_pq, void *workspace,
                       size_t ws_bytes, spec_stream_t stream);

/*
 * Tuning of the linear verifier's schedule. A call with rule
 * SPEC_RULE_STRICT or SPEC_RULE_GREEDY, draft logits or probabilities and
 * no options runs as one fused kernel, one block per request, when V is at
 * most 8192, a request's rows ((max_k + 1) target rows and max_k draft rows)
 * total at most 1 MiB and all B requests' rows at most `bytes`. Such calls
 * are decode steps over short rows, where one launch costs less than the
 * multi-kernel schedule. A call of the same rules on bf16 draft logits with
 * longer rows (V a multiple of 8), at most 128 requests and at most 8
 * drafts each, whose (2 max_k + 1) row slices of V/8 logits fit 100 KB of
 * shared memory (V up to about 37000 at max_k = 5), runs as one cluster
 * kernel instead: a cluster of 8 CTAs per request streams the request's
 * rows through a few row-slice buffers per CTA, exchanges their statistics
 * once and draws the final token from the two rows it needs, copied again.
 * Same results either way, up to the rounding of the row sums. `bytes` = 0 turns both kernels off; the default is
 * 32 MiB. A process-wide setting, read when a call is made. Returns the
 * previous value.
 */
size_t spec_set_fused_limit(size_t bytes);

/*
 * Options of spec_verify_linear_ext (host memory, read during the call).
 *   alpha     SPEC_RULE_CACTUS divergence budget, finite and >= 0; 0 makes
 *             gamma = p, the lossless test.
 *   max_rank  guard: reject d_i when its target rank (1 + the number of
 *             tokens whose target logit is strictly larger than d_i's; ties
 *             share the better rank) exceeds max_rank; 0 = off. Used by
 *             SPEC_RULE_CACTUS only.
 *   min_prob  guard: reject d_i when p_i(d_i) < min_prob; 0 = off.
 *             SPEC_RULE_CACTUS only.
 *   flags     0, SPEC_EXT_LAZY, SPEC_EXT_RESIDENT or SPEC_EXT_EAGER.
 *             SPEC_EXT_LAZY: position-lazy verification. Position
 *             i is decided only when drafts 1..i-1 were accepted, so a
 *             request's decisions use rows 1..n+1 only (nalar.dev "Penolakan
 *             memendekkan pekerjaan speculative": proposals after a rejected
 *             one are discarded). Same tokens and counts as the eager call;
 *             out_pq is NaN and out_rank -1 on the positions after n+1.
 *             Dense bf16 logits with V a multiple of 8 and no out_kl run as
 *             one persistent kernel that scans every position's rows in
 *             layer order, skips a request's rows once it has rejected, and
 *             checks every draft token; it may still read some rows after a
 *             rejection (never used, so they are not checked). Other inputs
 *             run one row pass and one decision per position (max_k + 1
 *             rounds), read rows 1..n+1 only and do not check the tokens
 *             after n+1. The top-128 rule still cuts every draft row.
 *             SPEC_EXT_RESIDENT: the position-lazy schedule with every
 *             needed row read from HBM exactly once. A cluster of 8 CTAs
 *             holds the current position's target and draft rows in shared
 *             memory (1/8 each) while it decides, and draws the final token
 *             from that copy. Same results as SPEC_EXT_LAZY. It reads fewer bytes
 *             but waits on a cluster-wide exchange per position, so it is
 *             slower on a GPU of its own (B = 1024, K = 4, V = 201088:
 *             0.97 ms against 0.54 ms); it suits calls that share HBM with
 *             other work. Takes the strict or greedy rule on dense bf16
 *             logits with V a multiple of 8 and 16384 <= V <= 204800, and
 *             no rank or KL output; other calls run as SPEC_EXT_LAZY.
 *             SPEC_EXT_EAGER: read every row of every position (the
 *             eager schedule), also where a plain call would take the
 *             position-lazy one. Not combined with the other two.
 *   out_rank  optional device [R_d] int32: the target rank of every draft
 *             token (every request and rule; also after the first
 *             rejection unless lazy). NULL to skip.
 *   out_kl    optional device [R_d] f32: KL(p_i || q_i) in nats for every
 *             draft position of a sampling request, with p and q the laws
 *             the verifier uses; NaN for greedy requests (and, lazy, after
 *             position n+1). The distillation signal of "Test-Time
 *             Speculation" §2 step 3, taken from the same single read: each
 *             target row is streamed together with its draft row. Needs
 *             draft logits (SPEC_DRAFT_LOGITS) of the target's dtype, rows
 *             whose byte length is a multiple of 16, and a rule other than
 *             SPEC_RULE_STRICT_TOP128 (whose truncated q makes it +inf).
 *             NULL to skip.
 *   seed_dev  optional device uint64, 8-byte aligned: when set, the kernels
 *             read the seed from it as they run and the `seed` argument is
 *             ignored. A call captured in a CUDA graph then draws new
 *             uniforms on every replay after the caller writes a new seed
 *             there. NULL to use `seed`.
 * The guard and the relaxed coin apply to sampling requests; greedy
 * requests (T < 0.05) keep the greedy rule.
 */
#define SPEC_EXT_LAZY 1
#define SPEC_EXT_RESIDENT 2
#define SPEC_EXT_EAGER 4
typedef struct {
  float alpha;
  int32_t max_rank;
  float min_prob;
  int32_t flags;
  int32_t *out_rank;
  float *out_kl;
  const uint64_t *seed_dev;
} spec_linear_ext;

/*
 * spec_verify_linear with options: the same arguments and semantics, plus
 * `ext` (NULL = no options, then identical to spec_verify_linear).
 * SPEC_RULE_CACTUS requires ext. Needs spec_verify_linear_workspace(B,
 * max_k, V, rule) bytes of workspace.
 */
int spec_verify_linear_ext(const void *target, int tdt, const void *draft,
                           int ddt, int dk, const int32_t *draft_idx,
                           const int32_t *draft_tokens,
                           const int32_t *cu_draft, const float *temperature,
                           int B, int V, int max_k, uint64_t seed, int rule,
                           const spec_linear_ext *ext, int32_t *out_tokens,
                           int32_t *out_accepted, float *out_pq,
                           void *workspace, size_t ws_bytes,
                           spec_stream_t stream);

/*
 * No-allocation variant of spec_verify_linear. The paper has no counterpart:
 * this exists for callers that cannot supply device scratch, such as serving
 * engines that reserve nearly all of HBM for their KV cache at start-up (a
 * later cudaMalloc fails) and decode loops that must not call
 * cudaMalloc/cudaFree because those calls synchronise the device.
 *
 * Same inputs, outputs and semantics as spec_verify_linear; the scratch is a
 * SPEC_NOALLOC_SCRATCH_BYTES array compiled into the library, which every GPU
 * that loads the library holds until the process exits. Sizes whose
 * spec_verify_linear_workspace() exceeds it return SPEC_ERR_UNSUPPORTED.
 * All calls on a device share that array: calls that overlap on the GPU
 * race, so order them (one stream, or events). The first call on each device
 * looks up the array's address (cudaGetSymbolAddress, with that device
 * current); make it before any stream capture. The address is kept per
 * device context: the first call after cudaDeviceReset looks it up again,
 * so make that call before any stream capture as well. Nothing is
 * allocated.
 *
 *   out_status  optional device int32: receives the call's device status word
 *               (SPEC_OK or a negative spec_status) once the call's work is
 *               done on `stream`; NULL to skip.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (16u << 20)
int spec_verify_linear_noalloc(const void *target, int tdt, const void *draft,
                               int ddt, int dk, const int32_t *draft_idx,
                               const int32_t *draft_tokens,
                               const int32_t *cu_draft,
                               const float *temperature, int B, int V,
                               int max_k, uint64_t seed, int rule,
                               int32_t *out_tokens, int32_t *out_accepted,
                               float *out_pq, int32_t *out_status,
                               spec_stream_t stream);

/* Bytes of workspace spec_verify_tree needs (0 on invalid sizes). */
size_t spec_verify_tree_workspace(int B, int n_nodes, int V, int max_depth,
                                  int max_branch);

/*
 * Tree verification (RRSw) of B request trees.
 *
 *   target      [n_nodes, V] logits (tdt). Row n is the target law after the
 *               path root..n ("RheoSampling 2026", §4).
 *   draft       [n_nodes, V] logits (dk == LOGITS) or probabilities
 *               (dk == PROBS) (ddt). Row n is the law node n's children were
 *               drawn from, without replacement; rows of leaves are unused.
 *               May be NULL when every tree is greedy.
 *   node_token  [n_nodes] int32: the token of each node (roots unused).
 *   parent      [n_nodes] int32: LOCAL parent id, -1 for the root (local
 *               node 0); parent[c] < c. Siblings carry distinct tokens, in
 *               the order they were drawn (a repeated token is invalid
 *               input: SPEC_ERR_INVALID_ARG in the status word).
 *   cu_nodes    [B+1] int32 node offsets, cu_nodes[B] = n_nodes, at most
 *               SPEC_MAX_TREE_NODES nodes per tree.
 *   max_depth   bound on the depth of every tree (out width max_depth+1).
 *   max_branch  bound on the children of any node.
 *   out_tokens  [B, max_depth+1] int32: accepted path tokens, the final
 *               token, then -1.
 *   out_accepted [B] int32: number of accepted nodes.
 *   out_path    [B, max_depth+1] int32: local ids of the accepted nodes, -1
 *               padded. May be NULL.
 * Only the rows of the nodes the walk visits (the root and the accepted
 * path) are read: a node's statistics are computed when the walk reaches it,
 * so rows of other nodes are neither read nor checked.
 */
int spec_verify_tree(const void *target, int tdt, const void *draft, int ddt,
                     int dk, const int32_t *node_token, const int32_t *parent,
                     const int32_t *cu_nodes, const float *temperature, int B,
                     int n_nodes, int V, int max_depth, int max_branch,
                     uint64_t seed, int32_t *out_tokens, int32_t *out_accepted,
                     int32_t *out_path, void *workspace, size_t ws_bytes,
                     spec_stream_t stream);

/*
 * spec_verify_tree with point-mass children ("RheoSampling 2026", §4 with
 * deterministic candidates, such as the leads spec_rheo_expand builds).
 * Same arguments and semantics, plus
 *   node_fixed  [n_nodes] int32 or NULL (= spec_verify_tree): nonzero marks
 *               a node that was not drawn from its parent's draft law. Such
 *               a child x is accepted with probability p_j(x), p_j the
 *               parent's current target law; on rejection p_{j+1} is p_j
 *               without x, renormalised, and the draft law of the drawn
 *               siblings is unchanged (without replacement runs over drawn
 *               children only). Roots' flags are ignored.
 * Children are still tested in node-index order. The test is lossless when
 * a fixed child's token does not depend on the draws of the siblings tested
 * after it: for a RheoSampling node list the probe (slot m of
 * spec_rheo_expand) first, then the other slots in order. Drawn siblings
 * carry distinct tokens; a fixed child may repeat a sibling's token.
 *   seed_dev    optional device uint64, 8-byte aligned: when set, the walk
 *               reads the seed from it as it runs and `seed` is ignored (for
 *               calls replayed from a CUDA graph). NULL to use `seed`.
 */
int spec_verify_tree_ext(const void *target, int tdt, const void *draft,
                         int ddt, int dk, const int32_t *node_token,
                         const int32_t *parent, const int32_t *node_fixed,
                         const int32_t *cu_nodes, const float *temperature,
                         int B, int n_nodes, int V, int max_depth,
                         int max_branch, uint64_t seed,
                         const uint64_t *seed_dev, int32_t *out_tokens,
                         int32_t *out_accepted, int32_t *out_path,
                         void *workspace, size_t ws_bytes,
                         spec_stream_t stream);

/*
 * Bytes of workspace draft_topk_softmax needs (0 on invalid sizes): a
 * 256-byte header, and for V % 8 == 0 with V >= 4096 the candidate lists of
 * the two-launch select (4 KB and 4 bytes per row).
 */
size_t draft_topk_softmax_workspace(int rows, int V);

/*
 * Sparse top-128 draft law ("RheoSampling 2026", §3): for every draft row the
 * ids of its 128 largest logits (ties to the lower id) in ascending id order,
 * and softmax(z/T) over those 128 only. Rows of request b (cu_rows[b] ..
 * cu_rows[b+1]-1) use temperature[b]; T < 0.05 gives probability 1 on the
 * argmax. When V < 128 the tail slots hold id -1 and probability 0.
 *
 *   draft_logits [rows, V] (dt); cu_rows [B+1] int32 with cu_rows[B] = rows;
 *   k must be 128; out_idx [rows, 128] int32; out_prob [rows, 128] f32;
 *   workspace of draft_topk_softmax_workspace(rows, V) bytes, 256-byte
 *   aligned (smaller or misaligned: SPEC_ERR_WORKSPACE).
 */
int draft_topk_softmax(const void *draft_logits, int dt, int rows, int V,
                       const int32_t *cu_rows, const float *temperature, int B,
                       int k, int32_t *out_idx, float *out_prob,
                       void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * RheoSampling dynamic-tree construction, one expansion level for B trees
 * ("RheoSampling 2026": §2 "Dual-Identity Decoupling", §3 "Parameter
 * Kendali Rheostat & Optimasi Sparse Top-128", §7 "Rekomendasi"). Every
 * frontier node f of tree b gets K children in slot order:
 *   - slots 0..m-1: the m best tokens of its draft row other than the probe
 *     (the deterministic lead);
 *   - slot m: the probe, a token drawn from q~ = softmax(z/T_b) over the
 *     row's 128 largest logits (ties to the lower id; T < 0.05: the argmax)
 *     by inverse CDF in ascending id at u(seed, b = f, pos = level,
 *     stream 3) as defined above;
 *   - slots m+1..K-1: the next best tokens other than the probe.
 * "Best" ranks by the logit, descending, ties to the lower id, among the
 * row's top 128; siblings are distinct. Ranking uses q = softmax(z) over
 * the same 128 logits, with no temperature (§7). q_proxy of a deterministic
 * child is its q; the probe's is q(x_{m+1}) + eps, x_j the row's j-th best
 * token (0 + eps when m+1 exceeds the survivors), which at m = 0 is the
 * page's q(x_1) + eps. score = frontier_score[f] + ln q_proxy. Each tree
 * then keeps the n_keep candidates with the largest scores (ties to the
 * lower candidate index f*K + slot), best first (§2, global pruning). The
 * children depend on the probe, so a verifier of the resulting trees should
 * test the probe first ("RheoSampling 2026", §4 step 1), then the
 * deterministic children as point masses.
 *
 *   draft          [F, V] draft logits (ddt), 16-byte aligned: row f is the
 *                  draft model's output at frontier node f.
 *   cu_frontier    [B+1] int32: tree b owns frontier rows cu_frontier[b] ..
 *                  cu_frontier[b+1]-1; cu_frontier[0] = 0,
 *                  cu_frontier[B] = F; at most SPEC_RHEO_MAX_CANDIDATES
 *                  candidates (rows x K) per tree.
 *   frontier_score [F] f32: ln of each frontier node's path score (0 at a
 *                  root), finite or -inf.
 *   temperature    [B] f32 >= 0, finite.
 *   K              children per frontier node, 1 <= K <= min(V, 128).
 *   m              rheostat, 0 <= m < K (the page recommends m = 1).
 *   eps            >= 0, finite: the probe's proxy margin.
 *   n_keep         candidates kept per tree, 0 .. SPEC_RHEO_MAX_CANDIDATES.
 *   level          0 <= level < 2^24, keys the probe draws of this level.
 *   child_token    [F, K] int32 out.   child_score [F, K] f32 out.
 *   child_qproxy   [F, K] f32 out, or NULL.
 *   child_qtrue    [F, K] f32 out, or NULL: q~ of each child's token (the
 *                  probe's true sampling probability in slot m).
 *   keep           [B, n_keep] int32 out: candidate ids f*K + slot, -1 when
 *                  a tree has fewer candidates. NULL only when n_keep == 0.
 *   workspace      >= spec_rheo_expand_workspace(F, V) bytes, 256-byte
 *                  aligned.
 * A device-side status (read with spec_get_status) reports bad offsets,
 * temperatures or scores (SPEC_ERR_INVALID_ARG) and trees over the
 * candidate limit (SPEC_ERR_UNSUPPORTED); outputs are then unspecified.
 */
#define SPEC_RHEO_MAX_CANDIDATES 8192
/*
 * Bytes of workspace spec_rheo_expand needs (0 on invalid sizes): a 256-byte
 * header, and for V % 8 == 0 with V >= 4096 the candidate lists of the
 * two-launch top-128 select (4 KB and 4 bytes per frontier row).
 */
size_t spec_rheo_expand_workspace(int F, int V);
int spec_rheo_expand(const void *draft, int ddt, const int32_t *cu_frontier,
                     const float *frontier_score, const float *temperature,
                     int B, int F, int V, int K, int m, float eps, int n_keep,
                     uint64_t seed, int level, int32_t *child_token,
                     float *child_qproxy, float *child_qtrue,
                     float *child_score, int32_t *keep, void *workspace,
                     size_t ws_bytes, spec_stream_t stream);

/*
 * Synchronises `stream` and reads the device status word that the last call
 * using `workspace` left: *device_status = SPEC_OK or a negative spec_status.
 * Returns SPEC_OK or SPEC_ERR_CUDA / SPEC_ERR_INVALID_ARG.
 */
int spec_get_status(const void *workspace, spec_stream_t stream,
                    int *device_status);

/*
 * The uniforms the verifier draws: out[i] = u(seed, b[i], pos[i], stream[i])
 * as defined above (device arrays of length n). For reproducing or auditing
 * a verification.
 */
int spec_uniforms(uint64_t seed, const int32_t *b, const int32_t *pos,
                  const int32_t *stream_id, int n, float *out,
                  spec_stream_t stream);

/*
 * Self-test of the bounds-checked build (libspecverify_checked.so, built
 * with SPEC_CHECKED; no counterpart on the pages: a test aid). That build
 * checks every global access of the kernels against the byte ranges of the
 * call's buffers (inputs, outputs, workspace), skips an access outside them
 * (a load gives 0, a store or copy is dropped) and reports it in the status
 * word as SPEC_ERR_BOUNDS, with the source line of the access as detail.
 * This call registers only the first 256 bytes of `workspace` (at least 512
 * bytes, 256-byte aligned, caller-owned) and reads the word after them, so
 * the status word then reads SPEC_ERR_BOUNDS; no memory outside the
 * workspace is touched. Calls that overlap on the device share the checked
 * build's range lists and must be ordered. The product library returns
 * SPEC_ERR_UNSUPPORTED.
 */
int spec_check_selftest(void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Self-test of the device-side bounded waits (failure detection without a
 * GPU fault). Launches one small kernel that waits, with the verifier
 * kernels' own waiting code, on something nothing completes: kind 0 a
 * shared-memory mbarrier phase (the waits of the TMA rings), kind 1 a global
 * word (the streaming verifier's producers). After limit_ns (1 ns .. 10 s)
 * of the GPU's global timer the wait gives up and the kernel records
 * SPEC_ERR_TIMEOUT in the status word of `workspace` (256 bytes, 256-byte
 * aligned) and returns; the context stays usable. Asynchronous on `stream`;
 * read the result with spec_get_status. Returns SPEC_ERR_INVALID_ARG for
 * another kind or limit, SPEC_ERR_WORKSPACE for a missing or misaligned
 * workspace.
 */
int spec_wait_selftest(int kind, unsigned long long limit_ns, void *workspace,
                       spec_stream_t stream);

/*
 * Profiling aid. Registers two CUDA events (cudaEvent_t, created by the
 * caller) for the next spec_verify_linear, spec_verify_tree,
 * draft_topk_softmax or spec_rheo_expand call made by the calling host
 * thread: that call records `before` immediately before it launches its
 * dominant kernel and `after` immediately after, on the call's stream, then
 * forgets them. Pass NULLs to clear. The dominant kernel is the
 * row-statistics pass of an eager linear call (it streams every vocabulary
 * row once), the top-128 select under SPEC_RULE_STRICT_TOP128 and in
 * draft_topk_softmax (for bf16 rows with V % 8 == 0 and V >= 4096, its scan
 * launch, which reads every row; the short finishing launch follows), the
 * streaming kernel of a position-lazy call (SPEC_EXT_LAZY) or,
 * on its multi-launch schedule, all its rounds (every row pass and every
 * per-round decision), the one kernel of a small call (fused or one cluster
 * per request), the cluster-resident kernel (SPEC_EXT_RESIDENT), the walk of
 * a tree call, and the top-128 select of spec_rheo_expand. So
 * cudaEventElapsedTime(before, after) is that kernel's duration.
 */
int spec_profile_row_pass(void *before, void *after);

/*
 * 1 while events registered with spec_profile_row_pass on the calling host
 * thread have not been taken by a call, else 0: after a call it tells whether
 * that call recorded them.
 */
int spec_profile_pending(void);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
