/*
 * sv.h -- C ABI of the GB300 (sm_103a) verify step of speculative decoding.
 *
 * One verify step = tree attention of the flattened candidate tree against the KV
 * prefix (sv_tree_attention), token acceptance over the vocabulary (sv_accept_chain /
 * sv_accept_tree) and the KV commit of the accepted path (sv_commit_kv); the fused
 * calls sv_accept_chain_commit / sv_accept_tree_commit do the last two in one launch
 * pair.  sv_accept_tree_recursive is the tree acceptance that tries a node's children
 * in turn (siblings drawn from q keep the target's distribution), sv_accept_tree_noalloc
 * the tree acceptance without a workspace, and sv_ngram_draft proposes prompt-lookup
 * drafts on the device; sv_lm_head is the LM-head projection on the tensor cores, and
 * sv_accept_chain_lmhead / sv_accept_tree_lmhead fuse it with the acceptance (the target
 * rows' statistics come from the projection's epilogue).
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is caller-owned DEVICE memory, dense row-major in the layout
 *    given next to it, 16-byte aligned.  The library never allocates device memory:
 *    scratch comes from a caller workspace sized by the matching *_workspace_size().
 *  - Trees: `parent` (BFS ordered: parent[0] = -1 and 0 <= parent[i] < i, at most
 *    SV_MAX_TREE_NODES nodes) with `parent_stride`.  parent_stride == 0: `parent` is a
 *    HOST array [N], one tree shared by every sequence of the batch (a static Medusa tree
 *    or a chain); it is validated and copied at the call, so the host array may be reused
 *    as soon as the call returns.  parent_stride >= N: `parent` is a DEVICE array
 *    [B, parent_stride] int32, row b the tree of sequence b (trees pruned or built per
 *    request, all with N rows); the kernels read and check it (a row that is not a
 *    BFS-ordered tree sets SV_DEV_BAD_TREE), so it must stay valid until the call's work
 *    on the stream is done.  With per-sequence trees the path and token outputs have N
 *    columns (the deepest possible path) instead of tree depth + 1.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only enqueue
 *    work and return without synchronising.  Each call that launches work opens an NVTX
 *    range named after it (e.g. "sv_accept_chain_commit") for the duration of the host
 *    call, so profiler timelines attribute the kernels to the call.
 *  - Arguments are validated on the host before anything is launched; a failed check
 *    returns SV_ERR_INVALID_ARG / SV_ERR_UNSUPPORTED / SV_ERR_WORKSPACE and launches
 *    nothing.  An empty batch (B = 0, or R = 0 rows for sv_lm_head) validates the other
 *    arguments and returns SV_OK without launching, reading any tensor or calling the
 *    CUDA runtime: its tensor pointers and workspace may be NULL.  A launch failure returns SV_ERR_CUDA.  sv_last_error() gives the
 *    message of the last failure in the calling thread.
 *  - Data-dependent problems found on the device (a token id outside [0,V), a block
 *    id outside the pool, a prefix longer than the cache, a draft with q(x) = 0) never
 *    trap: the kernel skips the offending access, ORs an SV_DEV_* bit into a sticky
 *    device status word and carries on.  Read (and clear) it with
 *    sv_read_device_status().
 *  - Near ties.  Every acceptance call can report, per sequence, the decisions and
 *    samples that lie so close to their threshold that another rounding of the same
 *    arithmetic could take them the other way (reported, not hidden).  out_near_ties[b]
 *    packs two counts: bits 0-15 count DECISION ties (a decision with |u_acc - ratio| <
 *    1e-6 whose parent lies on an accepted path, a top-p cut within 1e-6 of top_p, and
 *    for the sibling rule an empty residual handed to the next sibling: any of these may
 *    change which nodes are accepted), bits 16-31 count SAMPLE ties (the final token's
 *    u_smp * sum(w) within the window of a CDF boundary, or its residual empty: only the
 *    last emitted token is in doubt).  SV_NEAR_DECISIONS() / SV_NEAR_SAMPLES() unpack it.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t sv_status;
#define SV_OK 0
#define SV_ERR_INVALID_ARG 1 /* bad pointer, size, tree, temperature or top-k */
#define SV_ERR_UNSUPPORTED 2 /* valid, but not a compiled shape (dtype, head dim, N) */
#define SV_ERR_WORKSPACE 3   /* workspace missing or smaller than *_workspace_size() */
#define SV_ERR_CUDA 4        /* a CUDA call or kernel launch failed */

/* Bits of the device status word. */
#define SV_DEV_BAD_TOKEN 0x1u      /* a candidate token id outside [0, V) (rejected) */
#define SV_DEV_BAD_BLOCK 0x2u      /* a block-table entry outside the pool (skipped) */
#define SV_DEV_BAD_PREFIX 0x4u     /* prefix_len < 0 or beyond the cache (clamped) */
#define SV_DEV_ZERO_DRAFT_PROB 0x8u /* a draft with q(x) = 0: ratio taken as +inf/0 */
#define SV_DEV_TIMEOUT 0x10u       /* a pipeline wait gave up after its time limit; the
                                      outputs of that call are not valid */
#define SV_DEV_LAYOUT 0x20u        /* shared memory was not 1024-byte aligned; the call
                                      did nothing (outputs not valid) */
#define SV_DEV_BAD_TREE 0x40u      /* a per-sequence parent row is not a BFS-ordered tree
                                      (or, in exact acceptance, deeper than q's Dq rows):
                                      that sequence's outputs are not meaningful (its
                                      acceptance keeps the root alone) */

/* The two counts of a packed near-tie word (see "Near ties" above). */
#define SV_NEAR_DECISIONS(w) ((uint32_t)(w) & 0xFFFFu)
#define SV_NEAR_SAMPLES(w) ((uint32_t)(w) >> 16)

#define SV_MAX_TREE_NODES 64 /* one 64-bit ancestor word per node */
#define SV_MAX_TOP_K 1024

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;
typedef enum { SV_GREEDY = 0, SV_EXACT = 1 } sv_mode;
/* How the draft distribution q is given: as float32 probabilities used as they are,
 * or as draft logits (dtype of the target logits) to which the same temperature and
 * top-k are applied as to the target, or -- for deterministic drafts such as prompt-lookup
 * copies (jennyma11 blog, section "Prompt Lookup / N-gram": the copied tokens still go to
 * the target's verification) -- as a one-hot row at each draft token: q(x) = 1 for the
 * draft x and 0 elsewhere, so a draft is accepted iff u_acc < p(x) and the token after a
 * rejection comes from norm([p - e_x]+), p without x.  With SV_Q_DRAFT_ONEHOT no q rows
 * exist (the q pointer is not read and may be NULL); chains only. */
typedef enum { SV_Q_PROBS_F32 = 0, SV_Q_LOGITS = 1, SV_Q_DRAFT_ONEHOT = 2 } sv_q_kind;

/* The KV prefix cache of one attention layer.
 *  contiguous (block_table == NULL): k, v are [B, Lmax, Hkv, D]; sequence b's prefix
 *    occupies positions [0, prefix_len[b]).
 *  paged (block_table != NULL): k, v are a pool [num_blocks, block_size, Hkv, D];
 *    position p of sequence b lives in block block_table[b*max_blocks + p/block_size],
 *    row p % block_size.
 * prefix_len [B] is read by attention and updated in place by sv_commit_kv. */
typedef struct {
  void *k;
  void *v;
  int32_t *prefix_len;
  const int32_t *block_table;
  int32_t Lmax;
  int32_t block_size;
  int32_t max_blocks;
  int32_t num_blocks;
} sv_kv_cache;

/* ------------------------------------------------------------------ attention */

/* Tree attention (pages: "推测解码技术详解", section "Tree Attention验证" -- the flattened
 * candidate tree and its ancestor mask; lpnh.cn Medusa walkthrough section 3.2 -- a
 * node's context is its root path; qwbw.cn section 3.1.2 -- the prefix KV is reused
 * and only the candidates' KV is new).
 * For every sequence b, tree node n and query head h, with KV head g = h / (Hq/Hkv):
 *   keys  = prefix positions [0, prefix_len[b])  U  tree nodes j on n's root path,
 *   out   = softmax(scale * q . K^T) V over those keys.
 * q [B,N,Hq,D]; k_tree, v_tree [B,N,Hkv,D] (the candidates' fresh K/V, root = node 0);
 * cache as above (read only); parent, parent_stride as under "Trees" above; out
 * [B,N,Hq,D].
 * dt: SV_BF16 (fp32 accumulation, bf16 output) or SV_F32 (fp32 throughout).
 * Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= N <= 64; block_size % 16 == 0 for
 * paged caches.  Workspace: sv_tree_attention_workspace_size() bytes (may be 0).  The
 * workspace must be zero-filled before its first use with this function (it keeps a
 * generation counter and per-piece completion words that later calls rely on); each call
 * leaves it ready for the next, whatever the shape, including after a call that reported
 * SV_DEV_TIMEOUT.  Calls sharing one workspace must be stream-ordered. */
sv_status sv_tree_attention(sv_dtype dt, int B, int N, int Hq, int Hkv, int D, const void *q,
                            const void *k_tree, const void *v_tree, sv_kv_cache cache,
                            const int32_t *parent, int parent_stride, float scale, void *out,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Which kernel sv_tree_attention runs for these sizes: 1 = the tensor-core kernel
 * (tcgen05 MMA into TMEM, TMA-fed), 0 = the general kernel (mma.sync for bf16, FFMA for
 * f32), -1 = sizes it rejects.  block_size: the paged cache's block size, 0 for a
 * contiguous cache.  Host only; no device work. */
int sv_tree_attention_path(sv_dtype dt, int N, int Hq, int Hkv, int D, int block_size);

/* Workspace bytes sv_tree_attention needs for these sizes; max_prefix is the largest
 * prefix the cache can hold (Lmax, or max_blocks*block_size when paged). */
size_t sv_tree_attention_workspace_size(sv_dtype dt, int B, int N, int Hq, int Hkv, int D,
                                        int max_prefix);

/* ----------------------------------------------------------------- acceptance */

/* Chain acceptance (hncyxsy.com sections 2.1-2.2; jennyma11 blog "先弄清无损验证"):
 * draft i (1..gamma) is accepted with probability min(1, p_{i-1}(x_i)/q_i(x_i)) using
 * u_acc(b, i); at the first rejection the next token is sampled from
 * norm([p_{i-1} - q_i]+), if all pass the bonus is sampled from p_gamma, both with
 * u_smp(b, node) by inverse CDF in ascending token order.  p and q are the effective
 * distributions: logits / temperature, top-k (ties keep lower ids), softmax.  Greedy
 * (or temperature == 0): accept while x_i == argmax row i-1 (lowest id on ties) and
 * emit that row's argmax.
 * Uniforms: Philox4x32-10 with key (seed_lo, seed_hi) and counter (node, b, round_lo,
 * round_hi); u_acc = word0, u_smp = word1, u = ((w >> 8) + 0.5) * 2^-24.
 * target_logits [B,gamma+1,V] (row i = target distribution after node i); q
 * [B,gamma,V] (row i-1 = draft distribution of draft i; unused in greedy mode and with
 * SV_Q_DRAFT_ONEHOT, may then be NULL); draft_tokens [B,gamma] int32.  A draft token of
 * -1 ends that sequence's chain: a sequence with k < gamma drafts has -1 from position k
 * on (what sv_ngram_draft writes), and when its k drafts are all accepted the bonus is
 * drawn from row k.  (Tokens after the first -1 are not decided; values outside [0, V)
 * other than -1 are bad tokens.)
 * Outputs: out_tokens [B,gamma+1] (accepted drafts then the sampled token, -1 after),
 * out_num_emitted [B] (= accepted + 1), out_num_accepted [B], out_near_ties [B] (the
 * packed near-tie word: decisions with |u_acc - ratio| < 1e-6 and near top-p cuts in
 * bits 0-15, a final sample within 1e-6 (probability units) of a CDF boundary or with
 * an empty residual in bits 16-31; may be NULL).
 * logit_dt: SV_BF16 or SV_F32.  V % 8 == 0, 1 <= gamma <= 63, 0 <= top_k <= 1024
 * (0 = off).  top_p in (0, 1], 1 = off: below 1 the nucleus of the top-k distribution
 * is kept (top-k first, then top-p; needs 0 < top_k < V, else SV_ERR_UNSUPPORTED): in the
 * top-k ranking an entry stays while the mass ranked above it is below top_p, and p is
 * renormalised over the kept entries; a cut whose mass lies within 1e-6 of top_p counts
 * as one near tie of the sequence (the lpnh.cn walkthrough, section 4.2, and the
 * jennyma11 blog name top-p among the sampling settings the effective distributions
 * carry).  Ignored in greedy mode.
 * Workspace: sv_accept_workspace_size(B, gamma+1, V, gamma). */
sv_status sv_accept_chain(sv_mode mode, sv_dtype logit_dt, int B, int gamma, int V,
                          const void *target_logits, const void *q, sv_q_kind q_kind,
                          const int32_t *draft_tokens, float temperature, int top_k, float top_p,
                          uint64_t seed, uint64_t round, int32_t *out_tokens,
                          int32_t *out_num_emitted, int32_t *out_num_accepted,
                          uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                          void *stream);

/* Tree acceptance (qwbw.cn section 2.3 -- keep the longest correct path; jennyma11
 * blog section "Medusa" -- only the contiguous accepted prefix from the root is
 * committed).  Every non-root node c (parent a, depth d) is decided independently:
 * accept iff u_acc(b, c) < p_a(x_c) / q_d(x_c) (greedy: x_c == argmax p_a).  The chosen
 * node a* is the deepest node whose whole root path is accepted (ties: smallest row).
 * The emitted tokens are those of the path nodes 1..a*, then a token sampled with
 * u_smp(b, a*) from norm([p_{a*} - q_{d(a*)+1}]+) if a* has children, else from p_{a*}.
 * parent, parent_stride as under "Trees" above (per-sequence trees: a node deeper than
 * Dq sets SV_DEV_BAD_TREE in exact mode); node_tokens [B,N] (column 0, the root, is not
 * read);
 * target_logits [B,N,V]; q [B,Dq,V] with row d-1 = depth d (Dq >= tree depth); q_kind
 * SV_Q_PROBS_F32 or SV_Q_LOGITS (SV_Q_DRAFT_ONEHOT: SV_ERR_UNSUPPORTED in exact mode).
 * temperature, top_k, top_p, the uniforms and the near-tie reports as sv_accept_chain.
 * Outputs (W = tree depth + 1; N with per-sequence trees): out_path_nodes [B,W] (root..a*,
 * -1 after), out_tokens [B,W], out_num_emitted [B], out_num_accepted [B], out_near_ties [B].
 * Workspace: sv_accept_workspace_size(B, N, V, Dq). */
sv_status sv_accept_tree(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                         const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                         const void *target_logits, const void *q, sv_q_kind q_kind, int Dq,
                         float temperature, int top_k, float top_p, uint64_t seed, uint64_t round,
                         int32_t *out_path_nodes, int32_t *out_tokens,
                         int32_t *out_num_emitted, int32_t *out_num_accepted,
                         uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Exact tree acceptance with the siblings of a node tried in turn (hncyxsy.com sections
 * 2.1-2.2: after a rejected candidate the target becomes the residual norm([p - q]+);
 * jennyma11 blog, section "Medusa": lossless tree verification).  From the root, the
 * children of the current node are tried in row order: child c (token x_c) is accepted iff
 * u_acc(b, c) < r(x_c) / q_{d+1}(x_c), where r starts as the node's effective target p and
 * after each rejected child becomes norm([r - q_{d+1}]+) (kept unchanged, and counted as a
 * near tie, when that has no mass); an accepted child becomes the current node.  When all
 * children are rejected the token is drawn with u_smp(b, node) from norm([r - q_{d+1}]+)
 * of the last r (r itself when that has no mass); a leaf draws the bonus from its p.  With
 * drafts drawn independently from q this keeps the emitted tokens distributed as the
 * target's; with one child per node it equals sv_accept_chain.
 * Exact mode only: temperature must be > 0 (else SV_ERR_UNSUPPORTED; greedy trees use
 * sv_accept_tree).  Every other argument, the outputs, the uniforms, the workspace
 * (sv_accept_workspace_size(B, N, V, Dq)) and the errors as sv_accept_tree; the packed
 * near-tie word counts, as decision ties, decisions with |u_acc - ratio| within 1e-6 (or
 * within the float error bound of the residual's mass, when that is wider), residuals
 * handed to a sibling with no mass (or less than that error bound) and one near top-p
 * cut on a visited row; and as sample ties a final sample within 1e-6 of a CDF boundary
 * (in units of the normalised residual, or the error bound when wider) or with an empty
 * residual.  Launches: the statistics kernel, then one thread-block cluster of up to 16
 * CTAs per sequence (each on a slice of the vocabulary). */
sv_status sv_accept_tree_recursive(sv_dtype logit_dt, int B, int N, int V, const int32_t *parent,
                                   int parent_stride,
                                   const int32_t *node_tokens, const void *target_logits,
                                   const void *q, sv_q_kind q_kind, int Dq, float temperature,
                                   int top_k, float top_p, uint64_t seed, uint64_t round,
                                   int32_t *out_path_nodes, int32_t *out_tokens,
                                   int32_t *out_num_emitted, int32_t *out_num_accepted,
                                   uint32_t *out_near_ties, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Typical acceptance (named beside lossless verification by the jennyma11 blog, section
 * "Medusa", without a rule; the rule is the Medusa paper's -- T. Cai et al., "Medusa: Simple
 * LLM Inference Acceleration Framework with Multiple Decoding Heads", 2024, section
 * "Typical Acceptance"): node c (parent a) is accepted iff
 *   p_a(x_c) > min(epsilon, delta * exp(-H(p_a))),
 * p_a the parent's target distribution at the given temperature (> 0; no top-k), H its
 * entropy in nats.  No draft distribution and no uniforms: it is not distribution
 * preserving, it trades exactness for longer accepted runs.  The kept node a* is the
 * deepest one whose whole root path is accepted (ties: smallest row); the emitted tokens are
 * those of path nodes 1..a*, then the target's most likely token at a* (argmax, lowest id),
 * so every call emits at least one token.  Trees, node_tokens, target_logits, the outputs
 * and the near-tie word as sv_accept_tree (decision ties: |p_a(x_c) - threshold| < 1e-6 on
 * an accepted path).  Workspace: sv_accept_workspace_size(B, N, V, 0). */
sv_status sv_accept_typical(sv_dtype logit_dt, int B, int N, int V, const int32_t *parent,
                           int parent_stride, const int32_t *node_tokens,
                           const void *target_logits, float temperature, float epsilon,
                           float delta, int32_t *out_path_nodes, int32_t *out_tokens,
                           int32_t *out_num_emitted, int32_t *out_num_accepted,
                           uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Workspace bytes for sv_accept_chain (N = gamma+1, Dq = gamma) / sv_accept_tree. */
size_t sv_accept_workspace_size(int B, int N, int V, int Dq);

/* sv_accept_tree without a workspace argument, for callers that cannot allocate device
 * memory (no cudaMalloc or allocating library call on their path: fixed-memory
 * embedded runtimes, callers holding no allocator handle).  No counterpart on the
 * pages: it is a deployment convenience.  Arguments, outputs and results are those of
 * sv_accept_tree; the per-row statistics go to a fixed device array inside the library
 * of SV_NOALLOC_ACCEPT_ROWS rows (32 bytes each, 2 MiB), held by every GPU that
 * loads the library until the process exits.  B*(N+Dq) logit rows (B*N in greedy
 * mode) must not exceed SV_NOALLOC_ACCEPT_ROWS, else SV_ERR_UNSUPPORTED and nothing is
 * launched.  The first call on a device looks the array's address up on that device
 * (make that first call before any stream capture).  Every call shares the one array,
 * so calls that overlap on the GPU (other streams, other threads) race on it: order
 * them on one stream.  Each call writes every statistic it reads, so nothing needs
 * clearing between calls. */
#define SV_NOALLOC_ACCEPT_ROWS 65536
sv_status sv_accept_tree_noalloc(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                                 const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                                 const void *target_logits, const void *q, sv_q_kind q_kind,
                                 int Dq, float temperature, int top_k, float top_p, uint64_t seed,
                                 uint64_t round, int32_t *out_path_nodes, int32_t *out_tokens,
                                 int32_t *out_num_emitted, int32_t *out_num_accepted,
                                 uint32_t *out_near_ties, void *stream);

/* --------------------------------------------------------------- n-gram drafts */

/* Prompt-lookup (n-gram) drafting ("投机解码的五条路线" (jennyma11 blog), section "Prompt
 * Lookup / N-gram"): take the last n tokens of a sequence's history, find the same n
 * tokens earlier in it, and propose the tokens that follow that occurrence; the drafts
 * still go to the target's verification (sv_accept_chain) like any other.  For n from
 * max_ngram down to min_ngram the first n with a match wins; among its matches the most
 * recent (largest start) is taken; a match must end before the last token; up to gamma
 * tokens follow it (fewer when the history ends).
 * history [B,Lmax] int32 (device); length [B] int32 (device; a value outside [0, Lmax]
 * is clamped and sets SV_DEV_BAD_PREFIX).  1 <= min_ngram <= max_ngram <= SV_MAX_NGRAM,
 * 1 <= gamma <= 63.  Outputs: out_drafts [B,gamma] (-1 after the proposed tokens) and
 * out_num_drafts [B] (0 when nothing matches).  No workspace. */
#define SV_MAX_NGRAM 32
sv_status sv_ngram_draft(int B, int Lmax, const int32_t *history, const int32_t *length,
                         int max_ngram, int min_ngram, int gamma, int32_t *out_drafts,
                         int32_t *out_num_drafts, void *stream);

/* --------------------------------------------------------------------- commit */

/* KV commit (qwbw.cn sections 3.1.4 and 6.3; hncyxsy.com section 4.3: keep the KV of
 * accepted tokens, roll the rest back by the valid length).  For each sequence b the
 * tree K/V rows of path_nodes[b, 0..num_accepted[b]] (root first, depth order) are
 * copied to cache positions prefix_len[b] + i, then prefix_len[b] += num_accepted[b]+1.
 * Rejected rows are simply not copied; nothing is freed (the caller owns the pages,
 * which must already cover the new positions).
 * k_tree, v_tree [B,N,Hkv,D]; path_nodes [B,path_stride] int32; num_accepted [B].
 * dt: element type of the K/V rows (SV_BF16 or SV_F32). */
sv_status sv_commit_kv(sv_dtype dt, int B, int N, int Hkv, int D, const void *k_tree,
                       const void *v_tree, const int32_t *path_nodes, int path_stride,
                       const int32_t *num_accepted, sv_kv_cache cache, void *stream);

/* Acceptance and the KV commit of its kept path in one call: the same results as
 * sv_accept_tree (resp. sv_accept_chain) followed by sv_commit_kv with path_nodes =
 * out_path_nodes (resp. nodes 0..accepted), path_stride = tree depth + 1 and
 * num_accepted = out_num_accepted (qwbw.cn sections 3.1.4 and 6.3 for the commit).
 * The commit runs inside the acceptance's second kernel, split over the CTAs that
 * already hold the sequence, so it costs no launch of its own.  kv_dt, Hkv, D, k_tree,
 * v_tree and cache are the sv_commit_kv arguments (same layout, ownership and
 * checks); the acceptance arguments, outputs and workspace are those of the separate
 * call.  prefix_len[b] is read before any K/V is written and advanced once, after. */
sv_status sv_accept_tree_commit(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                                const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                                const void *target_logits, const void *q, sv_q_kind q_kind,
                                int Dq, float temperature, int top_k, float top_p, uint64_t seed,
                                uint64_t round, sv_dtype kv_dt, int Hkv, int D,
                                const void *k_tree, const void *v_tree, sv_kv_cache cache,
                                int32_t *out_path_nodes, int32_t *out_tokens,
                                int32_t *out_num_emitted, int32_t *out_num_accepted,
                                uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                                void *stream);
sv_status sv_accept_chain_commit(sv_mode mode, sv_dtype logit_dt, int B, int gamma, int V,
                                 const void *target_logits, const void *q, sv_q_kind q_kind,
                                 const int32_t *draft_tokens, float temperature, int top_k, float top_p,
                                 uint64_t seed, uint64_t round, sv_dtype kv_dt, int Hkv, int D,
                                 const void *k_tree, const void *v_tree, sv_kv_cache cache,
                                 int32_t *out_tokens, int32_t *out_num_emitted,
                                 int32_t *out_num_accepted, uint32_t *out_near_ties,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------ LM head */

/* The LM-head projection ("推测解码技术详解", section "Medusa Heads": the original LM head
 * and the Medusa heads read the backbone's last hidden states; lpnh.cn walkthrough,
 * section 3.1: a head is a Linear(H, V) from h_t to V logits): logits[r, v] =
 * sum_k hidden[r, k] * weight[v, k] with fp32 accumulation on the tensor cores, stored in
 * bf16.  hidden [R, Dm] bf16, weight [V, Dm] bf16 (row v = token v's output embedding; no
 * bias), logits [R, V] bf16 (written).  Dm and V positive multiples of 8.  No workspace. */
sv_status sv_lm_head(int R, int Dm, int V, const void *hidden, const void *weight, void *logits,
                     void *stream);

/* Acceptance fused with the LM-head projection of the target rows: the projection above
 * computes the target logits from the hidden states (stored in target_logits, which the
 * final sample reads) and, without top-k, its epilogue also takes each row's statistics
 * (max, argmax, softmax sum at the given temperature), so the logits are not read back for
 * them; with top-k the statistics kernel reads the stored rows.  Then the acceptance of
 * sv_accept_chain / sv_accept_tree runs on the stored bf16 logits: every argument, output,
 * uniform and near-tie report as there, with logit_dt = SV_BF16.
 * hidden [B, gamma+1, Dm] (chain) or [B, N, Dm] (tree) bf16, row order of the target rows;
 * weight [V, Dm] bf16; target_logits [B, gamma+1 or N, V] bf16 (written).
 * Workspace: sv_accept_lmhead_workspace_size(B, N, V, Dq) (N = gamma+1, Dq = gamma for a
 * chain). */
size_t sv_accept_lmhead_workspace_size(int B, int N, int V, int Dq);
sv_status sv_accept_chain_lmhead(sv_mode mode, int B, int gamma, int V, int Dm, const void *hidden,
                                 const void *weight, void *target_logits, const void *q,
                                 sv_q_kind q_kind, const int32_t *draft_tokens, float temperature,
                                 int top_k, float top_p, uint64_t seed, uint64_t round,
                                 int32_t *out_tokens, int32_t *out_num_emitted,
                                 int32_t *out_num_accepted, uint32_t *out_near_ties,
                                 void *workspace, size_t workspace_bytes, void *stream);
sv_status sv_accept_tree_lmhead(sv_mode mode, int B, int N, int V, int Dm, const void *hidden,
                                const void *weight, void *target_logits, const int32_t *parent,
                                int parent_stride, const int32_t *node_tokens, const void *q,
                                sv_q_kind q_kind, int Dq, float temperature, int top_k,
                                float top_p, uint64_t seed, uint64_t round,
                                int32_t *out_path_nodes, int32_t *out_tokens,
                                int32_t *out_num_emitted, int32_t *out_num_accepted,
                                uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                                void *stream);

/* ---------------------------------------------------------------- tree helper */

/* Host helper: validate a tree and derive per node its ancestor bitmask (bit j set
 * iff j is the node or one of its ancestors -- the rows of the tree-attention mask)
 * and its depth; position id of node n = prefix_len + depth[n].  anc/depth may be
 * NULL.  Returns SV_ERR_INVALID_ARG for an invalid tree. */
sv_status sv_tree_prepare(int N, const int32_t *parent, uint64_t *anc, int32_t *depth);

/* ---------------------------------------------------------- status and errors */

/* Copy the sticky device status word (SV_DEV_* bits) to *host_out and clear it.
 * Synchronises `stream`. */
sv_status sv_read_device_status(uint32_t *host_out, void *stream);

/* Message of the last failed call in this thread ("" if none). */
const char *sv_last_error(void);

/* Library version string. */
const char *sv_version(void);

/* Number of CUDA kernels this library has launched in this process so far (all calls,
 * all threads); the difference around a region counts the region's launches. */
uint64_t sv_kernel_launches(void);

/* The time after which a wait for progress inside the tensor-core attention kernel gives
 * up (a copy, an MMA, or another CTA's piece of a split unit that does not arrive): the
 * kernel then lets its copies and MMAs in flight land, frees its tensor memory, sets
 * SV_DEV_TIMEOUT and returns; the workspace stays usable for the next call.  Default 2 s;
 * 0 restores it.  Process-wide, read at each sv_tree_attention call.  A limit shorter
 * than the kernel's normal waits makes the calls fail with SV_DEV_TIMEOUT: it exists to
 * exercise that path. */
void sv_set_wait_limit_ns(uint64_t ns);
uint64_t sv_get_wait_limit_ns(void);

/* Failure injection on the host, for tests of a caller's error handling: the next n kernel
 * launch requests of the library (process-wide, each entry point's launches counted in
 * order) report a launch failure instead of launching -- the call returns SV_ERR_CUDA with
 * its message in sv_last_error(), and neither that launch nor any later one of the same
 * call is enqueued (a call stops at its first failed launch).  No kernel runs and no GPU
 * state changes.  n <= 0 clears the count. */
void sv_inject_launch_failures(int n);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
