/*
 * oracle.c -- plain, slow, double-precision CPU oracle for the speculative-decoding
 * verify step (tree attention, token acceptance, KV commit).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference legs may load this library.  It shares no code, header,
 * table or helper with the CUDA path and must never be used as a fallback for it.
 *
 * Sources (web pages on speculative decoding; cited by page title and section):
 *  - "推测解码技术详解：加速LLM推理的关键", section "Tree Attention验证": a candidate tree
 *    is flattened into rows; a node attends to itself and its ancestors only (7-node
 *    example with its printed mask).
 *  - lpnh.cn Medusa walkthrough, section 3.2: a tree node's context is its root path.
 *  - hncyxsy.com article, sections 2.1-2.2: accept a draft x with probability
 *    min(1, p(x)/q(x)); on rejection resample from norm(max(0, p-q)) and drop the rest;
 *    if all gamma drafts pass, sample one bonus token from the target's next position.
 *  - "投机解码的五条路线" (jennyma11 blog), section "先弄清无损验证": p and q are the
 *    effective sampling distributions (temperature, top-k applied); greedy checks the
 *    candidates against the target's per-position best token.  Section
 *    "怎么选,以及怎么算收益": expected emitted tokens sum_{k=0..gamma} alpha^k.
 *  - qwbw.cn article, section 2.3: choose the longest accepted path of the tree;
 *    sections 3.1.4 / 6.3: keep the KV of accepted tokens, drop the rest.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *    1, 2, 3", SC'11 (the published counter-based generator).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - tree acceptance: every non-root node c is decided independently against its
 *    parent's p and the q of its depth; the chosen node is the deepest one whose whole
 *    root path is accepted (ties: smallest row index); the final token is sampled
 *    from norm([p_a - q_{d+1}]+) if that node has children, else the bonus from p_a.
 *  - tree acceptance with siblings tried in turn (orc_accept_tree_recursive): the
 *    children of the current node in row order; after a rejected child the target
 *    becomes norm([r - q]+) (kept, as a near tie, when that has no mass); after the
 *    last rejection the token is drawn from norm([r - q]+) of the last r.
 *  - LM head (orc_lm_head): z = h W^T with no bias, h already normalised; the result is
 *    read by the acceptance functions as double logits (dtype ORC_F64).
 *  - top-k ties at the k-th value keep the lower token ids; argmax ties pick the
 *    lowest token id; temperature T == 0 means greedy.
 *  - top-p (nucleus; named as a sampling knob by the jennyma11 blog, section
 *    "先弄清无损验证", and the lpnh.cn walkthrough, section 4.2): applied within the
 *    top-k distribution (top-k first, then top-p; top_p < 1 needs 0 < top_k < V).  In
 *    the top-k ranking an entry stays while the mass ranked above it is below top_p,
 *    then p is renormalised over the kept entries; a cut within 1e-6 of top_p counts as
 *    one near tie of the sequence.
 *  - uniforms: counter (node, seq, round_lo, round_hi ^ domain), key (seed_lo, seed_hi);
 *    u_acc from word 0 and u_smp from word 1, u = ((w >> 8) + 0.5) * 2^-24.
 *  - inverse CDF in ascending token order: smallest j with C_j > u * sum(w).
 *  - near ties (reported, not hidden): |u_acc - ratio| < 1e-6 for a decision that
 *    matters (its parent lies on an accepted path), or u*sum(w) within 1e-6 of a CDF
 *    boundary around the chosen token (w is in probability units: p and q are
 *    normalised, so the window is absolute), or sum(w) == 0 (then sample from p).
 *    The count is reported in two classes packed in one word: decision ties (a near
 *    decision, a near top-p cut, and for the sibling rule an empty residual handed to
 *    the next sibling: anything that can change which nodes are accepted) in the low 16
 *    bits, and sample ties (a near CDF boundary or an empty residual in the final
 *    sample: only the last emitted token is in doubt) times 65536 in the high 16 bits.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -o liboracle.so oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2
#define ORC_GREEDY 0
#define ORC_EXACT 1
#define ORC_Q_PROBS_F32 0
#define ORC_Q_LOGITS 1
#define ORC_Q_DRAFT_ONEHOT 2 /* deterministic drafts: q = e_x at each draft token x */
#define ORC_NEAR_TIE 1e-6
/* weight of one sample-class near tie in the packed near-tie word */
#define ORC_SAMPLE_TIE 65536u

/* Host memory for scratch; a failed allocation stops the process with a message. */
static void *orc_alloc(size_t n) {
  void *p = malloc(n > 0 ? n : 1);
  if (!p) {
    fprintf(stderr, "oracle: out of host memory (%zu bytes)\n", n);
    abort();
  }
  return p;
}

/* ------------------------------------------------------------------ threads */

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* --------------------------------------------------------- element loading */

/* Widen one stored element to double.  bf16 is the upper half of an IEEE binary32
 * word, so shifting its 16 bits up gives the same value exactly. */
static double orc_elem(const void *base, int dtype, size_t i) {
  if (dtype == ORC_F64) return ((const double *)base)[i];
  if (dtype == ORC_F32) return (double)((const float *)base)[i];
  uint32_t w = ((uint32_t)((const uint16_t *)base)[i]) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static size_t orc_esize(int dtype) { return dtype == ORC_F64 ? 8 : dtype == ORC_F32 ? 4 : 2; }

/* --------------------------------------------------------- Philox4x32-10 */

/* Philox4x32 with 10 rounds (Salmon et al., SC'11): each round multiplies words 0
 * and 2 by the two Philox multipliers, mixes the high halves with words 1 and 3 and
 * the key, and the key is bumped by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t m0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t m1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(m0 >> 32), lo0 = (uint32_t)m0;
    uint32_t hi1 = (uint32_t)(m1 >> 32), lo1 = (uint32_t)m1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static double orc_word_to_uniform(uint32_t w) {
  return ((double)(w >> 8) + 0.5) * (1.0 / 16777216.0);
}

/* The two uniforms of (sequence b, node c) in one verify round. */
void orc_uniforms(uint64_t seed, uint64_t round, uint32_t domain, int b, int c,
                  double *u_acc, double *u_smp) {
  uint32_t ctr[4] = {(uint32_t)c, (uint32_t)b, (uint32_t)round,
                     (uint32_t)(round >> 32) ^ domain};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t x[4];
  orc_philox4x32_10(ctr, key, x);
  *u_acc = orc_word_to_uniform(x[0]);
  *u_smp = orc_word_to_uniform(x[1]);
}

/* ----------------------------------------------------------------- trees */

/* Is node j the node n itself or one of its ancestors?  Walk n's parent chain. */
static int orc_on_root_path(const int32_t *parent, int n, int j) {
  for (int a = n; a >= 0; a = parent[a])
    if (a == j) return 1;
  return 0;
}

static int orc_depth(const int32_t *parent, int n) {
  int d = 0;
  for (int a = parent[n]; a >= 0; a = parent[a]) ++d;
  return d;
}

/* 0 if parent[] is a valid BFS-ordered tree: parent[0] = -1 and 0 <= parent[i] < i. */
int orc_check_tree(int N, const int32_t *parent) {
  if (N < 1 || parent[0] != -1) return 1;
  for (int i = 1; i < N; ++i)
    if (parent[i] < 0 || parent[i] >= i) return 1;
  return 0;
}

/* Mask rows of the flattened tree, one row per node: mask[n*N + j] = 1 iff node j is
 * on the root path of node n (the tree-attention mask of the 7-node example). */
void orc_tree_mask(int N, const int32_t *parent, uint8_t *mask) {
  for (int n = 0; n < N; ++n)
    for (int j = 0; j < N; ++j) mask[(size_t)n * N + j] = (uint8_t)orc_on_root_path(parent, n, j);
}

/* ------------------------------------------------------------- attention */

/* Row index of prefix position pos of sequence b in the K/V cache. */
static size_t orc_cache_row(int b, int pos, const int32_t *block_table, int max_blocks,
                            int block_size, int Lmax) {
  if (block_table == NULL) return (size_t)b * Lmax + pos;
  int blk = block_table[(size_t)b * max_blocks + pos / block_size];
  return (size_t)blk * block_size + pos % block_size;
}

/* Tree attention by its definition.  For every sequence b in [b_begin, b_end), node n
 * and query head h (KV head g = h / (Hq/Hkv)):
 *   keys = prefix positions 0..L_b-1 of the cache  U  tree nodes on n's root path,
 *   s_j  = scale * <q, k_j>,  o = sum_j softmax(s)_j v_j.
 * q [B,N,Hq,D]; k_tree, v_tree [B,N,Hkv,D]; cache [B,Lmax,Hkv,D] (block_table NULL)
 * or [num_blocks,block_size,Hkv,D]; out [(b_end-b_begin),N,Hq,D] in double.  The tree of
 * sequence b is parent[b * parent_stride .. + N): parent_stride 0 shares one tree. */
void orc_tree_attention(int dtype, int B, int N, int Hq, int Hkv, int D, const void *q,
                        const void *k_tree, const void *v_tree, const void *cache_k,
                        const void *cache_v, const int32_t *prefix_len,
                        const int32_t *block_table, int max_blocks, int block_size, int Lmax,
                        const int32_t *parent, int parent_stride, double scale, int b_begin,
                        int b_end, double *out) {
  (void)B;
  int G = Hq / Hkv;
  int rows = (b_end - b_begin) * N * Hq;
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < rows; ++r) {
    int h = r % Hq;
    int n = (r / Hq) % N;
    int b = b_begin + r / (Hq * N);
    int g = h / G;
    int L = prefix_len[b];
    int nk = L + N;
    const int32_t *par = parent + (size_t)b * parent_stride; /* this sequence's tree */
    double *s = (double *)orc_alloc(sizeof(double) * (size_t)nk);
    size_t qoff = (((size_t)b * N + n) * Hq + h) * D;
    double smax = -INFINITY;
    for (int j = 0; j < nk; ++j) {
      s[j] = -INFINITY;
      size_t koff;
      const void *kb;
      if (j < L) {
        koff = (orc_cache_row(b, j, block_table, max_blocks, block_size, Lmax) * Hkv + g) * D;
        kb = cache_k;
      } else {
        int t = j - L;
        if (!orc_on_root_path(par, n, t)) continue;
        koff = (((size_t)b * N + t) * Hkv + g) * D;
        kb = k_tree;
      }
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += orc_elem(q, dtype, qoff + d) * orc_elem(kb, dtype, koff + d);
      s[j] = scale * dot;
      if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    for (int j = 0; j < nk; ++j) {
      s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - smax);
      denom += s[j];
    }
    double *o = out + (((size_t)(b - b_begin) * N + n) * Hq + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = 0; j < nk; ++j) {
      if (s[j] == 0.0) continue;
      size_t voff;
      const void *vb;
      if (j < L) {
        voff = (orc_cache_row(b, j, block_table, max_blocks, block_size, Lmax) * Hkv + g) * D;
        vb = cache_v;
      } else {
        voff = (((size_t)b * N + (j - L)) * Hkv + g) * D;
        vb = v_tree;
      }
      double w = s[j] / denom;
      for (int d = 0; d < D; ++d) o[d] += w * orc_elem(vb, dtype, voff + d);
    }
    free(s);
  }
}

/* ------------------------------------------------- sampling distributions */

typedef struct {
  double value;
  int index;
} orc_ranked;

/* Order: larger value first; equal values -> lower index first. */
static int orc_cmp_desc_value_asc_index(const void *pa, const void *pb) {
  const orc_ranked *a = (const orc_ranked *)pa, *b = (const orc_ranked *)pb;
  if (a->value > b->value) return -1;
  if (a->value < b->value) return 1;
  return (a->index > b->index) - (a->index < b->index);
}

/* Lowest index of the largest entry. */
static int orc_argmax(const double *z, int V) {
  int best = 0;
  for (int j = 1; j < V; ++j)
    if (z[j] > z[best]) best = j;
  return best;
}

/* Effective sampling distribution of one logit row: y = z / T, keep the top_k
 * largest y (if 0 < top_k < V; ties keep lower ids), p = softmax over the kept set.
 * With top_p < 1 (only together with top-k), the nucleus of that distribution is kept
 * instead: in the same ranking, an entry stays while the mass ranked above it is below
 * top_p (the smallest set with mass >= top_p; the first entry always stays), and p is
 * renormalised over it.  A cut whose mass lies within 1e-6 of top_p on either side sets
 * *near (if near is not NULL). */
static void orc_effective_dist(const double *z, int V, double T, int top_k, double top_p,
                               double *p, int *near) {
  double *y = (double *)orc_alloc(sizeof(double) * (size_t)V);
  unsigned char *keep = (unsigned char *)orc_alloc((size_t)V);
  orc_ranked *r = NULL;
  for (int j = 0; j < V; ++j) {
    y[j] = z[j] / T;
    keep[j] = 1;
  }
  if (top_k > 0 && top_k < V) {
    r = (orc_ranked *)orc_alloc(sizeof(orc_ranked) * (size_t)V);
    for (int j = 0; j < V; ++j) {
      r[j].value = y[j];
      r[j].index = j;
    }
    qsort(r, (size_t)V, sizeof(orc_ranked), orc_cmp_desc_value_asc_index);
    memset(keep, 0, (size_t)V);
    for (int i = 0; i < top_k; ++i) keep[r[i].index] = 1;
  }
  double ymax = -INFINITY;
  for (int j = 0; j < V; ++j)
    if (keep[j] && y[j] > ymax) ymax = y[j];
  double sum = 0.0;
  for (int j = 0; j < V; ++j) {
    p[j] = keep[j] ? exp(y[j] - ymax) : 0.0;
    sum += p[j];
  }
  for (int j = 0; j < V; ++j) p[j] /= sum;
  if (r != NULL && top_p < 1.0) {
    double c = 0.0;
    int m = top_k - 1;
    for (int i = 0; i < top_k; ++i) {
      double before = c;
      c += p[r[i].index];
      if (c >= top_p) {
        m = i;
        if (near && (c - top_p < ORC_NEAR_TIE || (i > 0 && top_p - before < ORC_NEAR_TIE)))
          *near = 1;
        break;
      }
    }
    double kept = 0.0;
    for (int i = 0; i <= m; ++i) kept += p[r[i].index];
    for (int i = m + 1; i < top_k; ++i) p[r[i].index] = 0.0;
    for (int i = 0; i <= m; ++i) p[r[i].index] /= kept;
  }
  free(r);
  free(y);
  free(keep);
}

static void orc_load_row(const void *base, int dtype, size_t row, int V, double *z) {
  for (int j = 0; j < V; ++j) z[j] = orc_elem(base, dtype, row * (size_t)V + j);
}

/* Inverse CDF in ascending token order: smallest j with C_j > u * sum(w).  Returns
 * the token; *near is set when u*sum(w) lies within 1e-6 of C_{j-1} or C_j. */
static int orc_inverse_cdf(const double *w, int V, double u, int *near) {
  double total = 0.0;
  for (int j = 0; j < V; ++j) total += w[j];
  double t = u * total, c = 0.0, tol = ORC_NEAR_TIE;
  int last_pos = -1;
  for (int j = 0; j < V; ++j) {
    if (w[j] <= 0.0) continue;
    double prev = c;
    c += w[j];
    last_pos = j;
    if (c > t) {
      if (t - prev < tol || c - t < tol) *near = 1;
      return j;
    }
  }
  /* rounding put t at or past the end of the CDF: take the last token with w > 0 */
  *near = 1;
  return last_pos < 0 ? 0 : last_pos;
}

/* Sample from norm([p - q]+), or from p if q is NULL; falls back to p (and reports
 * a near tie) when the residual has no mass. */
static int orc_sample_residual(const double *p, const double *q, int V, double u, int *near) {
  double *w = (double *)orc_alloc(sizeof(double) * (size_t)V);
  double total = 0.0;
  for (int j = 0; j < V; ++j) {
    w[j] = q ? (p[j] - q[j] > 0.0 ? p[j] - q[j] : 0.0) : p[j];
    total += w[j];
  }
  if (!(total > 0.0)) {
    *near = 1;
    for (int j = 0; j < V; ++j) w[j] = p[j];
  }
  int tok = orc_inverse_cdf(w, V, u, near);
  free(w);
  return tok;
}

/* Effective q row for depth d (1-based): from draft logits (T, top-k applied) or given
 * directly as probabilities (f32). */
static void orc_q_row(const void *q, int q_kind, int dtype, int b, int Dq, int d, int V,
                      double T, int top_k, double top_p, double *zbuf, double *out, int *near) {
  size_t row = (size_t)b * Dq + (d - 1);
  if (q_kind == ORC_Q_PROBS_F32) {
    orc_load_row(q, ORC_F32, row, V, out);
  } else {
    orc_load_row(q, dtype, row, V, zbuf);
    orc_effective_dist(zbuf, V, T, top_k, top_p, out, near);
  }
}

/* -------------------------------------------------- acceptance: tree form */

/* Tree acceptance (see the readings at the top of this file).  parent [N] shared by
 * all sequences; node_tokens [B,N] (column 0 = root, unused); target_logits [B,N,V];
 * q [B,Dq,V] with row d-1 for depth d.  Outputs have Dmax+1 columns, unused -1.
 * out_acc / out_ratio [B,N] are optional (per-node decision and p/q, root = 1 / nan).
 * out_flags [B] optional: bit0 = a draft had q(x)=0, bit1 = token id out of range. */
int orc_accept_tree(int mode, int dtype, int B, int N, int V, const int32_t *parent_all,
                    int parent_stride, const int32_t *node_tokens, const void *target_logits, const void *q,
                    int q_kind, int Dq, double T, int top_k, double top_p, uint64_t seed,
                    uint64_t round, int32_t *out_path_nodes, int32_t *out_tokens, int32_t *out_num_emitted,
                    int32_t *out_num_accepted, uint32_t *out_near_ties, uint8_t *out_acc,
                    double *out_ratio, uint32_t *out_flags) {
  int Dmax = 0;
  for (int b = 0; b < (parent_stride ? B : 1); ++b) {
    const int32_t *par = parent_all + (size_t)b * parent_stride;
    if (orc_check_tree(N, par)) return 1;
    for (int n = 0; n < N; ++n) {
      int d = orc_depth(par, n);
      if (d > Dmax) Dmax = d;
    }
  }
  int greedy = (mode == ORC_GREEDY) || (T == 0.0);
  if (!greedy && Dq < Dmax) return 2;
  if (!greedy && q_kind == ORC_Q_DRAFT_ONEHOT) return 4; /* one-hot drafts: chains only */
  /* output columns: the deepest path + 1 (per-sequence trees: N, the deepest possible) */
  int W = parent_stride ? N : Dmax + 1;
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    const int32_t *parent = parent_all + (size_t)b * parent_stride; /* this sequence's tree */
    int *depth = (int *)orc_alloc(sizeof(int) * (size_t)N);
    for (int n = 0; n < N; ++n) depth[n] = orc_depth(parent, n);
    double *z = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *pa = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *qd = (double *)orc_alloc(sizeof(double) * (size_t)V);
    unsigned char *acc = (unsigned char *)calloc((size_t)N, 1);
    unsigned char *ok = (unsigned char *)calloc((size_t)N, 1);
    double *ratio = (double *)orc_alloc(sizeof(double) * (size_t)N);
    unsigned char *dec_near = (unsigned char *)calloc((size_t)N, 1);
    uint32_t flags = 0;
    int nuc_near = 0;  /* a nucleus cut of one of the rows used was a near tie */
    for (int c = 0; c < N; ++c) ratio[c] = NAN;

    /* decisions: node c against its parent's p and the q of its depth */
    for (int a = 0; a < N; ++a) {
      int has_child = 0;
      for (int c = a + 1; c < N; ++c)
        if (parent[c] == a) has_child = 1;
      if (!has_child) continue;
      orc_load_row(target_logits, dtype, (size_t)b * N + a, V, z);
      int amax = orc_argmax(z, V);
      if (!greedy) {
        orc_effective_dist(z, V, T, top_k, top_p, pa, &nuc_near);
        orc_q_row(q, q_kind, dtype, b, Dq, depth[a] + 1, V, T, top_k, top_p, z, qd, &nuc_near);
      }
      for (int c = a + 1; c < N; ++c) {
        if (parent[c] != a) continue;
        int x = node_tokens[(size_t)b * N + c];
        if (x < 0 || x >= V) {
          flags |= 2u;
          acc[c] = 0;
          continue;
        }
        if (greedy) {
          acc[c] = (x == amax);
          continue;
        }
        double u_acc, u_smp;
        orc_uniforms(seed, round, 0u, b, c, &u_acc, &u_smp);
        double pr = pa[x], qr = qd[x], r;
        if (qr > 0.0) {
          r = pr / qr;
        } else {
          flags |= 1u;
          r = pr > 0.0 ? INFINITY : 0.0;
        }
        ratio[c] = r;
        acc[c] = (u_acc < r);
        dec_near[c] = (fabs(u_acc - r) < ORC_NEAR_TIE);
      }
    }

    /* path: node on an accepted root path; chosen = deepest, ties -> smallest row */
    ok[0] = 1;
    int best = 0;
    uint32_t near = 0;
    for (int c = 1; c < N; ++c) {
      ok[c] = ok[parent[c]] && acc[c];
      if (ok[parent[c]] && dec_near[c]) ++near;
      if (ok[c] && depth[c] > depth[best]) best = c;
    }

    /* final token: residual sample if the chosen node has children, else the bonus */
    int has_child = 0;
    for (int c = best + 1; c < N; ++c)
      if (parent[c] == best) has_child = 1;
    orc_load_row(target_logits, dtype, (size_t)b * N + best, V, z);
    int tok;
    if (greedy) {
      tok = orc_argmax(z, V);
    } else {
      double u_acc, u_smp;
      orc_uniforms(seed, round, 0u, b, best, &u_acc, &u_smp);
      orc_effective_dist(z, V, T, top_k, top_p, pa, &nuc_near);
      int near_s = 0;
      if (has_child) {
        orc_q_row(q, q_kind, dtype, b, Dq, depth[best] + 1, V, T, top_k, top_p, z, qd, &nuc_near);
        tok = orc_sample_residual(pa, qd, V, u_smp, &near_s);
      } else {
        tok = orc_sample_residual(pa, NULL, V, u_smp, &near_s);
      }
      near += (uint32_t)near_s * ORC_SAMPLE_TIE;
    }
    near += (uint32_t)nuc_near;

    /* outputs: path nodes root..best in depth order, their tokens, then the sample */
    int D = depth[best];
    int32_t *pn = out_path_nodes ? out_path_nodes + (size_t)b * W : NULL;
    int32_t *tk = out_tokens + (size_t)b * W;
    for (int i = 0; i < W; ++i) {
      if (pn) pn[i] = -1;
      tk[i] = -1;
    }
    for (int a = best, i = D; a >= 0; a = parent[a], --i) {
      if (pn) pn[i] = a;
      if (i >= 1) tk[i - 1] = node_tokens[(size_t)b * N + a];
    }
    tk[D] = tok;
    out_num_emitted[b] = D + 1;
    out_num_accepted[b] = D;
    if (out_near_ties) out_near_ties[b] = near;
    if (out_acc)
      for (int c = 0; c < N; ++c) out_acc[(size_t)b * N + c] = c == 0 ? 1 : acc[c];
    if (out_ratio)
      for (int c = 0; c < N; ++c) out_ratio[(size_t)b * N + c] = ratio[c];
    if (out_flags) out_flags[b] = flags;
    free(z); free(pa); free(qd); free(acc); free(ok); free(ratio); free(dec_near); free(depth);
  }
  return 0;
}

/* ------------------------------------------------- acceptance: chain form */

/* Chain acceptance as the left-to-right procedure: for i = 1..gamma accept draft x_i
 * with probability min(1, p_{i-1}(x_i)/q_i(x_i)); at the first rejection sample from
 * norm([p_{i-1} - q_i]+) and stop; if all pass, sample the bonus from p_gamma.
 * Greedy: accept while x_i == argmax z_{i-1}; then emit argmax of that row.
 * target_logits [B,gamma+1,V]; q [B,gamma,V]; draft_tokens [B,gamma];
 * out_tokens [B,gamma+1] (unused -1).  Node ids for the uniforms: draft i is node i.
 * A draft of -1 ends the sequence's chain (a prompt lookup may propose fewer than gamma
 * tokens): if the k drafts before it pass, the bonus comes from p_k.  q_kind
 * ORC_Q_DRAFT_ONEHOT takes q_i = e_{x_i} (deterministic drafts: accept iff u < p(x_i), and
 * after a rejection norm([p - e_x]+) is p without x); q is then not read. */
int orc_accept_chain(int mode, int dtype, int B, int gamma, int V, const void *target_logits,
                     const void *q, int q_kind, const int32_t *draft_tokens, double T,
                     int top_k, double top_p, uint64_t seed, uint64_t round, int32_t *out_tokens,
                     int32_t *out_num_emitted, int32_t *out_num_accepted,
                     uint32_t *out_near_ties, uint32_t *out_flags) {
  int greedy = (mode == ORC_GREEDY) || (T == 0.0);
  int W = gamma + 1;
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    double *z = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *p = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *qi = (double *)orc_alloc(sizeof(double) * (size_t)V);
    int32_t *tk = out_tokens + (size_t)b * W;
    uint32_t near = 0, flags = 0;
    int nuc_near = 0;  /* a nucleus cut of one of the rows used was a near tie */
    for (int i = 0; i < W; ++i) tk[i] = -1;
    int i = 1, tok = -1, ended = 0;
    for (; i <= gamma; ++i) {
      int x = draft_tokens[(size_t)b * gamma + (i - 1)];
      if (x == -1) { /* no more drafts: the bonus is taken below */
        ended = 1;
        break;
      }
      orc_load_row(target_logits, dtype, (size_t)b * W + (i - 1), V, z);
      if (greedy) {
        int amax = orc_argmax(z, V);
        if (x >= 0 && x < V && x == amax) {
          tk[i - 1] = x;
          continue;
        }
        if (x < 0 || x >= V) flags |= 2u;
        tok = amax;
        break;
      }
      orc_effective_dist(z, V, T, top_k, top_p, p, &nuc_near);
      if (q_kind == ORC_Q_DRAFT_ONEHOT) {
        for (int j = 0; j < V; ++j) qi[j] = (j == x) ? 1.0 : 0.0;
      } else {
        orc_q_row(q, q_kind, dtype, b, gamma, i, V, T, top_k, top_p, z, qi, &nuc_near);
      }
      double u_acc, u_smp;
      orc_uniforms(seed, round, 0u, b, i, &u_acc, &u_smp);
      int accepted = 0;
      if (x >= 0 && x < V) {
        double r;
        if (qi[x] > 0.0) {
          r = p[x] / qi[x];
        } else {
          flags |= 1u;
          r = p[x] > 0.0 ? INFINITY : 0.0;
        }
        if (fabs(u_acc - r) < ORC_NEAR_TIE) ++near;
        accepted = (u_acc < r);
      } else {
        flags |= 2u;
      }
      if (accepted) {
        tk[i - 1] = x;
        continue;
      }
      /* first rejection: resample from the residual at this position (node i-1) */
      double ua, us;
      orc_uniforms(seed, round, 0u, b, i - 1, &ua, &us);
      int near_s = 0;
      tok = orc_sample_residual(p, qi, V, us, &near_s);
      near += (uint32_t)near_s * ORC_SAMPLE_TIE;
      break;
    }
    if (i > gamma || ended) { /* every draft present accepted: bonus from row (node) i-1 */
      int last = i - 1;
      orc_load_row(target_logits, dtype, (size_t)b * W + last, V, z);
      if (greedy) {
        tok = orc_argmax(z, V);
      } else {
        orc_effective_dist(z, V, T, top_k, top_p, p, &nuc_near);
        double ua, us;
        orc_uniforms(seed, round, 0u, b, last, &ua, &us);
        int near_s = 0;
        tok = orc_sample_residual(p, NULL, V, us, &near_s);
        near += (uint32_t)near_s * ORC_SAMPLE_TIE;
      }
    }
    near += (uint32_t)nuc_near;
    int acc_n = i - 1;
    tk[acc_n] = tok;
    out_num_emitted[b] = acc_n + 1;
    out_num_accepted[b] = acc_n;
    if (out_near_ties) out_near_ties[b] = near;
    if (out_flags) out_flags[b] = flags;
    free(z); free(p); free(qi);
  }
  return 0;
}

/* ------------------------------------------------ acceptance: typical rule */

/* Typical acceptance (the Medusa paper: T. Cai et al., "Medusa: Simple LLM Inference
 * Acceleration Framework with Multiple Decoding Heads", 2024, section "Typical Acceptance";
 * the jennyma11 blog, section "Medusa", names it beside lossless verification without a
 * rule).  Node c (parent a) is accepted iff p_a(x_c) > min(epsilon, delta * exp(-H(p_a))),
 * p_a the parent's target distribution at temperature T (T > 0, no top-k), H its entropy in
 * nats; no draft distribution and no uniforms are used.  The kept node a* is the deepest
 * one whose whole root path is accepted (ties: smallest row); the tokens of its path are
 * emitted, then the target's most likely token at a* (argmax, lowest id), so that every
 * step emits at least one token.  Near ties (decision class): |p_a(x_c) - threshold| <
 * 1e-6 on a decision whose parent lies on an accepted path.  parent_all / parent_stride
 * as orc_accept_tree; outputs as orc_accept_tree (W = depth + 1, or N per sequence). */
int orc_accept_typical(int dtype, int B, int N, int V, const int32_t *parent_all,
                       int parent_stride, const int32_t *node_tokens, const void *target_logits,
                       double T, double epsilon, double delta, int32_t *out_path_nodes,
                       int32_t *out_tokens, int32_t *out_num_emitted, int32_t *out_num_accepted,
                       uint32_t *out_near_ties, double *out_entropy) {
  if (!(T > 0.0)) return 3;
  int Dmax = 0;
  for (int b = 0; b < (parent_stride ? B : 1); ++b) {
    const int32_t *par = parent_all + (size_t)b * parent_stride;
    if (orc_check_tree(N, par)) return 1;
    for (int n = 0; n < N; ++n) {
      int d = orc_depth(par, n);
      if (d > Dmax) Dmax = d;
    }
  }
  int W = parent_stride ? N : Dmax + 1;
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    const int32_t *parent = parent_all + (size_t)b * parent_stride;
    double *z = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *pa = (double *)orc_alloc(sizeof(double) * (size_t)V);
    unsigned char *acc = (unsigned char *)calloc((size_t)N, 1);
    unsigned char *ok = (unsigned char *)calloc((size_t)N, 1);
    unsigned char *dec_near = (unsigned char *)calloc((size_t)N, 1);
    int *depth = (int *)orc_alloc(sizeof(int) * (size_t)N);
    for (int n = 0; n < N; ++n) depth[n] = orc_depth(parent, n);
    for (int a = 0; a < N; ++a) {
      orc_load_row(target_logits, dtype, (size_t)b * N + a, V, z);
      orc_effective_dist(z, V, T, 0, 1.0, pa, NULL);
      double H = 0.0; /* entropy in nats */
      for (int j = 0; j < V; ++j)
        if (pa[j] > 0.0) H -= pa[j] * log(pa[j]);
      if (out_entropy) out_entropy[(size_t)b * N + a] = H;
      double thr = delta * exp(-H);
      if (epsilon < thr) thr = epsilon;
      for (int c = a + 1; c < N; ++c) {
        if (parent[c] != a) continue;
        int x = node_tokens[(size_t)b * N + c];
        if (x < 0 || x >= V) continue; /* rejected */
        acc[c] = pa[x] > thr;
        dec_near[c] = fabs(pa[x] - thr) < ORC_NEAR_TIE;
      }
    }
    ok[0] = 1;
    int best = 0;
    uint32_t near = 0;
    for (int c = 1; c < N; ++c) {
      ok[c] = ok[parent[c]] && acc[c];
      if (ok[parent[c]] && dec_near[c]) ++near;
      if (ok[c] && depth[c] > depth[best]) best = c;
    }
    orc_load_row(target_logits, dtype, (size_t)b * N + best, V, z);
    int tok = orc_argmax(z, V);
    int D = depth[best];
    int32_t *pn = out_path_nodes ? out_path_nodes + (size_t)b * W : NULL;
    int32_t *tk = out_tokens + (size_t)b * W;
    for (int i = 0; i < W; ++i) {
      if (pn) pn[i] = -1;
      tk[i] = -1;
    }
    for (int a = best, i = D; a >= 0; a = parent[a], --i) {
      if (pn) pn[i] = a;
      if (i >= 1) tk[i - 1] = node_tokens[(size_t)b * N + a];
    }
    tk[D] = tok;
    out_num_emitted[b] = D + 1;
    out_num_accepted[b] = D;
    if (out_near_ties) out_near_ties[b] = near;
    free(z); free(pa); free(acc); free(ok); free(dec_near); free(depth);
  }
  return 0;
}

/* ------------------------------------------------------------- KV commit */

/* Copy the tree K/V rows of the path nodes (root, then accepted nodes in depth order)
 * to cache positions L_b .. L_b + num_accepted, then advance prefix_len by
 * num_accepted + 1.  Byte copies of whole (node, kv-head) rows; nothing else changes. */
void orc_commit_kv(int dtype, int B, int N, int Hkv, int D, const void *k_tree,
                   const void *v_tree, const int32_t *path_nodes, int path_stride,
                   const int32_t *num_accepted, void *cache_k, void *cache_v,
                   int32_t *prefix_len, const int32_t *block_table, int max_blocks,
                   int block_size, int Lmax) {
  size_t es = orc_esize(dtype);
  size_t row_bytes = (size_t)Hkv * D * es;
  for (int b = 0; b < B; ++b) {
    int L = prefix_len[b];
    for (int i = 0; i <= num_accepted[b]; ++i) {
      int node = path_nodes[(size_t)b * path_stride + i];
      size_t dst = orc_cache_row(b, L + i, block_table, max_blocks, block_size, Lmax) * row_bytes;
      size_t src = ((size_t)b * N + node) * row_bytes;
      memcpy((char *)cache_k + dst, (const char *)k_tree + src, row_bytes);
      memcpy((char *)cache_v + dst, (const char *)v_tree + src, row_bytes);
    }
    prefix_len[b] = L + num_accepted[b] + 1;
  }
}

/* ------------------------------------------------------------------- LM head */

/* Logits from hidden states: z[r, v] = sum_k h[r, k] * W[v, k].  "推测解码技术详解：加速LLM
 * 推理的关键", section "Medusa Heads", architecture figure: the original LM head and the
 * Medusa heads all read the backbone's hidden states; lpnh.cn section 3.1: a head is a
 * Linear(H, V) from the hidden state h_t to V logits.  hidden [rows, Dm] and weight
 * [V, Dm] (row v = token v's output embedding) in f32 or bf16; out [rows, V] in double,
 * each sum taken in ascending k.  Readings: no bias term; the hidden state arrives
 * already normalised (the final norm is the model's, outside the verify step).  The
 * acceptance functions read the result with dtype ORC_F64. */
void orc_lm_head(int rows, int Dm, int V, const void *hidden, int h_dtype, const void *weight,
                 int w_dtype, double *out) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int k = 0; k < Dm; ++k)
        acc += orc_elem(hidden, h_dtype, (size_t)r * Dm + k) * orc_elem(weight, w_dtype, (size_t)v * Dm + k);
      out[(size_t)r * V + v] = acc;
    }
  }
}

/* ------------------------------------------------------ n-gram (prompt lookup) drafts */

/* Prompt-lookup drafting ("投机解码的五条路线" (jennyma11 blog), section "Prompt Lookup /
 * N-gram"): take the last n tokens of the history, find the same n tokens earlier in
 * it, and propose the tokens that follow that earlier occurrence.  Readings: n runs
 * from max_n down to min_n and the first n with a match wins; among matches the most
 * recent one (largest start j) is taken; a match must end before the last token so that
 * at least one token follows it; the drafts are the up to gamma tokens after the match
 * (fewer when the history ends), unused slots -1.  history [B,Lmax]; length [B] (clamped
 * to [0, Lmax]); out_drafts [B,gamma]; out_num [B] (0 when nothing matches). */
void orc_ngram_draft(int B, int Lmax, const int32_t *history, const int32_t *length, int max_n,
                     int min_n, int gamma, int32_t *out_drafts, int32_t *out_num) {
  for (int b = 0; b < B; ++b) {
    const int32_t *h = history + (size_t)b * Lmax;
    int L = length[b];
    if (L < 0) L = 0;
    if (L > Lmax) L = Lmax;
    int32_t *d = out_drafts + (size_t)b * gamma;
    for (int i = 0; i < gamma; ++i) d[i] = -1;
    out_num[b] = 0;
    for (int n = max_n; n >= min_n; --n) {
      if (n < 1 || L < n + 1) continue;
      int found = -1;
      for (int j = L - n - 1; j >= 0 && found < 0; --j) {
        int same = 1;
        for (int t = 0; t < n; ++t)
          if (h[j + t] != h[L - n + t]) {
            same = 0;
            break;
          }
        if (same) found = j;
      }
      if (found >= 0) {
        int cnt = 0;
        for (int i = 0; i < gamma && found + n + i < L; ++i) d[cnt++] = h[found + n + i];
        out_num[b] = cnt;
        break;
      }
    }
  }
}

/* ------------------------------------ acceptance: tree, siblings tried in rank order */

/* Exact tree acceptance with the siblings of a node tried in turn (the multi-candidate
 * form of the acceptance rule of hncyxsy.com sections 2.1-2.2: after a rejected
 * candidate the target distribution becomes the residual norm([p - q]+) for the next
 * one; the jennyma11 blog, section "Medusa", separates this lossless tree verification
 * from typical acceptance).  From the root: the children of the current node are tried
 * in row (rank) order, child c accepted iff u_acc(b, c) < p_cur(x_c) / q_{d+1}(x_c), where
 * p_cur starts as the node's effective target distribution and after each rejection is
 * replaced by norm([p_cur - q_{d+1}]+) (kept unchanged, and reported as a near tie, when
 * that residual has no mass).  An accepted child becomes the current node; when the last
 * child is rejected the next token is sampled with u_smp(b, node) from the residual of the
 * last p_cur; a leaf reached draws the bonus from its p.  For drafts sampled independently
 * from q this keeps the output distributed as p; with one child per node it is the chain
 * procedure.  Exact mode only (greedy: orc_accept_tree).  Arguments and outputs as
 * orc_accept_tree (no per-node decision outputs). */
int orc_accept_tree_recursive(int dtype, int B, int N, int V, const int32_t *parent_all,
                              int parent_stride, const int32_t *node_tokens, const void *target_logits,
                              const void *q, int q_kind, int Dq, double T, int top_k,
                              double top_p, uint64_t seed, uint64_t round,
                              int32_t *out_path_nodes, int32_t *out_tokens,
                              int32_t *out_num_emitted, int32_t *out_num_accepted,
                              uint32_t *out_near_ties, uint32_t *out_flags) {
  if (T == 0.0) return 3;
  int Dmax = 0;
  for (int b = 0; b < (parent_stride ? B : 1); ++b) {
    const int32_t *par = parent_all + (size_t)b * parent_stride;
    if (orc_check_tree(N, par)) return 1;
    for (int n = 0; n < N; ++n) {
      int d = orc_depth(par, n);
      if (d > Dmax) Dmax = d;
    }
  }
  if (Dq < Dmax || q_kind == ORC_Q_DRAFT_ONEHOT) return 2;
  int W = parent_stride ? N : Dmax + 1;
#pragma omp parallel for schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    const int32_t *parent = parent_all + (size_t)b * parent_stride; /* this sequence's tree */
    int *depth = (int *)orc_alloc(sizeof(int) * (size_t)N);
    for (int n = 0; n < N; ++n) depth[n] = orc_depth(parent, n);
    double *z = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *pc = (double *)orc_alloc(sizeof(double) * (size_t)V);
    double *qd = (double *)orc_alloc(sizeof(double) * (size_t)V);
    uint32_t near = 0, flags = 0;
    int nuc_near = 0;
    int node = 0, tok = -1;
    for (;;) {
      int first = -1, last = -1;
      for (int c = node + 1; c < N; ++c)
        if (parent[c] == node) {
          if (first < 0) first = c;
          last = c;
        }
      orc_load_row(target_logits, dtype, (size_t)b * N + node, V, z);
      orc_effective_dist(z, V, T, top_k, top_p, pc, &nuc_near);
      double ua, us;
      orc_uniforms(seed, round, 0u, b, node, &ua, &us);
      int near_s = 0;
      if (first < 0) { /* a leaf: the bonus from its p */
        tok = orc_sample_residual(pc, NULL, V, us, &near_s);
        near += (uint32_t)near_s * ORC_SAMPLE_TIE;
        break;
      }
      orc_q_row(q, q_kind, dtype, b, Dq, depth[node] + 1, V, T, top_k, top_p, z, qd, &nuc_near);
      int next = -1;
      for (int c = first; c <= last; ++c) {
        if (parent[c] != node) continue;
        int x = node_tokens[(size_t)b * N + c];
        int accepted = 0;
        if (x >= 0 && x < V) {
          double u_acc, u_smp, r;
          orc_uniforms(seed, round, 0u, b, c, &u_acc, &u_smp);
          if (qd[x] > 0.0) {
            r = pc[x] / qd[x];
          } else {
            flags |= 1u;
            r = pc[x] > 0.0 ? INFINITY : 0.0;
          }
          if (fabs(u_acc - r) < ORC_NEAR_TIE) ++near;
          accepted = (u_acc < r);
        } else {
          flags |= 2u;
        }
        if (accepted) {
          next = c;
          break;
        }
        if (c == last) break; /* the residual of this p_cur is sampled below */
        /* the next sibling sees the residual */
        double total = 0.0;
        for (int j = 0; j < V; ++j) total += pc[j] - qd[j] > 0.0 ? pc[j] - qd[j] : 0.0;
        if (total > 0.0) {
          for (int j = 0; j < V; ++j) pc[j] = pc[j] - qd[j] > 0.0 ? (pc[j] - qd[j]) / total : 0.0;
        } else {
          ++near;
        }
      }
      if (next >= 0) {
        node = next;
        continue;
      }
      tok = orc_sample_residual(pc, qd, V, us, &near_s);
      near += (uint32_t)near_s * ORC_SAMPLE_TIE;
      break;
    }
    near += (uint32_t)nuc_near;
    int D = depth[node];
    int32_t *pn = out_path_nodes ? out_path_nodes + (size_t)b * W : NULL;
    int32_t *tk = out_tokens + (size_t)b * W;
    for (int i = 0; i < W; ++i) {
      if (pn) pn[i] = -1;
      tk[i] = -1;
    }
    for (int a = node, i = D; a >= 0; a = parent[a], --i) {
      if (pn) pn[i] = a;
      if (i >= 1) tk[i - 1] = node_tokens[(size_t)b * N + a];
    }
    tk[D] = tok;
    out_num_emitted[b] = D + 1;
    out_num_accepted[b] = D;
    if (out_near_ties) out_near_ties[b] = near;
    if (out_flags) out_flags[b] = flags;
    free(z); free(pc); free(qd); free(depth);
  }
  return 0;
}
