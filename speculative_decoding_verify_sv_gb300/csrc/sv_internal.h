// Internal launch parameters of the verify-step kernels (host and device).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sv.h"

namespace sv {

constexpr int kMaxNodes = SV_MAX_TREE_NODES;

// The candidate tree, passed by value: parent (BFS order, parent[0] = -1) and depth.
// Per-sequence trees (rows != NULL): sequence b's parent array is rows[b*stride ..
// b*stride + N) in device memory, checked on the device; parent, depth and has_child are
// then unused and Dmax = N - 1 (the widest path, which sizes the outputs).
struct Tree {
  int N;
  int Dmax;
  int8_t parent[kMaxNodes];
  int8_t depth[kMaxNodes];
  int8_t has_child[kMaxNodes];
  const int32_t *rows;
  int stride;
};

// ---------------------------------------------------------------- attention

struct AttnParams {
  const void *q, *k_tree, *v_tree;  // [B,N,Hq,D], [B,N,Hkv,D] x2
  const void *cache_k, *cache_v;    // [B,Lmax,Hkv,D] or [num_blocks,block_size,Hkv,D]
  const int32_t *prefix_len;        // [B]
  const int32_t *block_table;       // [B,max_blocks] or NULL
  void *out;                        // [B,N,Hq,D]
  float *part_o;                    // [B,Hkv,S,Mpad,D] unnormalised partial outputs
  float *part_ml;                   // [B,Hkv,S,Mpad,2] running max (log2 units) and sum
  unsigned int *status;
  int B, N, Hq, Hkv, G, D;
  int Lmax, block_size, max_blocks, num_blocks, cap;  // cap = largest valid prefix
  int M, m_tiles, Mpad;  // query rows per (b, kv head) = N*G, tiles of 64 rows
  int splits, chunk;     // prefix split: split s covers [s*chunk, (s+1)*chunk)
  float scale_log2;      // softmax scale * log2(e)
  float scale;
  Tree tree;
  unsigned long long wait_ns;  // limit of the tensor-core kernel's waits for progress
};

struct AttnPlan {
  int m_tiles, Mpad, splits, chunk;
  size_t ws_bytes;
};

AttnPlan attn_plan(sv_dtype dt, int B, int N, int Hq, int Hkv, int D, int max_prefix,
                   int num_sms);
cudaError_t launch_attention(sv_dtype dt, const AttnParams &p, cudaStream_t s);

// Tensor-core (tcgen05) tree attention: persistent CTAs over a stream-K split of the
// flattened (unit, key tile) space.
struct TcParams {
  CUtensorMap tm_q, tm_kt, tm_vt, tm_kc, tm_vc;  // Q, tree K/V, cache K/V (128B swizzle)
  // paged cache pages as (64, 8, 2, rows/8, Hkv) boxes: both 64-column halves of a page in
  // one copy, into the grouped tile layout (used when pg_grouped != 0)
  CUtensorMap tm_kc5, tm_vc5;
  int pg_grouped;
  const int32_t *prefix_len;
  const int32_t *block_table;
  void *out;
  float *part_o;          // [slots, rows, D] fp32 partial outputs of cut units
  float *part_ml;         // [slots, rows, 2] running max (log2) and sum
  unsigned long long *hdr;    // [0] generation of the last completed call, [1] low: CTAs done
  unsigned long long *flags;  // [slots] epoch of the call that published each partial
  unsigned int *status;
  int B, N, Hq, Hkv, G, M, m_groups, upb, bn;
  int vt;  // empty slots charged for the start of each unit in the work split
  int Lmax, block_size, max_blocks, num_blocks, cap, paged, page_rows;
  float scale_log2;
  Tree tree;
  unsigned long long wait_ns;  // a wait for progress gives up after this long
};

struct TcPlan {
  int MT, m_groups, grid, CP, BN;
  size_t off_hdr, off_flags, off_ml, off_o, ws_bytes;
};

// paged_block_size: the cache's block size, or 0 for a contiguous cache
bool tc_eligible(sv_dtype dt, int N, int Hq, int Hkv, int D, int paged_block_size);
TcPlan tc_plan(int B, int N, int Hq, int Hkv, int D, int num_sms);
cudaError_t launch_attention_tc(const AttnParams &p, const TcPlan &pl, void *ws, cudaStream_t s);

// Kernels launched by this library so far (all devices, all threads).
void count_launches(unsigned n);

// --------------------------------------------------------------- acceptance

struct RowStat {
  float zmax;     // largest logit of the row
  int32_t argmax; // its lowest index
  uint32_t key_k; // top-k threshold key (kept: key > key_k, or == key_k and idx <= idx_k)
  int32_t idx_k;
  float S;        // sum over kept entries of exp((z - zmax) / T)
  uint32_t flags; // bit 0: the top-p cut lies within 1e-6 of top_p (a near tie)
  float H;        // entropy of the row's distribution in nats (typical acceptance only)
  uint32_t pad;
};

// ------------------------------------------------------------------- commit

struct CommitParams {
  const void *k_tree, *v_tree;
  const int32_t *path_nodes;
  int path_stride;
  const int32_t *num_accepted;
  void *cache_k, *cache_v;
  int32_t *prefix_len;
  const int32_t *block_table;
  int B, N, Hkv, D, esize;
  int Lmax, block_size, max_blocks, num_blocks;
  unsigned int *status;
};

struct AcceptParams {
  int mode;        // SV_GREEDY / SV_EXACT
  int B, N, V, Dq;
  int q_kind;      // SV_Q_PROBS_F32 / SV_Q_LOGITS
  const void *target;        // [B,N,V]
  const void *q;             // [B,Dq,V]
  const int32_t *tokens;     // token of node c of seq b = tokens[b*tok_stride + c - tok_offset]
  int tok_stride, tok_offset;
  int chain_end;             // chains: a token of -1 ends the sequence's drafts
  float temperature;
  float c_log2;              // log2(e) / T
  int top_k;                 // 0 = off
  float top_p;               // 1 = off; < 1 only with top-k (the nucleus of its distribution)
  int ring_stages;           // stages of the select kernel's ring (set at its launch)
  int stat_row0;             // first row of the statistics kernel's grid (q rows only: B*N)
  // typical acceptance (mode SV_GREEDY in the select kernel, entropy in the statistics):
  // node accepted iff p_parent(x) > min(typ_eps, typ_delta * exp(-H(p_parent)))
  int typical;
  float typ_eps, typ_delta;
  uint64_t seed, round;
  RowStat *stats;            // [B*N + B*Dq]
  int32_t *out_path_nodes;   // [B,Dmax+1] or NULL
  int32_t *out_tokens;       // [B,Dmax+1]
  int32_t *out_num_emitted, *out_num_accepted;
  uint32_t *out_near_ties;   // or NULL
  unsigned int *status;
  Tree tree;
  // commit of the kept path in the same launch (commit != 0): cm's cache, tree K/V and
  // sizes are used; its path_nodes / num_accepted are the kernel's own results
  int commit;
  CommitParams cm;
};

size_t accept_ws_bytes(int B, int N, int Dq);

// ------------------------------------------------------------ n-gram drafts

struct NgramParams {
  const int32_t *history;  // [B,Lmax]
  const int32_t *length;   // [B]
  int B, Lmax, max_n, min_n, gamma;
  int32_t *out_drafts;     // [B,gamma]
  int32_t *out_num;        // [B]
  unsigned int *status;
};
cudaError_t launch_ngram(const NgramParams &p, cudaStream_t s);
cudaError_t launch_accept(sv_dtype dt, const AcceptParams &p, int num_sms, cudaStream_t s);
// The statistics kernel alone (every target row, then every q row for q logits).
cudaError_t launch_accept_stats(sv_dtype dt, const AcceptParams &p, cudaStream_t s);
// Exact tree acceptance with siblings tried in rank order: the statistics kernel, then one
// CTA per sequence walking the tree (exact mode only; no commit).
cudaError_t launch_accept_recursive(sv_dtype dt, const AcceptParams &p, cudaStream_t s);

cudaError_t launch_commit(const CommitParams &p, cudaStream_t s);

// ---------------------------------------------------------------- LM head

struct LmHeadParams {
  CUtensorMap tm_h, tm_w;  // hidden [R, Dm] and weight [V, Dm] as K-major operand views
  void *z;                 // [R, V] bf16 logits (out)
  float4 *part;            // [R, ntiles] per (row, 256-column tile): max, sum, argmax bits
  unsigned int *status;
  int R, V, Dm, mtiles, ntiles;
  float c_log2;            // log2(e) / T (0: statistics without the softmax sum)
};
// Bytes of the per-(row, tile) partial statistics of the projection.
size_t lm_head_part_bytes(int R, int V);
// z = hidden W^T (bf16 out), then, when stats is not NULL, the rows' statistics (max,
// argmax, softmax sum at temperature 1 / (c_log2 ln 2); no top-k) into stats[0..R).
cudaError_t launch_lm_head(const void *hidden, const void *weight, int R, int Dm, int V,
                           float c_log2, void *z, void *part, RowStat *stats, unsigned int *status,
                           int num_sms, cudaStream_t s);
// The acceptance with the target rows' statistics already in p.stats (from the projection):
// the statistics kernel over the q rows only (q logits), then the select kernel.
cudaError_t launch_accept_given_target_stats(sv_dtype dt, const AcceptParams &p, int num_sms,
                                             cudaStream_t s);

}  // namespace sv
