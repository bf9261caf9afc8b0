// Prompt-lookup (n-gram) drafting (sm_103a).
//
// Method ("投机解码的五条路线" (jennyma11 blog), section "Prompt Lookup / N-gram"): take the
// last n tokens of the history, find the same n tokens earlier in it, and propose the
// tokens that follow that occurrence as drafts for the target to verify.  Readings where
// the page is silent: n runs from max_n down to min_n and the first n with a match wins;
// the most recent occurrence (largest start) is taken; it must end before the last token,
// so that at least one token follows; up to gamma tokens are proposed, fewer when the
// history ends, unused slots -1.
//
// One CTA per sequence.  The history streams through shared memory in tiles of 4096
// tokens (plus the max_n - 1 that follow a tile, so that every n-gram starting in it is
// whole): each thread issues its 16 loads of a tile before any is used, so a tile costs
// one memory round trip.  Every candidate start j in the tile is tested against every n
// at once (the suffix of each n staged once in shared memory; a mismatch of the first
// token ends the test); each thread keeps its largest matching start per n (starts grow
// along its loop), a shared atomic maximum gives the most recent one per n, and the
// largest n with a match wins.
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kNgramThreads = 256;
constexpr int kNgramTile = 4096;

__global__ void __launch_bounds__(kNgramThreads) ngram_draft_kernel(const NgramParams p) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t *h = p.history + (size_t)b * p.Lmax;
  int L = p.length[b];
  if (L < 0 || L > p.Lmax) {
    if (tid == 0) set_status(p.status, SV_DEV_BAD_PREFIX);
    L = L < 0 ? 0 : p.Lmax;
  }
  __shared__ int32_t tile[kNgramTile + SV_MAX_NGRAM];
  __shared__ int32_t suf[SV_MAX_NGRAM + 1][SV_MAX_NGRAM];  // suf[n][t] = h[L - n + t]
  __shared__ int s_best[SV_MAX_NGRAM + 1];
  const int n_lo = p.min_n, n_hi = min(p.max_n, L - 1);  // an n-gram needs L >= n + 1
  for (int i = tid; i < (SV_MAX_NGRAM + 1) * SV_MAX_NGRAM; i += kNgramThreads) {
    const int n = i / SV_MAX_NGRAM, t = i % SV_MAX_NGRAM;
    if (n >= n_lo && n <= n_hi && t < n) suf[n][t] = h[L - n + t];
  }
  if (tid <= SV_MAX_NGRAM) s_best[tid] = -1;
  int best[SV_MAX_NGRAM + 1];
#pragma unroll
  for (int n = 0; n <= SV_MAX_NGRAM; ++n) best[n] = -1;
  // candidate starts j <= L - n_lo - 1 (the largest range, that of the smallest n)
  const int j_end = L - n_lo;
  for (int base = 0; base < j_end; base += kNgramTile) {
    __syncthreads();  // the previous tile (and, first, suf) is no longer read / is written
    const int cnt = min(kNgramTile + n_hi - 1, L - base);
    int32_t v[kNgramTile / kNgramThreads];
#pragma unroll
    for (int k = 0; k < kNgramTile / kNgramThreads; ++k) {
      const int i = tid + k * kNgramThreads;
      v[k] = i < cnt ? __ldg(h + base + i) : 0;
    }
#pragma unroll
    for (int k = 0; k < kNgramTile / kNgramThreads; ++k) {
      const int i = tid + k * kNgramThreads;
      if (i < cnt) tile[i] = v[k];
    }
    for (int i = kNgramTile + tid; i < cnt; i += kNgramThreads) tile[i] = __ldg(h + base + i);
    __syncthreads();
    const int jl_end = min(kNgramTile, j_end - base);
    for (int jl = tid; jl < jl_end; jl += kNgramThreads) {
      const int j = base + jl;
      const int32_t x = tile[jl];
      for (int n = n_lo; n <= n_hi; ++n) {
        if (j > L - n - 1 || x != suf[n][0]) continue;
        bool same = true;
        for (int t = 1; t < n && same; ++t) same = tile[jl + t] == suf[n][t];
        if (same) best[n] = j;  // j grows along the loop: the last hit is the largest
      }
    }
  }
  for (int n = n_lo; n <= n_hi; ++n)
    if (best[n] >= 0) atomicMax(&s_best[n], best[n]);
  __syncthreads();
  int found = -1, nf = 0;
  for (int n = n_hi; n >= n_lo; --n)  // the same in every thread
    if (s_best[n] >= 0) {
      found = s_best[n];
      nf = n;
      break;
    }
  if (tid < p.gamma) {
    int32_t v = -1;
    if (found >= 0 && found + nf + tid < L) v = h[found + nf + tid];
    p.out_drafts[(size_t)b * p.gamma + tid] = v;
  }
  if (tid == 0) p.out_num[b] = found >= 0 ? min(p.gamma, L - (found + nf)) : 0;
}

}  // namespace

cudaError_t launch_ngram(const NgramParams &p, cudaStream_t s) {
  ngram_draft_kernel<<<p.B, kNgramThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sv
