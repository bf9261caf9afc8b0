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
// One CTA per sequence.  For each n, the suffix is staged in shared memory and the
// threads scan the candidate starts in index order (coalesced reads of the history, the
// first token tested before the rest); each keeps its largest matching start and a
// shared atomic maximum gives the most recent one.  The first n with a match ends the
// loop for the whole CTA.
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kNgramThreads = 256;

__global__ void __launch_bounds__(kNgramThreads) ngram_draft_kernel(const NgramParams p) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t *h = p.history + (size_t)b * p.Lmax;
  int L = p.length[b];
  if (L < 0 || L > p.Lmax) {
    if (tid == 0) set_status(p.status, SV_DEV_BAD_PREFIX);
    L = L < 0 ? 0 : p.Lmax;
  }
  __shared__ int32_t suf[SV_MAX_NGRAM];
  __shared__ int s_best;
  int found = -1, nf = 0;
  for (int n = p.max_n; n >= p.min_n; --n) {
    if (L < n + 1) continue;  // the same in every thread
    __syncthreads();          // the previous n's reads of suf and s_best are done
    if (tid < n) suf[tid] = h[L - n + tid];
    if (tid == 0) s_best = -1;
    __syncthreads();
    const int32_t first = suf[0];
    int best = -1;
    for (int j = tid; j <= L - n - 1; j += kNgramThreads) {
      if (h[j] != first) continue;
      bool same = true;
      for (int t = 1; t < n && same; ++t) same = h[j + t] == suf[t];
      if (same) best = j;  // j grows along the loop: the last hit is this thread's largest
    }
    if (best >= 0) atomicMax(&s_best, best);
    __syncthreads();
    if (s_best >= 0) {  // read by every thread after the barrier: the same everywhere
      found = s_best;
      nf = n;
      break;
    }
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
