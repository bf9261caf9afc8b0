// Reading the per-row statistics of the acceptance kernels (sm_103a).
//
// A logit row's effective distribution (temperature, top-k, then top-p within the top k)
// is described by its RowStat: the row maximum, the kept set as a threshold on an
// order-preserving key (index tie-break: lower ids first), and the softmax sum over the
// kept entries.  p(j) = kept(j) ? exp((z_j - zmax) / T) / S : 0.
#pragma once

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

// Row statistics written by another kernel or by other CTAs of the same launch: read from
// L2, not L1.
__device__ __forceinline__ RowStat load_stat(const RowStat *s) {
  RowStat r;
  r.zmax = __ldcg(&s->zmax);
  r.argmax = __ldcg(&s->argmax);
  r.key_k = __ldcg(&s->key_k);
  r.idx_k = __ldcg(&s->idx_k);
  r.S = __ldcg(&s->S);
  r.flags = __ldcg(&s->flags);
  r.H = __ldcg(&s->H);
  r.pad = 0u;
  return r;
}

// Is entry (value z, index j) inside the row's kept set?
template <typename T>
__device__ __forceinline__ bool kept(float z, int j, const RowStat &st) {
  const uint32_t k = Elem<T>::key(z);
  return k > st.key_k || (k == st.key_k && j <= st.idx_k);
}

}  // namespace sv
