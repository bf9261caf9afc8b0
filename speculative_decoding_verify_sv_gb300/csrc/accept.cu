// Token acceptance over the vocabulary (sm_103a).
//
// Method (hncyxsy.com sections 2.1-2.2; jennyma11 blog, "先弄清无损验证" and "Medusa";
// qwbw.cn section 2.3): a draft x checked against target row p and draft row q is
// accepted iff u_acc < p(x)/q(x); at the first rejection the next token is drawn from
// norm([p - q]+); if every draft passes, a bonus token is drawn from the target's next
// row; p and q are the effective distributions (temperature, top-k).  Greedy accepts
// while the draft is the target's argmax.  For a tree every node is decided against
// its parent's row and the q row of its depth; the deepest node whose root path is all
// accepted is kept.
//
// Kernel 1 (one CTA per logit row, target rows then q rows): one coalesced pass of
// 16-byte loads gives the row max / argmax and, without top-k, the softmax sum by a
// per-thread online accumulation.  With top-k, a second pass gathers the few entries
// that can be in the top k (those at or above the smallest of k disjoint group
// maxima) into shared memory, ranks them, and sums the kept ones.
// Kernel 2 (one CTA per sequence): per-node ratios in double from the row statistics
// and the two logits of the candidate, the longest accepted path, and the final
// sample: a coalesced pass summing w = [p - q]+ (or p) per warp segment, then the
// owning warp re-walks its segment with a warp scan to find the inverse-CDF token.
#include <cfloat>
#include <climits>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kStatThreads = 512;
constexpr int kSelThreads = 512;
constexpr int kMaxCand = 4096;
constexpr double kNearTie = 1e-6;

struct Cand {
  float z;
  int idx;
};

template <typename T>
__device__ __forceinline__ const T *row_ptr(const void *base, size_t row, int V) {
  return static_cast<const T *>(base) + row * (size_t)V;
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Block-wide argmax (lowest index on ties); every thread gets the result.
template <int NT>
__device__ void block_argmax(float &v, int &i, float *shv, int *shi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (better(ov, oi, v, i)) v = ov, i = oi;
  }
  if (lane == 0) shv[warp] = v, shi[warp] = i;
  __syncthreads();
  if (warp == 0) {
    v = lane < NT / 32 ? shv[lane] : -INFINITY;
    i = lane < NT / 32 ? shi[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
      if (better(ov, oi, v, i)) v = ov, i = oi;
    }
    if (lane == 0) shv[0] = v, shi[0] = i;
  }
  __syncthreads();
  v = shv[0];
  i = shi[0];
  __syncthreads();
}

template <int NT>
__device__ double block_sum_d(double v, double *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < NT / 32 ? sh[lane] : 0.0;
    v = warp_sum_d(v);
    if (lane == 0) sh[0] = v;
  }
  __syncthreads();
  v = sh[0];
  __syncthreads();
  return v;
}

template <int NT>
__device__ unsigned block_sum_u(unsigned v, unsigned *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < NT / 32 ? sh[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) sh[0] = v;
  }
  __syncthreads();
  v = sh[0];
  __syncthreads();
  return v;
}

template <typename T>
__device__ __forceinline__ float key_to_value(uint32_t key);
template <>
__device__ __forceinline__ float key_to_value<bf16>(uint32_t key) {
  const uint32_t h = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  return __uint_as_float(h << 16);
}
template <>
__device__ __forceinline__ float key_to_value<float>(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Is entry (value z, index j) inside the row's top-k set?
template <typename T>
__device__ __forceinline__ bool kept(float z, int j, const RowStat &st) {
  const uint32_t k = Elem<T>::key(z);
  return k > st.key_k || (k == st.key_k && j <= st.idx_k);
}

// ------------------------------------------------------------ kernel 1

template <typename T, bool GREEDY, bool TOPK>
__global__ void __launch_bounds__(kStatThreads) accept_stats_kernel(const AcceptParams p) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NT = kStatThreads;
  __shared__ float sh_v[32];
  __shared__ int sh_i[32];
  __shared__ double sh_d[32];
  __shared__ unsigned sh_u[32];

  const int tid = threadIdx.x;
  const size_t row = blockIdx.x;
  const size_t nt_rows = (size_t)p.B * p.N;
  const T *x = row < nt_rows ? row_ptr<T>(p.target, row, p.V)
                             : row_ptr<T>(p.q, row - nt_rows, p.V);
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  const int nvec = p.V / VEC;
  const float c = p.c_log2;

  float vmax = -INFINITY;
  int imax = INT_MAX;
  float m = -INFINITY;
  KahanF acc;
  uint32_t umax[2] = {0u, 0u};  // TOPK: per-unit max key (units: even / odd lanes)

  for (int v = tid; v < nvec; v += NT) {
    const uint4 raw = __ldg(xv + v);
    float f[VEC];
    Elem<T>::unpack(raw, f);
    float vm = f[0];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      if (f[e] > vmax) vmax = f[e], imax = v * VEC + e;
      vm = fmaxf(vm, f[e]);
      if (TOPK) umax[e & 1] = max(umax[e & 1], Elem<T>::key(f[e]));
    }
    if (!GREEDY && !TOPK) {
      if (vm > m) {
        if (m != -INFINITY) {
          const float s = exp2f((m - vm) * c);
          acc.s *= s;
          acc.c *= s;
        }
        m = vm;
      }
      if (m != -INFINITY) {
        float vs = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) vs += exp2f((f[e] - m) * c);
        acc.add(vs);
      }
    }
  }

  float zmax = vmax;
  int amax = imax;
  block_argmax<NT>(zmax, amax, sh_v, sh_i);

  RowStat st;
  st.zmax = zmax;
  st.argmax = amax;
  st.key_k = 0u;
  st.idx_k = INT_MAX;
  st.S = 0.0;

  if constexpr (!GREEDY && !TOPK) {
    const double part = m == -INFINITY ? 0.0 : acc.value() * (double)exp2f((m - zmax) * c);
    st.S = block_sum_d<NT>(part, sh_d);
  }

  if constexpr (TOPK) {
    __shared__ uint32_t gmax[SV_MAX_TOP_K];
    __shared__ Cand cand[kMaxCand];
    __shared__ unsigned n_cand;
    __shared__ uint32_t tau_sh;
    const int k = p.top_k;
    for (int g = tid; g < k; g += NT) gmax[g] = 0u;
    if (tid == 0) n_cand = 0u, tau_sh = 0xFFFFFFFFu;
    __syncthreads();
    // k disjoint groups of units; the smallest group maximum bounds the k-th largest
#pragma unroll
    for (int u = 0; u < 2; ++u) atomicMax(&gmax[(2 * tid + u) % k], umax[u]);
    __syncthreads();
    for (int g = tid; g < k; g += NT) atomicMin(&tau_sh, gmax[g]);
    __syncthreads();
    const uint32_t tau = tau_sh;
    // gather the entries at or above tau
    for (int v = tid; v < nvec; v += NT) {
      const uint4 raw = __ldg(xv + v);
      float f[VEC];
      Elem<T>::unpack(raw, f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        if (Elem<T>::key(f[e]) >= tau) {
          const unsigned slot = atomicAdd(&n_cand, 1u);
          if (slot < kMaxCand) cand[slot] = Cand{f[e], v * VEC + e};
        }
      }
    }
    __syncthreads();
    const unsigned nc = n_cand;
    if (nc <= kMaxCand) {
      // rank every candidate: entries beating it (larger value, or equal and lower id)
      __shared__ uint32_t thr_key;
      __shared__ int thr_idx;
      double part = 0.0;
      for (unsigned i = tid; i < nc; i += NT) {
        const Cand ci = cand[i];
        unsigned rank = 0;
        for (unsigned j = 0; j < nc; ++j) {
          const Cand cj = cand[j];
          rank += (cj.z > ci.z || (cj.z == ci.z && cj.idx < ci.idx)) ? 1u : 0u;
        }
        if (rank < (unsigned)k) part += (double)exp2f((ci.z - zmax) * c);
        if (rank == (unsigned)k - 1u) thr_key = Elem<T>::key(ci.z), thr_idx = ci.idx;
      }
      __syncthreads();
      st.key_k = thr_key;
      st.idx_k = thr_idx;
      st.S = block_sum_d<NT>(part, sh_d);
    } else {
      // many equal values near the top: find the threshold key bit by bit with counting
      // passes, then the index cut among entries equal to it, then the kept sum
      uint32_t K = 0u;
      for (int bit = Elem<T>::kKeyBits - 1; bit >= 0; --bit) {
        const uint32_t cand_key = K | (1u << bit);
        unsigned cnt = 0;
        for (int v = tid; v < nvec; v += NT) {
          float f[VEC];
          Elem<T>::unpack(__ldg(xv + v), f);
#pragma unroll
          for (int e = 0; e < VEC; ++e) cnt += Elem<T>::key(f[e]) >= cand_key ? 1u : 0u;
        }
        cnt = block_sum_u<NT>(cnt, sh_u);
        if (cnt >= (unsigned)k) K = cand_key;
      }
      unsigned gt = 0;
      for (int v = tid; v < nvec; v += NT) {
        float f[VEC];
        Elem<T>::unpack(__ldg(xv + v), f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) gt += Elem<T>::key(f[e]) > K ? 1u : 0u;
      }
      gt = block_sum_u<NT>(gt, sh_u);
      const unsigned need = (unsigned)k - gt;  // >= 1 entries equal to K, lowest ids first
      // contiguous chunks per thread so that a block scan follows index order
      const int per = (nvec + NT - 1) / NT;
      const int v0 = tid * per, v1 = min(nvec, v0 + per);
      unsigned eq = 0;
      for (int v = v0; v < v1; ++v) {
        float f[VEC];
        Elem<T>::unpack(__ldg(xv + v), f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) eq += Elem<T>::key(f[e]) == K ? 1u : 0u;
      }
      __shared__ unsigned scan[NT];
      __shared__ int idx_sh;
      scan[tid] = eq;
      __syncthreads();
      if (tid == 0) {
        unsigned run = 0;
        for (int t = 0; t < NT; ++t) {
          const unsigned cnt = scan[t];
          scan[t] = run;
          run += cnt;
        }
      }
      __syncthreads();
      const unsigned before = scan[tid];
      if (before < need && before + eq >= need) {
        unsigned seen = before;
        for (int v = v0; v < v1; ++v) {
          float f[VEC];
          Elem<T>::unpack(__ldg(xv + v), f);
          bool done = false;
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            if (!done && Elem<T>::key(f[e]) == K && ++seen == need) {
              idx_sh = v * VEC + e;
              done = true;
            }
          }
          if (done) break;
        }
      }
      __syncthreads();
      st.key_k = K;
      st.idx_k = idx_sh;
      KahanF s2;
      for (int v = tid; v < nvec; v += NT) {
        float f[VEC];
        Elem<T>::unpack(__ldg(xv + v), f);
        float vs = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          vs += kept<T>(f[e], v * VEC + e, st) ? exp2f((f[e] - zmax) * c) : 0.f;
        s2.add(vs);
      }
      st.S = block_sum_d<NT>(s2.value(), sh_d);
    }
  }

  if (tid == 0) p.stats[row] = st;
}

// ------------------------------------------------------------ kernel 2

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kSelThreads) accept_select_kernel(const AcceptParams p) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NW = kSelThreads / 32;
  __shared__ int8_t s_par[kMaxNodes], s_dep[kMaxNodes], s_hc[kMaxNodes];
  __shared__ uint8_t s_acc[kMaxNodes], s_dnear[kMaxNodes];
  __shared__ int s_best, s_nd;
  __shared__ double seg_sum[NW];
  __shared__ int s_wstar, s_tok, s_snear, s_found;
  __shared__ double s_base, s_t;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int N = p.tree.N, V = p.V;
  if (tid < kMaxNodes) {
    s_par[tid] = p.tree.parent[tid];
    s_dep[tid] = p.tree.depth[tid];
    s_hc[tid] = p.tree.has_child[tid];
    s_acc[tid] = 0;
    s_dnear[tid] = 0;
  }
  __syncthreads();

  const RowStat *tstat = p.stats + (size_t)b * N;
  const RowStat *qstat = p.stats + (size_t)p.B * N + (size_t)b * p.Dq;
  const double temp = (double)p.temperature;

  // decisions, one thread per non-root node
  if (tid >= 1 && tid < N) {
    const int cnode = tid, a = s_par[cnode], d = s_dep[cnode];
    const int xt = p.tokens[(size_t)b * p.tok_stride + cnode - p.tok_offset];
    uint8_t acc = 0, dn = 0;
    if (xt < 0 || xt >= V) {
      set_status(p.status, SV_DEV_BAD_TOKEN);
    } else if (GREEDY) {
      acc = xt == tstat[a].argmax;
    } else {
      const RowStat sa = tstat[a];
      const float zp = Elem<T>::load(row_ptr<T>(p.target, (size_t)b * N + a, V) + xt);
      const double pp = kept<T>(zp, xt, sa) ? exp(((double)zp - (double)sa.zmax) / temp) / sa.S : 0.0;
      double qq;
      if (p.q_kind == SV_Q_LOGITS) {
        const RowStat sq = qstat[d - 1];
        const float zq = Elem<T>::load(row_ptr<T>(p.q, (size_t)b * p.Dq + d - 1, V) + xt);
        qq = kept<T>(zq, xt, sq) ? exp(((double)zq - (double)sq.zmax) / temp) / sq.S : 0.0;
      } else {
        qq = (double)(static_cast<const float *>(p.q)[((size_t)b * p.Dq + d - 1) * V + xt]);
      }
      double ratio;
      if (qq > 0.0) {
        ratio = pp / qq;
      } else {
        set_status(p.status, SV_DEV_ZERO_DRAFT_PROB);
        ratio = pp > 0.0 ? INFINITY : 0.0;
      }
      double u_acc, u_smp;
      verify_uniforms(p.seed, p.round, b, cnode, &u_acc, &u_smp);
      acc = u_acc < ratio;
      dn = fabs(u_acc - ratio) < kNearTie;
    }
    s_acc[cnode] = acc;
    s_dnear[cnode] = dn;
  }
  __syncthreads();

  if (tid == 0) {
    uint8_t ok[kMaxNodes];
    ok[0] = 1;
    int best = 0, nd = 0;
    for (int cn = 1; cn < N; ++cn) {
      const int a = s_par[cn];
      ok[cn] = ok[a] && s_acc[cn];
      if (ok[a] && s_dnear[cn]) ++nd;
      if (ok[cn] && s_dep[cn] > s_dep[best]) best = cn;
    }
    s_best = best;
    s_nd = nd;
    s_snear = 0;
    s_tok = -1;
  }
  __syncthreads();
  const int best = s_best;

  if constexpr (GREEDY) {
    if (tid == 0) s_tok = tstat[best].argmax;
  } else {
    // final sample: w = [p_best - q_{d+1}]+ if best has children, else p_best
    const RowStat sp = tstat[best];
    const uint4 *pv = reinterpret_cast<const uint4 *>(row_ptr<T>(p.target, (size_t)b * N + best, V));
    bool use_q = s_hc[best] != 0;
    const int qrow = s_dep[best];  // q row of depth d+1
    RowStat sq{};
    const uint4 *qv = nullptr;
    if (use_q) {
      if (p.q_kind == SV_Q_LOGITS) {
        sq = qstat[qrow];
        qv = reinterpret_cast<const uint4 *>(row_ptr<T>(p.q, (size_t)b * p.Dq + qrow, V));
      } else {
        qv = reinterpret_cast<const uint4 *>(static_cast<const float *>(p.q) +
                                             ((size_t)b * p.Dq + qrow) * V);
      }
    }
    const float c = p.c_log2;
    const float inv_sp = (float)(1.0 / sp.S);
    const float inv_sq = use_q && p.q_kind == SV_Q_LOGITS ? (float)(1.0 / sq.S) : 0.f;
    const int nvec = V / VEC;
    const int seg = (nvec + NW - 1) / NW;
    const int s0 = min(nvec, warp * seg), s1 = min(nvec, s0 + seg);
    const bool q_probs = p.q_kind == SV_Q_PROBS_F32;

    // weights of the VEC entries of vector v
    auto weights = [&](int v, float w[VEC], bool with_q) {
      float f[VEC];
      Elem<T>::unpack(__ldg(pv + v), f);
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        w[e] = kept<T>(f[e], v * VEC + e, sp) ? exp2f((f[e] - sp.zmax) * c) * inv_sp : 0.f;
      if (with_q) {
        float g[VEC];
        if (q_probs) {
          // float32 probabilities: a 16-byte vector holds 4, VEC may be 8
#pragma unroll
          for (int h = 0; h < VEC / 4; ++h) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                                        static_cast<const float *>(p.q) +
                                        ((size_t)b * p.Dq + qrow) * V) +
                                    (size_t)v * (VEC / 4) + h);
            g[4 * h] = __uint_as_float(raw.x);
            g[4 * h + 1] = __uint_as_float(raw.y);
            g[4 * h + 2] = __uint_as_float(raw.z);
            g[4 * h + 3] = __uint_as_float(raw.w);
          }
        } else {
          float fq[VEC];
          Elem<T>::unpack(__ldg(qv + v), fq);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            g[e] = kept<T>(fq[e], v * VEC + e, sq) ? exp2f((fq[e] - sq.zmax) * c) * inv_sq : 0.f;
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = fmaxf(w[e] - g[e], 0.f);
      }
    };

    double u_acc, u_smp;
    verify_uniforms(p.seed, p.round, b, best, &u_acc, &u_smp);

    for (int attempt = 0; attempt < 2; ++attempt) {
      // phase 1: per-warp segment sums (lanes interleave, Kahan per lane)
      KahanF ls;
      for (int v = s0 + lane; v < s1; v += 32) {
        float w[VEC];
        weights(v, w, use_q);
        float vs = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) vs += w[e];
        ls.add(vs);
      }
      const double wsum = warp_sum_d(ls.value());
      if (lane == 0) seg_sum[warp] = wsum;
      __syncthreads();
      if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < NW; ++w) total += seg_sum[w];
        if (!(total > 0.0)) {
          s_wstar = -1;  // residual has no mass: sample from p instead (reported)
        } else {
          const double t = u_smp * total;
          double run = 0.0;
          int ws = -1, last = -1;
          double last_base = 0.0;
          for (int w = 0; w < NW; ++w) {
            if (seg_sum[w] > 0.0) last = w, last_base = run;
            if (ws < 0 && run + seg_sum[w] > t) {
              ws = w;
              s_base = run;
            }
            run += seg_sum[w];
          }
          if (ws < 0) {  // rounding put t at the very end: last segment with mass
            ws = last;
            s_base = last_base;
          }
          s_wstar = ws;
          s_t = t;
        }
      }
      __syncthreads();
      if (s_wstar >= 0 || attempt == 1) break;
      use_q = false;
      if (tid == 0) s_snear = 1;
      __syncthreads();
    }

    // phase 2: the owning warp walks its segment in index order
    if (warp == s_wstar) {
      const double t = s_t;
      double base = s_base;
      int found = 0, tok = -1, near = 0, last_pos = -1;
      for (int v0 = s0; v0 < s1 && !found; v0 += 32) {
        const int v = v0 + lane;
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = 0.f;
        if (v < s1) weights(v, w, use_q);
        float lsum = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          lsum += w[e];
          if (w[e] > 0.f) last_pos = v * VEC + e;
        }
        double incl = (double)lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, base + incl > t);
        if (hit) {
          const int L = __ffs(hit) - 1;
          if (lane == L) {
            double cum = base + incl - (double)lsum;
            int j = -1, lastp = -1;
            for (int e = 0; e < VEC; ++e) {
              if (w[e] <= 0.f) continue;
              const double prev = cum;
              cum += (double)w[e];
              lastp = v * VEC + e;
              if (cum > t) {
                j = v * VEC + e;
                near = (t - prev < kNearTie) || (cum - t < kNearTie);
                break;
              }
            }
            if (j < 0) j = lastp, near = 1;
            tok = j;
          }
          tok = __shfl_sync(0xFFFFFFFFu, tok, L);
          near = __shfl_sync(0xFFFFFFFFu, near, L);
          found = 1;
        }
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (!found) {
        int lp = last_pos;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xFFFFFFFFu, lp, o));
        tok = lp;
        near = 1;
      }
      if (lane == 0) {
        s_tok = tok;
        s_snear |= near;
      }
    }
  }
  __syncthreads();

  if (tid == 0) {
    const int W = p.tree.Dmax + 1;
    const int depth = s_dep[best];
    int32_t *tk = p.out_tokens + (size_t)b * W;
    int32_t *pn = p.out_path_nodes ? p.out_path_nodes + (size_t)b * W : nullptr;
    for (int i = 0; i < W; ++i) {
      tk[i] = -1;
      if (pn) pn[i] = -1;
    }
    for (int a = best, i = depth; a >= 0; a = s_par[a], --i) {
      if (pn) pn[i] = a;
      if (i >= 1) tk[i - 1] = p.tokens[(size_t)b * p.tok_stride + a - p.tok_offset];
    }
    tk[depth] = s_tok;
    p.out_num_emitted[b] = depth + 1;
    p.out_num_accepted[b] = depth;
    if (p.out_near_ties) p.out_near_ties[b] = (uint32_t)(s_nd + s_snear);
  }
}

template <typename T>
cudaError_t launch_typed(const AcceptParams &p, cudaStream_t s) {
  const bool greedy = p.mode == SV_GREEDY;
  const bool topk = !greedy && p.top_k > 0 && p.top_k < p.V;
  const int rows = p.B * p.N + ((!greedy && p.q_kind == SV_Q_LOGITS) ? p.B * p.Dq : 0);
  if (greedy)
    accept_stats_kernel<T, true, false><<<rows, kStatThreads, 0, s>>>(p);
  else if (topk)
    accept_stats_kernel<T, false, true><<<rows, kStatThreads, 0, s>>>(p);
  else
    accept_stats_kernel<T, false, false><<<rows, kStatThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (greedy)
    accept_select_kernel<T, true><<<p.B, kSelThreads, 0, s>>>(p);
  else
    accept_select_kernel<T, false><<<p.B, kSelThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t accept_ws_bytes(int B, int N, int Dq) {
  return (size_t)B * (size_t)(N + Dq) * sizeof(RowStat);
}

cudaError_t launch_accept(sv_dtype dt, const AcceptParams &p, cudaStream_t s) {
  return dt == SV_F32 ? launch_typed<float>(p, s) : launch_typed<bf16>(p, s);
}

}  // namespace sv
