// Token acceptance over the vocabulary (sm_103a).
//
// Method (hncyxsy.com sections 2.1-2.2; jennyma11 blog, "先弄清无损验证" and "Medusa";
// qwbw.cn section 2.3): a draft x checked against target row p and draft row q is
// accepted iff u_acc < p(x)/q(x); at the first rejection the next token is drawn from
// norm([p - q]+); if every draft passes, a bonus token is drawn from the target's next
// row; p and q are the effective distributions (temperature, top-k, then top-p within
// the top k).  Greedy accepts while the draft is the target's argmax.  For a tree every
// node is decided against its parent's row and the q row of its depth; the deepest node
// whose root path is all accepted is kept.
//
// Kernel 1 (one CTA per logit row, target rows then q rows): one coalesced pass of
// 16-byte loads gives the row max / argmax and, without top-k, the softmax sum by a
// per-thread online accumulation.  With top-k, the pass also keeps packed unit maxima
// and one key per batch of loads; the batches that can hold an entry of the top k (a
// maximum at or above the smallest of k group maxima) are re-read as one list, their
// candidates ranked and the kept ones summed; top-p cuts the ranked list by cumulative
// mass.
// Kernel 2 (one cluster of CTAs per sequence): per-node ratios from the row statistics
// and the two logits of the candidate, the longest accepted path, and the final sample:
// a pass summing w = [p - q]+ (or p) per chunk of 32 vectors over each CTA's slice of
// the vocabulary (long slices streamed through a shared-memory ring of bulk copies),
// slice totals exchanged through distributed shared memory, then one warp of the CTA
// whose slice holds the target finds the chunk and, in it, the inverse-CDF token.
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>

#include "sv_common.cuh"
#include "row_stat.cuh"
#include "sv_internal.h"
#include "tc_primitives.cuh"

namespace sv {

namespace {

// Threads per row of the statistics kernel: 256, four CTAs per SM, so that a batch's rows
// are in flight together and one row's top-k work overlaps the others' reads (with top-k
// each thread keeps 4 units, enough groups for k up to SV_MAX_TOP_K).
template <bool TOPK>
__host__ __device__ constexpr int stat_threads() { return 256; }
constexpr int kSelThreads = 256;  // two CTAs per SM
constexpr int kMaxCand = 2048;
// Batches (of 4 vectors per thread) whose maximum the top-k statistics remember: rows of up
// to 32 * 256 * 4 * 8 = 262,144 bf16 entries; later batches are always re-read.
constexpr int kMaxTopkBatches = 32;
// Batches the top-k gather lists for its cooperative re-read (else each thread re-reads
// its own).
constexpr int kMaxGatherList = 2048;
constexpr double kNearTie = 1e-6;
// weight of one sample-class near tie in the packed near-tie word (decision ties count 1)
constexpr uint32_t kSampleTie = 65536u;
constexpr float kNearTieF = 1e-6f;

// ------------------------------------------------- float-pair arithmetic
//
// FP64 instructions have a latency of hundreds of cycles on this part, so the running
// sums and prefixes that need more than float precision (the inverse-CDF search) carry
// a value as an unevaluated sum hi + lo of two floats (Knuth's TwoSum, then a
// renormalising Fast2Sum): about 2^-44 relative, from a few FP32 operations.
// 8-byte aligned: a pair is read from a peer CTA's shared memory as one 64-bit load
// (ld.shared::cluster.v2.f32), which faults on a 4-byte boundary
struct __align__(8) F2 {
  float hi, lo;
};
static_assert(sizeof(F2) == 8 && alignof(F2) == 8, "one 64-bit word per pair");
__device__ __forceinline__ F2 f2(float x) { return F2{x, 0.f}; }
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  float e = (a.hi - (s - bb)) + (b.hi - bb);  // exact error of s
  e += a.lo + b.lo;
  const float hi = s + e;
  return F2{hi, e - (hi - s)};
}
__device__ __forceinline__ F2 f2_add(F2 a, float b) { return f2_add(a, f2(b)); }
__device__ __forceinline__ F2 f2_neg(F2 a) { return F2{-a.hi, -a.lo}; }
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) { return f2_add(a, f2_neg(b)); }
// a > b for normalised pairs
__device__ __forceinline__ bool f2_gt(F2 a, F2 b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ float f2_val(F2 a) { return a.hi + a.lo; }
// (k + 0.5) * 2^-24 * t for a 24-bit k: k * 2^-24 and 2^-25 are exact floats, and the
// product k * 2^-24 * t.hi is split exactly with an FMA
__device__ __forceinline__ F2 f2_uniform_times(uint32_t k, F2 t) {
  const float uh = (float)k * (1.f / 16777216.f);
  const float p = uh * t.hi;
  const float pe = fmaf(uh, t.hi, -p);
  return f2_add(F2{p, 0.f}, f2_add(f2(pe), f2(fmaf(uh, t.lo, t.hi * (1.f / 33554432.f)))));
}
__device__ __forceinline__ F2 shfl_up_f2(F2 v, int o) {
  return F2{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
}
__device__ __forceinline__ F2 shfl_f2(F2 v, int src) {
  return F2{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}
__device__ __forceinline__ F2 shfl_xor_f2(F2 v, int o) {
  return F2{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
}

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

// Block sum of per-thread float partials: a butterfly of float additions whose rounding
// errors (TwoSum, exact) are summed alongside, within each warp and then over the warp
// totals.  Every thread gets the result.
__device__ __forceinline__ void warp_sum_c(float &v, float &c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const float yc = __shfl_xor_sync(0xFFFFFFFFu, c, o);
    const float s = v + y;
    const float bb = s - v;
    const float e = (v - (s - bb)) + (y - bb);
    v = s;
    c = (c + yc) + e;
  }
}
template <int NT>
__device__ float block_sum_f(float v, float *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float c = 0.f;
  warp_sum_c(v, c);
  if (lane == 0) sh[warp] = v, sh[NT / 32 + warp] = c;
  __syncthreads();
  if (warp == 0) {
    float w = lane < NT / 32 ? sh[lane] : 0.f, wc = lane < NT / 32 ? sh[NT / 32 + lane] : 0.f;
    warp_sum_c(w, wc);
    if (lane == 0) sh[2 * (NT / 32)] = w + wc;
  }
  __syncthreads();
  const float r = sh[2 * (NT / 32)];
  __syncthreads();
  return r;
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

// Largest entry of one 16-byte vector (bf16: packed maxima, exact).
template <typename T>
__device__ __forceinline__ float vec_max(const uint4 &r) {
  if constexpr (Elem<T>::kVec == 8) {
    const uint32_t hm = max_bf16x2(max_bf16x2(r.x, r.y), max_bf16x2(r.z, r.w));
    return fmaxf(__uint_as_float(hm << 16), __uint_as_float(hm & 0xFFFF0000u));
  } else {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
}

// ------------------------------------------------------------ kernel 1

// Statistics of one logit row (all NT threads of the CTA): row max and its lowest index,
// the top-k threshold, and the softmax sum over the kept entries.  Thread 0 writes
// p.stats[row].  Rows 0..B*N-1 are target rows, then the q rows.
template <typename T, bool GREEDY, bool TOPK, int NT, bool ENT = false>
__device__ void row_stats(const AcceptParams &p, size_t row) {
  constexpr int VEC = Elem<T>::kVec;
  __shared__ float sh_v[32];
  __shared__ int sh_i[32];
  __shared__ float sh_d[2 * (NT / 32) + 1];
  __shared__ unsigned sh_u[32];
  __syncthreads();  // the shared scratch may still be read for the previous row

  const int tid = threadIdx.x;
  const size_t nt_rows = (size_t)p.B * p.N;
  const T *x = row < nt_rows ? row_ptr<T>(p.target, row, p.V)
                             : row_ptr<T>(p.q, row - nt_rows, p.V);
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  const int nvec = p.V / VEC;
  const float c = p.c_log2;

  float vmax = -INFINITY;
  int imax = INT_MAX;
  float m = -INFINITY;  // running maximum the partial sum is taken against
  KahanF acc;
  KahanF ent;  // ENT: sum of 2^t t, t = (z - m) c (the entropy's second term)
  // TOPK: the maxima of this thread's 4 units (fp32: units = element lanes 0..3 of each
  // vector; bf16: the low and high halves of words x, z and of words y, w, kept as two
  // packed pairs), and the top 16 bits of the key of each batch's maximum, so that the
  // gather re-reads only the batches that can hold an entry of the top k
  uint32_t umax[4] = {0u, 0u, 0u, 0u};
  uint32_t umw[2] = {Elem<T>::kNegInfWord, Elem<T>::kNegInfWord};
  constexpr int kKeyShift = Elem<T>::kKeyBits - 16;
  __shared__ uint16_t s_bkey[TOPK ? kMaxTopkBatches * NT : 1];

  // each thread takes vectors tid, tid + NT, ... in index order, four at a time; the
  // next four are loaded while the current four are worked on (two batches in flight);
  // vectors past the end read as -inf
  constexpr int U = 4;
  const uint4 ninf = make_uint4(Elem<T>::kNegInfWord, Elem<T>::kNegInfWord,
                                Elem<T>::kNegInfWord, Elem<T>::kNegInfWord);
  auto load_batch = [&](int v0, uint4 (&r)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = v0 + u * NT < nvec ? __ldg(xv + v0 + u * NT) : ninf;
  };
  uint4 nxt[U];
  load_batch(tid, nxt);
  for (int v0 = tid, jb = 0; v0 < nvec; v0 += NT * U, ++jb) {
    uint4 raws[U];
#pragma unroll
    for (int u = 0; u < U; ++u) raws[u] = nxt[u];
    if (v0 + NT * U < nvec) load_batch(v0 + NT * U, nxt);
    float f[U][VEC];
#pragma unroll
    for (int u = 0; u < U; ++u) Elem<T>::unpack(raws[u], f[u]);
    // the batch maximum first; the index scan runs only when it beats the running max
    // (bf16: lane-wise maxima of the packed words, exact)
    float mx;
    if constexpr (VEC == 8) {
      uint32_t h0 = max_bf16x2(raws[0].x, raws[0].z), h1 = max_bf16x2(raws[0].y, raws[0].w);
#pragma unroll
      for (int u = 1; u < U; ++u) {
        h0 = max_bf16x2(h0, max_bf16x2(raws[u].x, raws[u].z));
        h1 = max_bf16x2(h1, max_bf16x2(raws[u].y, raws[u].w));
      }
      const uint32_t hm = max_bf16x2(h0, h1);
      mx = fmaxf(__uint_as_float(hm << 16), __uint_as_float(hm & 0xFFFF0000u));
      if constexpr (TOPK) {
        umw[0] = max_bf16x2(umw[0], h0);
        umw[1] = max_bf16x2(umw[1], h1);
      }
    } else {
      mx = f[0][0];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < VEC; ++e) mx = fmaxf(mx, f[u][e]);
    }
    if constexpr (TOPK)
      if (jb < kMaxTopkBatches) s_bkey[jb * NT + tid] = (uint16_t)(Elem<T>::key(mx) >> kKeyShift);
    if (mx > vmax) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (f[u][e] > vmax) vmax = f[u][e], imax = (v0 + u * NT) * VEC + e;
    }
    if constexpr (TOPK && VEC != 8) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (v0 + u * NT < nvec)
#pragma unroll
          for (int e = 0; e < VEC; ++e) umax[e & 3] = max(umax[e & 3], Elem<T>::key(f[u][e]));
    }
    if constexpr (!GREEDY && !TOPK) {
      if (vmax > m) {  // vmax: the largest value this thread has seen
        if (m != -INFINITY) {
          const float sc = ex2_approx((m - vmax) * c);
          if constexpr (ENT) {
            // sum 2^(t - d) (t - d) = 2^-d (sum 2^t t - d sum 2^t), d = (vmax - m) c
            const float d = (vmax - m) * c;
            ent.s = sc * (ent.value() - d * acc.value());
            ent.c = 0.f;
          }
          acc.s *= sc;
          acc.c *= sc;
        }
        m = vmax;
      }
      if (m != -INFINITY) {
        // partial sums ps[e & 3] in lane pairs: (z - m) * c and the sums as packed f32x2
        // (the same roundings and order as the scalar form)
        float2 ps01 = make_float2(0.f, 0.f), ps23 = make_float2(0.f, 0.f);
        float es = 0.f;  // ENT: this batch's sum of 2^t t (2^-inf * -inf counts as 0)
        const float2 m2 = make_float2(m, m), c2 = make_float2(c, c);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 t = mul2(sub2(make_float2(f[u][e], f[u][e + 1]), m2), c2);
            const float2 x = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            if (e & 2) ps23 = add2(ps23, x);
            else ps01 = add2(ps01, x);
            if constexpr (ENT) {
              if (x.x > 0.f) es = fmaf(x.x, t.x, es);
              if (x.y > 0.f) es = fmaf(x.y, t.y, es);
            }
          }
        acc.add((ps01.x + ps01.y) + (ps23.x + ps23.y));
        if constexpr (ENT) ent.add(es);
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
  st.S = 0.f;
  st.flags = 0u;
  st.H = 0.f;
  st.pad = 0u;

  if constexpr (!GREEDY && !TOPK) {
    const float sc = m == -INFINITY ? 0.f : exp2f((m - zmax) * c);
    const float part = m == -INFINITY ? 0.f : acc.value() * sc;
    st.S = block_sum_f<NT>(part, sh_d);
    if constexpr (ENT) {
      // to the row maximum: sum 2^(t + d) (t + d) = 2^d (sum 2^t t + d sum 2^t), d = (m - zmax) c
      const float epart = m == -INFINITY ? 0.f : sc * (ent.value() + (m - zmax) * c * acc.value());
      const float E = block_sum_f<NT>(epart, sh_d);
      // p_j = 2^t_j / S: H = -sum p ln p = ln S - ln 2 * E / S
      st.H = st.S > 0.f ? (float)(log((double)st.S) - 0.6931471805599453 * (double)E / (double)st.S) : 0.f;
    }
  }

  if constexpr (TOPK) {
    __shared__ uint32_t gmax[SV_MAX_TOP_K];
    __shared__ Cand cand[kMaxCand];
    __shared__ uint32_t s_glist[kMaxGatherList];
    __shared__ unsigned n_cand, n_glist;
    __shared__ uint32_t tau_sh;
    const int k = p.top_k;
    for (int g = tid; g < k; g += NT) gmax[g] = 0u;
    if (tid == 0) n_cand = 0u, n_glist = 0u, tau_sh = 0xFFFFFFFFu;
    __syncthreads();
    if constexpr (VEC == 8) {
      umax[0] = Elem<T>::key(__uint_as_float(umw[0] << 16));
      umax[1] = Elem<T>::key(__uint_as_float(umw[0] & 0xFFFF0000u));
      umax[2] = Elem<T>::key(__uint_as_float(umw[1] << 16));
      umax[3] = Elem<T>::key(__uint_as_float(umw[1] & 0xFFFF0000u));
    }
    // k disjoint groups of units; the smallest group maximum bounds the k-th largest
#pragma unroll
    for (int u = 0; u < 4; ++u) atomicMax(&gmax[(4 * tid + u) % k], umax[u]);
    __syncthreads();
    for (int g = tid; g < k; g += NT) atomicMin(&tau_sh, gmax[g]);
    __syncthreads();
    const uint32_t tau = tau_sh;
    // the batches whose maximum reaches tau (those past the remembered ones always), as
    // a list; then the whole CTA re-reads the listed vectors with all loads in flight
    const uint32_t tau16 = tau >> kKeyShift;
    for (int v0 = tid, jb = 0; v0 < nvec; v0 += NT * U, ++jb) {
      if (jb < kMaxTopkBatches && (uint32_t)s_bkey[jb * NT + tid] < tau16) continue;
      const unsigned slot = atomicAdd(&n_glist, 1u);
      if (slot < kMaxGatherList) s_glist[slot] = (uint32_t)(jb * NT + tid);
    }
    __syncthreads();
    const unsigned nl = n_glist;
    auto gather_vec = [&](const uint4 &raw, int v) {
      float f[VEC];
      Elem<T>::unpack(raw, f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        if (Elem<T>::key(f[e]) >= tau) {
          const unsigned slot = atomicAdd(&n_cand, 1u);
          if (slot < kMaxCand) cand[slot] = Cand{f[e], v * VEC + e};
        }
      }
    };
    if (nl <= (unsigned)kMaxGatherList) {
      // item i: vector i % U of listed batch i / U
      const int items = (int)nl * U;
      constexpr int R = 4;
      for (int i0 = tid; i0 < items; i0 += NT * R) {
        uint4 raws[R];
        int vv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int i = i0 + r * NT;
          vv[r] = -1;
          if (i < items) {
            const uint32_t e = s_glist[i / U];
            const int v = (int)(e % NT) + (int)(e / NT) * NT * U + (i % U) * NT;
            if (v < nvec) {
              vv[r] = v;
              raws[r] = __ldg(xv + v);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (vv[r] >= 0) gather_vec(raws[r], vv[r]);
      }
    } else {
      for (int v0 = tid, jb = 0; v0 < nvec; v0 += NT * U, ++jb) {
        if (jb < kMaxTopkBatches && (uint32_t)s_bkey[jb * NT + tid] < tau16) continue;
        uint4 raws[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * NT < nvec) raws[u] = __ldg(xv + v0 + u * NT);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + u * NT < nvec) gather_vec(raws[u], v0 + u * NT);
      }
    }
    __syncthreads();
    unsigned nc = n_cand;
    if (nc > (unsigned)kMaxCand) {
      // many equal values near the top: find the threshold key bit by bit with counting
      // passes and the index cut among the entries equal to it; then the kept set
      // (exactly k entries) becomes the candidate list
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
        n_cand = 0u;
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
      RowStat cut{};
      cut.key_k = K;
      cut.idx_k = idx_sh;
      for (int v = tid; v < nvec; v += NT) {
        float f[VEC];
        Elem<T>::unpack(__ldg(xv + v), f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          if (kept<T>(f[e], v * VEC + e, cut)) {
            const unsigned slot = atomicAdd(&n_cand, 1u);
            if (slot < kMaxCand) cand[slot] = Cand{f[e], v * VEC + e};
          }
        }
      }
      __syncthreads();
      nc = min(n_cand, (unsigned)kMaxCand);
    }
    {
      // rank every candidate: entries beating it (larger value, or equal and lower id);
      // each candidate's comparisons are split over tpc adjacent threads (a power of two,
      // the same in every thread), whose counts are summed by shuffles.  With top-p the
      // kept entries are also laid out by rank (in the gather list's memory).
      __shared__ uint32_t thr_key;
      __shared__ int thr_idx;
      const bool nucleus = p.top_p < 1.f;
      float *srt_z = reinterpret_cast<float *>(s_glist);
      int *srt_i = reinterpret_cast<int *>(s_glist) + SV_MAX_TOP_K;
      static_assert(2 * SV_MAX_TOP_K <= kMaxGatherList, "ranked entries fit the gather list");
      int tpc = 1;
      while (tpc < 32 && nc * (unsigned)tpc * 2u <= (unsigned)NT) tpc *= 2;
      const int per_round = NT / tpc, sub = tid & (tpc - 1);
      float part = 0.f;
      for (unsigned base = 0; base < nc; base += (unsigned)per_round) {
        const unsigned i = base + (unsigned)(tid / tpc);
        unsigned rank = 0;
        Cand ci{0.f, 0};
        if (i < nc) {
          ci = cand[i];
          unsigned j = (unsigned)sub;
          for (; j + 3u * tpc < nc; j += 4u * tpc) {
            const Cand c0 = cand[j], c1 = cand[j + tpc], c2 = cand[j + 2 * tpc], c3 = cand[j + 3 * tpc];
            rank += (c0.z > ci.z || (c0.z == ci.z && c0.idx < ci.idx)) ? 1u : 0u;
            rank += (c1.z > ci.z || (c1.z == ci.z && c1.idx < ci.idx)) ? 1u : 0u;
            rank += (c2.z > ci.z || (c2.z == ci.z && c2.idx < ci.idx)) ? 1u : 0u;
            rank += (c3.z > ci.z || (c3.z == ci.z && c3.idx < ci.idx)) ? 1u : 0u;
          }
          for (; j < nc; j += tpc) {
            const Cand cj = cand[j];
            rank += (cj.z > ci.z || (cj.z == ci.z && cj.idx < ci.idx)) ? 1u : 0u;
          }
        }
        for (int o = 1; o < tpc; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
        if (i < nc && sub == 0) {
          if (rank < (unsigned)k) {
            part += exp2f((ci.z - zmax) * c);
            if (nucleus) {
              srt_z[rank] = ci.z;
              srt_i[rank] = ci.idx;
            }
          }
          if (rank == (unsigned)k - 1u) thr_key = Elem<T>::key(ci.z), thr_idx = ci.idx;
        }
      }
      __syncthreads();
      st.key_k = thr_key;
      st.idx_k = thr_idx;
      st.S = block_sum_f<NT>(part, sh_d);
      if (nucleus) {
        // top-p within the top-k distribution: the first rank whose cumulative mass (rank
        // order, float pairs) reaches top_p of the total becomes the cut (its key and
        // index; its cumulative mass the kept sum).  A cut within 1e-6 of top_p, in
        // probability units, is reported as a near tie of the row.
        __shared__ F2 s_wtot[NT / 32];
        __shared__ int s_cut;
        __shared__ float s_cut_S;
        __shared__ unsigned s_cut_near;
        const int lane = tid & 31, warp = tid >> 5;
        const int r0 = 4 * tid;
        F2 loc[4];
        F2 tsum = f2(0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = r0 + q;
          tsum = f2_add(tsum, r < k ? exp2f((srt_z[r] - zmax) * c) : 0.f);
          loc[q] = tsum;
        }
        F2 incl = tsum;
#pragma unroll 1
        for (int o = 1; o < 32; o <<= 1) {
          const F2 y = shfl_up_f2(incl, o);
          if (lane >= o) incl = f2_add(incl, y);
        }
        if (lane == 31) s_wtot[warp] = incl;
        if (tid == 0) s_cut = k - 1, s_cut_S = st.S, s_cut_near = 0u;
        __syncthreads();
        F2 wbase = f2(0.f), tot = f2(0.f);
        for (int w2 = 0; w2 < NT / 32; ++w2) {
          if (w2 < warp) wbase = f2_add(wbase, s_wtot[w2]);
          tot = f2_add(tot, s_wtot[w2]);
        }
        const F2 tbase = f2_add(wbase, f2_sub(incl, tsum));
        const double Sk = (double)tot.hi + (double)tot.lo;
        const double target = (double)p.top_p * Sk, tol = 1e-6 * Sk;
        double prev = (double)tbase.hi + (double)tbase.lo;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = r0 + q;
          if (r >= k) break;
          const F2 cf = f2_add(tbase, loc[q]);
          const double cur = (double)cf.hi + (double)cf.lo;
          if (cur >= target && prev < target) {
            s_cut = r;
            s_cut_S = (float)cur;
            s_cut_near = (cur - target < tol || (r > 0 && target - prev < tol)) ? 1u : 0u;
          }
          prev = cur;
        }
        __syncthreads();
        const int m = s_cut;
        st.key_k = Elem<T>::key(srt_z[m]);
        st.idx_k = srt_i[m];
        st.S = s_cut_S;
        st.flags |= s_cut_near;
      }
    }
  }

  if (tid == 0) p.stats[row] = st;
}

template <typename T, bool GREEDY, bool TOPK, bool ENT = false>
__global__ void __launch_bounds__(stat_threads<TOPK>(), 4) accept_stats_kernel(const AcceptParams p) {
  // the select kernel may be scheduled now; it waits for this grid before reading the
  // statistics (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  row_stats<T, GREEDY, TOPK, stat_threads<TOPK>(), ENT>(p, (size_t)p.stat_row0 + blockIdx.x);
}

// ------------------------------------------------------------ kernel 2
//
// One thread-block cluster of C CTAs per sequence.  Every CTA takes the node decisions
// (they are cheap and identical everywhere), so all know the kept path; the final
// sample's vocabulary pass is split over the cluster: CTA r sums the weights of its
// slice in chunks of 32 vectors (kept in shared memory), the CTAs read each other's
// slice totals through distributed shared memory, and in the CTA whose slice holds
// u * total one warp finds the chunk from the chunk sums and the token inside it.
// Every CTA runs the same sequence of cluster barriers: each branch that decides a
// barrier depends only on values that all CTAs of the cluster compute alike.
// FP64 throughput is low on this part: double arithmetic is kept to a few operations
// per thread (cumulative sums across chunks, and decisions within 1e-4 of u).

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_size() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// First lane (0..n-1) whose exclusive prefix + own value exceeds t, with that prefix; if
// none does (rounding put t at the very end), the last lane with a positive value.
// Warp-wide: lane i holds x (0 for i >= n); base is added to every prefix.
__device__ __forceinline__ int warp_find_cdf(F2 x, int n, F2 base, F2 t, F2 *before_out) {
  const int lane = threadIdx.x & 31;
  F2 incl = x;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const F2 y = shfl_up_f2(incl, o);
    if (lane >= o) incl = f2_add(incl, y);
  }
  const F2 before = f2_add(base, f2_sub(incl, x));
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < n && f2_gt(f2_add(before, x), t));
  const unsigned pos = __ballot_sync(0xFFFFFFFFu, lane < n && x.hi > 0.f);
  const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  *before_out = shfl_f2(before, L < 0 ? 0 : L);
  return L;
}
// Read a float pair from the same shared-memory variable of CTA `rank` in this cluster.
__device__ __forceinline__ F2 ld_peer_f2(const F2 *local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  F2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.hi), "=f"(v.lo) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_incl_scan_f(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

constexpr int kMaxCluster = 16;

// Commit of the kept path inside the select kernel (the work of the commit kernel): the
// tree K/V rows of path nodes path[0..count) (root first) go to cache positions L..L+count-1.
// The rows' 16-byte vectors are split over the `parts` CTAs of the cluster; loads are
// issued four at a time before the stores.  Bad block ids and positions past the cache
// are reported (by CTA 0) and skipped.
__device__ void commit_path_slice(const CommitParams &cm, int b, int L, const int8_t *path,
                                  int count, unsigned part, unsigned parts) {
  const long long row_vec = (long long)cm.Hkv * cm.D * cm.esize / 16;
  const long long total = (long long)count * row_vec;
  const long long i0 = total * part / parts, i1 = total * (part + 1) / parts;
  const uint4 *__restrict__ kt = static_cast<const uint4 *>(cm.k_tree);
  const uint4 *__restrict__ vt = static_cast<const uint4 *>(cm.v_tree);
  uint4 *__restrict__ ck = static_cast<uint4 *>(cm.cache_k);
  uint4 *__restrict__ cv = static_cast<uint4 *>(cm.cache_v);
  constexpr int U = 4;
  for (long long i = i0 + threadIdx.x; i < i1; i += (long long)blockDim.x * U) {
    uint4 kk[U], vv[U];
    long long dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      dst[u] = -1;
      const long long ii = i + (long long)u * blockDim.x;
      if (ii >= i1) continue;
      const int k = (int)(ii / row_vec);
      const long long e = ii % row_vec;
      const int node = path[k], pos = L + k;
      long long dst_row;
      if (cm.block_table) {
        const int bi = pos / cm.block_size;
        const int blk = bi < cm.max_blocks ? cm.block_table[(size_t)b * cm.max_blocks + bi] : -1;
        if (blk < 0 || blk >= cm.num_blocks) {
          if (e == 0) set_status(cm.status, SV_DEV_BAD_BLOCK);
          continue;
        }
        dst_row = (long long)blk * cm.block_size + pos % cm.block_size;
      } else {
        if (pos >= cm.Lmax) {
          if (e == 0) set_status(cm.status, SV_DEV_BAD_PREFIX);
          continue;
        }
        dst_row = (long long)b * cm.Lmax + pos;
      }
      const long long src = ((long long)b * cm.N + node) * row_vec + e;
      kk[u] = kt[src];
      vv[u] = vt[src];
      dst[u] = dst_row * row_vec + e;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0) {
        ck[dst[u]] = kk[u];
        cv[dst[u]] = vv[u];
      }
  }
}
// Requests into L2 the tree K/V rows that commit_path_slice(.., part, parts) will copy.
__device__ void commit_prefetch_slice(const CommitParams &cm, int b, const int8_t *path, int count,
                                      unsigned part, unsigned parts) {
  const long long row_vec = (long long)cm.Hkv * cm.D * cm.esize / 16;
  const long long total = (long long)count * row_vec;
  const long long i0 = total * part / parts, i1 = total * (part + 1) / parts;
  const uint4 *kt = static_cast<const uint4 *>(cm.k_tree);
  const uint4 *vt = static_cast<const uint4 *>(cm.v_tree);
  // one request per 128-byte line (8 vectors) of the slice
  for (long long i = (i0 & ~7ll) + 8ll * threadIdx.x; i < i1; i += 8ll * blockDim.x) {
    const long long ii = i < i0 ? i0 : i;
    const int k = (int)(ii / row_vec);
    const long long src = ((long long)b * cm.N + path[k]) * row_vec + ii % row_vec;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kt + src));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(vt + src));
  }
}
constexpr int kMaxChunks = 2048;          // chunk sums one CTA keeps (32 vectors each)
// Without top-k, the final sample's pass streams each CTA's slice of the p and q rows
// when its slice is long, through a ring of up to kRingStages shared-memory stages of
// kRingVec vectors (as many as the slice fills), filled by bulk asynchronous copies (up to
// 96 KB with q as logits) without holding them in registers.  A stage
// has 32 chunks; warp w sums chunks w, w + 8, w + 16, w + 24 together, so that their
// reductions overlap.
constexpr int kRingVec = 1024;
constexpr int kRingStages = 3;
constexpr int kRingMinVec = 2 * kRingVec;  // slices at least this long use the ring
constexpr int kRingChunks = kRingVec / 32;                    // chunks per stage
constexpr int kChunksPerWarp = kRingChunks / (kSelThreads / 32);
static_assert(kChunksPerWarp * (kSelThreads / 32) == kRingChunks, "whole chunks per warp");

// Bytes of one ring stage: kRingVec vectors of p and the matching q (one vector of
// logits, or VEC/4 vectors of f32 probabilities, per p vector).
template <typename T>
__host__ __device__ constexpr uint32_t ring_stage_bytes(bool q_probs) {
  return (uint32_t)kRingVec * 16u * (1u + (q_probs ? (uint32_t)(Elem<T>::kVec / 4) : 1u));
}

// One-dimensional bulk copy global -> shared, completing on an mbarrier (both addresses
// 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Wait for a phase with a fresh time limit of its own (used to let copies in flight land
// after a wait gave up).  False if the limit passed.
__device__ __noinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = tc::global_ns();
  while (!tc::mbar_try_wait(bar, parity))
    if (tc::global_ns() - t0 > tc::kWaitLimitNs) return false;
  return true;
}
constexpr float kDecideMarginF = 1e-4f;   // float ratio this close to u: decide in double

// The decision of a node whose float ratio fell within kDecideMarginF of u, in double
// (out of line: it is rarely taken).  Bit 0: accepted; bit 1: |u - ratio| < kNearTie.
__device__ __noinline__ int decide_double(uint32_t k_node, float zp, RowStat sa, bool logits, float zq,
                                          RowStat sq, float qprob, float temperature) {
  const double temp = (double)temperature;
  const double u_acc = ((double)k_node + 0.5) * (1.0 / 16777216.0);
  const double pp = exp(((double)zp - (double)sa.zmax) / temp) / (double)sa.S;
  const double qq = logits ? exp(((double)zq - (double)sq.zmax) / temp) / (double)sq.S : (double)qprob;
  const double ratio = pp / qq;
  return (u_acc < ratio ? 1 : 0) | (fabs(u_acc - ratio) < kNearTie ? 2 : 0);
}

// A typical-acceptance decision (the Medusa paper's rule): p(x) > min(eps, delta exp(-H)),
// taken in double from the parent row's statistics.  Bit 0: accepted; bit 1: a near tie
// (|p(x) - threshold| within 1e-6, widened by the float error of the entropy).
__device__ __noinline__ int decide_typical(float zp, RowStat sa, float temperature, float eps,
                                           float delta) {
  const double px = exp(((double)zp - (double)sa.zmax) / (double)temperature) / (double)sa.S;
  const double H = (double)sa.H;
  const double thr = fmin((double)eps, (double)delta * exp(-H));
  const double win = kNearTie + 1e-6 * thr * (1.0 + H);
  return (px > thr ? 1 : 0) | (fabs(px - thr) < win ? 2 : 0);
}

// Decisions, path, optional commit and final sample of sequence b by the CTA of rank
// `rank` in a thread-block cluster of C CTAs that split the vocabulary pass and exchange
// their slice totals through distributed shared memory (C = 1: one CTA, no exchange).
template <typename T, bool GREEDY, bool TOPK, bool RING, int NT>
__device__ void select_seq(const AcceptParams &p, int b, unsigned rank, unsigned C) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NW = NT / 32;
  constexpr int QV = VEC / 4;  // 16-byte vectors of f32 q probabilities per VEC entries
  __shared__ int8_t s_par[kMaxNodes], s_dep[kMaxNodes], s_hc[kMaxNodes];
  __shared__ uint8_t s_acc[kMaxNodes], s_dnear[kMaxNodes], s_end[kMaxNodes];
  __shared__ int s_xtok[kMaxNodes];
  __shared__ int s_best, s_nd;
  __shared__ F2 seg_sum[NW];
  __shared__ F2 s_slice[2];  // this CTA's slice total, per attempt (read by peers)
  __shared__ float s_chunk[kMaxChunks];
  __shared__ int s_wstar, s_tok, s_snear, s_rstar;
  __shared__ F2 s_base, s_t;
  __shared__ int8_t s_path[kMaxNodes];
  // the ring of the final sample's pass (no top-k): stages in dynamic shared memory
  extern __shared__ __align__(128) uint8_t sel_ring[];
  __shared__ uint64_t ring_full[kRingStages];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.tree.N, V = p.V;
  __syncthreads();  // the shared state may still be read for the previous sequence
  if (RING && tid == 0) {
    for (int i = 0; i < kRingStages; ++i) tc::mbar_init(&ring_full[i], 1);
    tc::fence_barrier_init();
    s_abort = 0;
  }
  // sequence b's tree: the shared one, or its own row checked here (a parent outside
  // [0, c), a root that is not -1, or a node deeper than the q rows make the sequence keep
  // its root alone); every row index below is formed from these checked values
  bool bad_node = false;
  if (tid < kMaxNodes) {
    int v = -1;
    if (tid < N) {
      v = tree_parent(p.tree, b, tid);
      bad_node = tid == 0 ? v != -1 : (v < 0 || v >= tid);
      if (bad_node) v = tid == 0 ? -1 : 0;
    }
    s_par[tid] = (int8_t)v;
    s_hc[tid] = 0;
    s_acc[tid] = 0;
    s_dnear[tid] = 0;
    s_end[tid] = 0;
    s_xtok[tid] = -1;
  }
  __syncthreads();
  if (tid < N) {
    uint64_t anc_unused;
    int d = 0;
    tree_walk(s_par, tid, &anc_unused, &d);  // (s_par holds a valid tree now)
    s_dep[tid] = (int8_t)d;
    if (!GREEDY && p.q_kind != SV_Q_DRAFT_ONEHOT && d > p.Dq) bad_node = true;
    if (tid > 0) s_hc[s_par[tid]] = 1;
  }
  const bool seq_bad = __syncthreads_or(bad_node) != 0;
  if (seq_bad) {
    // not a usable tree: keep the root alone (no decisions; the bonus from the root row)
    if (tid < kMaxNodes) s_hc[tid] = 0;
    if (tid == 0 && rank == 0) set_status(p.status, SV_DEV_BAD_TREE);
    __syncthreads();
  }

  const RowStat *tstat = p.stats + (size_t)b * N;
  const RowStat *qstat = p.stats + (size_t)p.B * N + (size_t)b * p.Dq;

  // Inputs that do not come from the statistics kernel are read before waiting for it:
  // the candidate token of each non-root node, the two logits at it (the parent's target
  // row, the q row of the node's depth), its uniforms, and the cache length for the commit.
  const bool has_node = tid >= 1 && tid < N && !seq_bad;
  const int cnode = tid, a_par = has_node ? s_par[cnode] : 0, d_node = has_node ? s_dep[cnode] : 1;
  const int xt = has_node ? p.tokens[(size_t)b * p.tok_stride + cnode - p.tok_offset] : -1;
  const bool tok_ok = xt >= 0 && xt < V;
  // a chain's draft of -1: this sequence has fewer drafts (no decision, no status)
  const bool absent = has_node && p.chain_end && xt == -1;
  const bool logits = p.q_kind == SV_Q_LOGITS;
  const bool onehot = p.q_kind == SV_Q_DRAFT_ONEHOT;  // q(x) = 1 at the draft token
  float zp = 0.f, zq = 0.f, qprob = 0.f;
  uint32_t k_node = 0u, k_unused = 0u;
  if (GREEDY && p.typical && has_node && tok_ok)  // typical acceptance: the parent's p(x)
    zp = Elem<T>::load(row_ptr<T>(p.target, (size_t)b * N + a_par, V) + xt);
  if (!GREEDY && has_node && tok_ok) {
    zp = Elem<T>::load(row_ptr<T>(p.target, (size_t)b * N + a_par, V) + xt);
    if (logits)
      zq = Elem<T>::load(row_ptr<T>(p.q, (size_t)b * p.Dq + d_node - 1, V) + xt);
    else if (onehot)
      qprob = 1.f;
    else
      qprob = static_cast<const float *>(p.q)[((size_t)b * p.Dq + d_node - 1) * V + xt];
    verify_uniform_ints(p.seed, p.round, b, cnode, &k_node, &k_unused);
  }
  if (has_node) {
    s_end[cnode] = absent ? 1 : 0;
    s_xtok[cnode] = xt;
  }
  const int commit_L = p.commit ? p.cm.prefix_len[b] : -1;

  // the row statistics come from the previous kernel (launched as its programmatic
  // dependent): wait for that grid and its memory
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Threads of a warp took different branches above (the root has no node): reconverge
  // them here, before the warp-wide work that follows.  (Left diverged, later full-warp
  // shuffles were measured to cost several hundred cycles each.)
  __syncwarp();
  // a row of this sequence whose top-p cut was a near tie counts as one near tie
  int nuc = 0;
  if (!GREEDY && p.top_p < 1.f) {
    if (tid < N) nuc = (int)(__ldcg(&tstat[tid].flags) & 1u);
    else if (logits && tid < N + p.Dq) nuc = (int)(__ldcg(&qstat[tid - N].flags) & 1u);
  }
  const int nuc_near = __syncthreads_or(nuc) ? 1 : 0;

  // decisions, one thread per non-root node: accept iff u_acc < p(x)/q(x).  The ratio
  // and u are formed in float; when the ratio falls within kDecideMargin (relative) of u
  // both are recomputed in double, so every decision is the one double precision takes.
  if (has_node) {
    const int a = a_par, d = d_node;
    uint8_t acc = 0, dn = 0;
    if (!tok_ok) {
      if (rank == 0 && !absent) set_status(p.status, SV_DEV_BAD_TOKEN);
    } else if (GREEDY) {
      if (p.typical) {
        const int r = decide_typical(zp, load_stat(tstat + a), p.temperature, p.typ_eps, p.typ_delta);
        acc = r & 1;
        dn = r >> 1;
      } else {
        acc = xt == __ldcg(&tstat[a].argmax);
      }
    } else {
      // u = (k + 0.5) 2^-24 in float (within 2^-25; exact for the k near kNearTie)
      const float u_f = ((float)k_node + 0.5f) * (1.f / 16777216.f);
      const RowStat sa = load_stat(tstat + a);
      const bool kp = kept<T>(zp, xt, sa);
      RowStat sq{};
      bool kq = true;
      if (logits) {
        sq = load_stat(qstat + (d - 1));
        kq = kept<T>(zq, xt, sq);
      }
      const bool q_zero = logits ? !kq : !(qprob > 0.f);
      if (q_zero) {
        if (rank == 0) set_status(p.status, SV_DEV_ZERO_DRAFT_PROB);
        acc = kp;  // ratio +inf when p > 0, else 0
      } else if (!kp) {
        acc = 0;  // ratio 0
        dn = u_f < kNearTieF;
      } else {
        const float cf = p.c_log2;
        float rf;
        if (logits)
          rf = exp2f(((zp - sa.zmax) - (zq - sq.zmax)) * cf) * (sq.S / sa.S);
        else
          rf = exp2f((zp - sa.zmax) * cf) / (sa.S * qprob);
        if (fabsf(u_f - rf) > kDecideMarginF * (1.f + rf)) {
          acc = u_f < rf;
        } else {
          const int r = decide_double(k_node, zp, sa, logits, zq, sq, qprob, p.temperature);
          acc = r & 1;
          dn = r >> 1;
        }
      }
    }
    s_acc[cnode] = acc;
    s_dnear[cnode] = dn;
  }
  __syncwarp();
  __syncthreads();

  // the kept path: node c is on it iff c and all its ancestors were accepted (the root
  // always is); best = the deepest such node, lowest index among equals.  Threads
  // 0..63 take one node each: ancestor masks from the parent chain, then ballots.
  if (tid == 0) {
    s_best = 0;
    s_nd = 0;
    s_snear = 0;
    s_tok = -1;
    s_wstar = -1;
    s_rstar = -1;
  }
  __syncthreads();
  if (tid < kMaxNodes) {
    const bool live = tid < N;
    uint64_t anc = 0;
    if (live)
      for (int a = tid; a >= 0; a = s_par[a]) anc |= 1ull << a;
    const bool acc_self = tid == 0 || (live && s_acc[tid]);
    const unsigned w = __ballot_sync(0xFFFFFFFFu, acc_self);
    __shared__ unsigned s_accw[2];
    if (lane == 0) s_accw[warp] = w;
    // both warps' ballots are needed: warps 0 and 1 meet at a named barrier
    asm volatile("bar.sync 1, 64;" ::: "memory");
    const uint64_t accm = (uint64_t)s_accw[0] | ((uint64_t)s_accw[1] << 32);
    const bool ok = live && (anc & ~accm) == 0;
    const bool ok_par = live && tid > 0 && ((anc & ~(1ull << tid)) & ~accm) == 0;
    if (ok) atomicMax(&s_best, (s_dep[tid] << 8) | (255 - tid));
    if (ok_par && s_dnear[tid]) atomicAdd(&s_nd, 1);
  }
  __syncthreads();
  if (tid == 0) s_best = 255 - (s_best & 255);
  __syncthreads();
  const int best = s_best;
  bool writer = rank == 0;  // the CTA that writes the sequence's outputs

  // commit of the kept path, split over the cluster: its tree K/V rows are requested into
  // L2 now and copied after the final sample.  Every CTA read prefix_len[b] before the
  // wait; the writer advances it at the very end, after the last cluster barrier (the
  // non-greedy path) or alone (greedy: one CTA per sequence).
  const int commit_count = s_dep[best] + 1;
  if (p.commit) {
    if (tid == 0)
      for (int a = best, i = s_dep[best]; a >= 0; a = s_par[a], --i) s_path[i] = (int8_t)a;
    __syncthreads();
    if (commit_L >= 0) commit_prefetch_slice(p.cm, b, s_path, commit_count, rank, C);
  }

  if constexpr (GREEDY) {
    if (tid == 0) s_tok = __ldcg(&tstat[best].argmax);
  } else {
    // final sample: w = [p_best - q_{d+1}]+ if best has children, else p_best (a chain
    // whose drafts end after best: best is its leaf)
    const RowStat sp = load_stat(tstat + best);
    const uint4 *pv = reinterpret_cast<const uint4 *>(row_ptr<T>(p.target, (size_t)b * N + best, V));
    bool use_q = s_hc[best] != 0 && !(p.chain_end && s_end[best + 1]);
    // one-hot drafts: [p - e_x]+ is p without the rejected draft x (no q row is read)
    int x_excl = -1;
    if (use_q && onehot) {
      x_excl = s_xtok[best + 1];  // a chain: the child of best is best + 1
      use_q = false;
    }
    const int qrow = s_dep[best];  // q row of depth d+1
    const bool q_probs = p.q_kind == SV_Q_PROBS_F32;
    RowStat sq{};
    const uint4 *qv = nullptr;
    if (use_q) {
      if (!q_probs) {
        sq = load_stat(qstat + qrow);
        qv = reinterpret_cast<const uint4 *>(row_ptr<T>(p.q, (size_t)b * p.Dq + qrow, V));
      } else {
        qv = reinterpret_cast<const uint4 *>(static_cast<const float *>(p.q) +
                                             ((size_t)b * p.Dq + qrow) * V);
      }
    }
    const float c = p.c_log2;
    // TOPK: the value of the row's k-th entry (a vector below it holds no kept entry)
    const float thr_p = TOPK && sp.key_k != 0u ? key_to_value<T>(sp.key_k) : -INFINITY;
    const float inv_sp = 1.f / sp.S;
    const float inv_sq = use_q && !q_probs ? 1.f / sq.S : 0.f;
    const int nvec = V / VEC;
    // this CTA's slice of the vectors and its chunks of 32 vectors (chunk k = vectors
    // [c0 + 32k, c0 + 32k + 32), its sum at s_chunk[k]).  Slices start at multiples of 32
    // vectors, so that every chunk is the same 32 vectors (and its float sum the same)
    // however many CTAs share the pass.  With top-k each warp takes a contiguous segment
    // of the slice (whole chunks); without, the slice streams through the ring and warp w
    // takes chunk w of every stage.
    const int per_cta = ((nvec + (int)C - 1) / (int)C + 31) / 32 * 32;
    const int c0 = min(nvec, (int)rank * per_cta), c1 = min(nvec, c0 + per_cta);
    const int seg = ((c1 - c0 + NW - 1) / NW + 31) / 32 * 32;
    const int s0 = min(c1, c0 + warp * seg), s1 = min(c1, s0 + seg);
    const int nchs = (c1 - c0 + 31) / 32;         // chunks of the slice
    const bool keep_chunks = nchs <= kMaxChunks;  // (only the owning CTA reads them)
    const uint32_t stage_bytes = ring_stage_bytes<T>(q_probs);
    const uint32_t nrs = RING ? (uint32_t)p.ring_stages : 1u;  // stages of the ring
    uint32_t ring_seq = 0;   // ring stages consumed so far (all attempts)
    uint32_t last_seq0 = 0;  // ring_seq at the start of the last attempt's pass
    int ring_last = 0;       // stages of the last attempt's pass

    struct Raw {
      uint4 p, q[QV > 0 ? QV : 1];
    };
    auto load_raw = [&](int v, bool with_q) -> Raw {
      Raw r;
      r.p = __ldg(pv + v);
      if (with_q) {
        if (q_probs) {
#pragma unroll
          for (int h = 0; h < QV; ++h) r.q[h] = __ldg(qv + (size_t)v * QV + h);
        } else {
          r.q[0] = __ldg(qv + v);
        }
      }
      return r;
    };
    // weights of the VEC entries of vector v (top-k membership checked only with top-k)
    // (the arguments and scalings as packed f32x2: the same roundings as the scalar form)
    const float2 c2 = make_float2(c, c), zp2 = make_float2(sp.zmax, sp.zmax);
    const float2 ip2 = make_float2(inv_sp, inv_sp);
    auto weights = [&](int v, const Raw &r, float w[VEC], bool with_q) {
      float f[VEC];
      Elem<T>::unpack(r.p, f);
#pragma unroll
      for (int e = 0; e < VEC; e += 2) {
        const float2 t = mul2(sub2(make_float2(f[e], f[e + 1]), zp2), c2);
        const float2 x = mul2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), ip2);
        w[e] = x.x;
        w[e + 1] = x.y;
      }
      if (x_excl >= 0) {  // one-hot q: [p - e_x]+ is 0 at x
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (v * VEC + e == x_excl) w[e] = 0.f;
      }
      if (TOPK) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (!kept<T>(f[e], v * VEC + e, sp)) w[e] = 0.f;
      }
      if (with_q) {
        float g[VEC];
        if (q_probs) {
#pragma unroll
          for (int h = 0; h < QV; ++h) {
            g[4 * h] = __uint_as_float(r.q[h].x);
            g[4 * h + 1] = __uint_as_float(r.q[h].y);
            g[4 * h + 2] = __uint_as_float(r.q[h].z);
            g[4 * h + 3] = __uint_as_float(r.q[h].w);
          }
        } else {
          float fq[VEC];
          Elem<T>::unpack(r.q[0], fq);
          const float2 zq2 = make_float2(sq.zmax, sq.zmax), iq2 = make_float2(inv_sq, inv_sq);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 t = mul2(sub2(make_float2(fq[e], fq[e + 1]), zq2), c2);
            const float2 x = mul2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), iq2);
            g[e] = x.x;
            g[e + 1] = x.y;
          }
          if (TOPK) {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              if (!kept<T>(fq[e], v * VEC + e, sq)) g[e] = 0.f;
          }
        }
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
          const float2 d = sub2(make_float2(w[e], w[e + 1]), make_float2(g[e], g[e + 1]));
          w[e] = fmaxf(d.x, 0.f);
          w[e + 1] = fmaxf(d.y, 0.f);
        }
      }
    };
    auto vec_sum = [&](int v, const Raw &r, bool with_q) -> float {
      float w[VEC];
      weights(v, r, w, with_q);
      float vs = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) vs += w[e];
      return vs;
    };

    uint32_t k_acc, k_smp;  // u_smp = (k_smp + 0.5) 2^-24
    verify_uniform_ints(p.seed, p.round, b, best, &k_acc, &k_smp);

    for (int attempt = 0; attempt < 2; ++attempt) {
      F2 wsum = f2(0.f);  // lane 0: the sum of this warp's chunks
      if constexpr (RING) {
        // phase 1 through the ring: stage i holds vectors [c0 + i kRingVec, ...) of p and
        // the matching q; thread 0 keeps nrs stages in flight
        const int nstage = (c1 - c0 + kRingVec - 1) / kRingVec;
        const uint32_t qmul = use_q ? (q_probs ? (uint32_t)QV : 1u) : 0u;
        last_seq0 = ring_seq;
        int issued = 0;
        auto issue = [&](int i) {
          const int sl = (int)((ring_seq + (uint32_t)i) % nrs);
          const int v0 = c0 + i * kRingVec, nv = min(kRingVec, c1 - v0);
          const uint32_t pb = (uint32_t)nv * 16u, qb = pb * qmul;
          uint8_t *dst = sel_ring + (size_t)sl * stage_bytes;
          tc::fence_proxy_async_smem();
          tc::mbar_expect_tx(&ring_full[sl], pb + qb);
          bulk_g2s(dst, pv + v0, pb, &ring_full[sl]);
          if (qb) bulk_g2s(dst + kRingVec * 16, qv + (size_t)v0 * (q_probs ? QV : 1), qb, &ring_full[sl]);
          issued = i + 1;
        };
        if (tid == 0)
          for (int i = 0; i < min(nstage, (int)nrs); ++i) issue(i);
        int waited_ok = 0;    // thread 0: stages whose copies are known to have landed
        F2 lacc = f2(0.f);    // lane k < kChunksPerWarp: this warp's chunks k (float pairs)
        for (int i = 0; i < nstage; ++i) {
          const uint32_t gi = ring_seq + (uint32_t)i;
          const int sl = (int)(gi % nrs);
          const bool ok = tc::mbar_wait(&ring_full[sl], (gi / nrs) & 1u, &s_abort);
          if (tid == 0 && ok && waited_ok == i) waited_ok = i + 1;
          const uint8_t *st = sel_ring + (size_t)sl * stage_bytes;
          const uint4 *sp4 = reinterpret_cast<const uint4 *>(st);
          const uint4 *sq4 = reinterpret_cast<const uint4 *>(st + kRingVec * 16);
          const int vs0 = c0 + i * kRingVec;  // first vector of the stage
          // chunk j = warp + 8k of the stage: vectors vs0 + 32 j + lane
          float cs[kChunksPerWarp];
#pragma unroll
          for (int k = 0; k < kChunksPerWarp; ++k) {
            const int e = 32 * (warp + (kSelThreads / 32) * k) + lane;  // vector of the stage
            const int v = vs0 + e;
            cs[k] = 0.f;
            if (v < c1) {
              Raw r;
              r.p = sp4[e];
              if (use_q) {
                if (q_probs) {
#pragma unroll
                  for (int h = 0; h < QV; ++h) r.q[h] = sq4[e * QV + h];
                } else {
                  r.q[0] = sq4[e];
                }
              }
              cs[k] = vec_sum(v, r, use_q);
            }
          }
          // the chunk sums, reduced together (every lane gets all of them)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int k = 0; k < kChunksPerWarp; ++k) cs[k] += __shfl_xor_sync(0xFFFFFFFFu, cs[k], o);
#pragma unroll
          for (int k = 0; k < kChunksPerWarp; ++k) {
            const int j = warp + (kSelThreads / 32) * k;  // chunk of the stage
            if (lane == k && vs0 + 32 * j < c1) {
              if (keep_chunks) s_chunk[i * kRingChunks + j] = cs[k];
              lacc = f2_add(lacc, cs[k]);
            }
          }
          __syncthreads();  // every warp is done with this stage
          if (tid == 0 && i + (int)nrs < nstage && !s_abort) issue(i + (int)nrs);
        }
        // the warp's total: a butterfly of float-pair adds over lanes 0..kChunksPerWarp-1
#pragma unroll 1
        for (int o = 1; o < kChunksPerWarp; o <<= 1) lacc = f2_add(lacc, shfl_xor_f2(lacc, o));
        if (lane == 0) wsum = lacc;
        ring_last = nstage;
        if (s_abort) {
          // a wait gave up: let this CTA's copies in flight land before leaving
          if (tid == 0) {
            set_status(p.status, SV_DEV_TIMEOUT);
            for (int i = waited_ok; i < issued; ++i) {
              const uint32_t gi = ring_seq + (uint32_t)i;
              mbar_wait_drain(&ring_full[gi % nrs], (gi / nrs) & 1u);
            }
          }
          __syncthreads();
        }
        ring_seq += (uint32_t)nstage;
      } else
      // phase 1 from registers: chunk k of the warp's segment = its vectors [s0 + 32k, s0 +
      // 32k + 32), lane i taking vector s0 + 32k + i; four chunks are loaded before any is
      // used
      for (int k0 = 0; s0 + 32 * k0 < s1; k0 += 4) {
        constexpr int U = 4;
        Raw r[U];
        bool live[U];
        if constexpr (TOPK) {
          // with top-k, w is zero wherever p is: a vector whose largest logit is below the
          // row's k-th value has weight 0 (its q is not read)
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = s0 + 32 * (k0 + u) + lane;
            if (v < s1) r[u].p = __ldg(pv + v);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = s0 + 32 * (k0 + u) + lane;
            live[u] = v < s1 && vec_max<T>(r[u].p) >= thr_p;
            if (live[u] && use_q) r[u] = load_raw(v, true);
          }
        } else {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = s0 + 32 * (k0 + u) + lane;
            live[u] = v < s1;
            if (live[u]) r[u] = load_raw(v, use_q);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v0 = s0 + 32 * (k0 + u);
          if (v0 >= s1) break;
          const float cs = warp_sum_f(live[u] ? vec_sum(v0 + lane, r[u], use_q) : 0.f);
          if (lane == 0) {
            if (keep_chunks) s_chunk[(s0 - c0) / 32 + k0 + u] = cs;
            wsum = f2_add(wsum, cs);
          }
        }
      }
      if (lane == 0) seg_sum[warp] = wsum;
      __syncthreads();
      if (tid == 0) {
        F2 tot = f2(0.f);
        for (int w = 0; w < NW; ++w) tot = f2_add(tot, seg_sum[w]);
        s_slice[attempt] = tot;
      }
      if (C > 1) cluster_sync_all();
      else __syncthreads();
      if (warp == 0) {
        __syncwarp();
        // every CTA finds the same slice (same totals, same scan): lane r reads CTA r's
        // slice total through distributed shared memory
        const F2 tr = lane < (int)C ? (C > 1 ? ld_peer_f2(&s_slice[attempt], (unsigned)lane)
                                             : s_slice[attempt])
                                    : f2(0.f);
        // the cluster total, summed alike in every lane (a butterfly of float-pair adds)
        F2 total = tr;
#pragma unroll 1
        for (int o = 16; o > 0; o >>= 1) total = f2_add(total, shfl_xor_f2(total, o));
        total = shfl_f2(total, 0);
        int rs = -1;
        F2 base_r = f2(0.f), t = f2(0.f);
        if (total.hi > 0.f) {
          t = f2_uniform_times(k_smp, total);
          rs = warp_find_cdf(tr, (int)C, f2(0.f), t, &base_r);
        }
        // in the CTA whose slice holds t, warp 0 finds the chunk and the token
        if ((int)rank == rs && lane == 0) s_wstar = 0, s_base = base_r, s_t = t;
        if (lane == 0) s_rstar = rs;
      }
      __syncthreads();
      if (s_rstar >= 0) break;
      // the residual has no mass: sample from p instead (reported)
      use_q = false;
      x_excl = -1;
      if (tid == 0) s_snear = 1;
    }
    // this CTA has read its peers' totals for the last time: let them go once all have
    if (C > 1) cluster_arrive();
    const int rstar = s_rstar;
    writer = (int)rank == (rstar < 0 ? 0 : rstar);

    // phase 2: the owning warp finds the chunk from the chunk sums, then the token in it.
    // A vector is re-read from the ring when its stage is still there (the last
    // nrs stages of the last pass), else from global memory.
    auto load_final = [&](int v) -> Raw {
      if constexpr (RING) {
        const int i = (v - c0) / kRingVec;
        if (i < ring_last && ring_last - i <= (int)nrs) {
          const uint8_t *st = sel_ring + (size_t)((last_seq0 + (uint32_t)i) % nrs) * stage_bytes;
          const int e = v - c0 - i * kRingVec;
          Raw r;
          r.p = reinterpret_cast<const uint4 *>(st)[e];
          if (use_q) {
            const uint4 *sq4 = reinterpret_cast<const uint4 *>(st + kRingVec * 16);
            if (q_probs) {
#pragma unroll
              for (int h = 0; h < QV; ++h) r.q[h] = sq4[e * QV + h];
            } else {
              r.q[0] = sq4[e];
            }
          }
          return r;
        }
      }
      return load_raw(v, use_q);
    };
    if ((int)rank == rstar && warp == s_wstar) {
      __syncwarp();
      const F2 t = s_t;
      F2 base = s_base;
      int found = 0, tok = -1, near = 0, last_pos = -1;
      const int nch = nchs;
      int k_first = 0;
      if (keep_chunks) {
        // first chunk whose end passes t (else the last one with mass), in two levels:
        // groups of 32 chunks (lane g sums group g, float pairs), then the chunks of the
        // group found; the prefixes are float-pair sums, only chunk sums are float
        const int ngr = (nch + 31) / 32;
        int gstar = ngr == 1 ? 0 : -1, glast = -1;  // one group: no group level
        F2 base_g = base, base_glast = base;
        for (int g0 = 0; g0 < ngr && gstar < 0; g0 += 32) {
          const int g = g0 + lane;
          F2 x = f2(0.f);
          if (g < ngr) {
            // lane g starts at chunk (g mod 32) of its group: no two lanes read one bank
            for (int i = 0; i < 32; ++i) {
              const int k = 32 * g + ((i + lane) & 31);
              if (k < nch) x = f2_add(x, s_chunk[k]);
            }
          }
          F2 incl = x;
#pragma unroll 1
          for (int o = 1; o < 32; o <<= 1) {
            const F2 y = shfl_up_f2(incl, o);
            if (lane >= o) incl = f2_add(incl, y);
          }
          const F2 before = f2_add(base, f2_sub(incl, x));
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, g < ngr && f2_gt(f2_add(before, x), t));
          const unsigned pos = __ballot_sync(0xFFFFFFFFu, g < ngr && x.hi > 0.f);
          if (pos) {
            const int L = 31 - __clz(pos);
            glast = g0 + L;
            base_glast = shfl_f2(before, L);
          }
          if (hit) {
            const int L = __ffs(hit) - 1;
            gstar = g0 + L;
            base_g = shfl_f2(before, L);
          }
          base = f2_add(base, shfl_f2(incl, 31));
        }
        if (gstar < 0) gstar = glast, base_g = base_glast;
        int kstar = -1;
        F2 base_k = s_base;
        if (gstar >= 0) {
          // the chunks of group gstar
          const int k = 32 * gstar + lane;
          const F2 x = f2(k < nch ? s_chunk[k] : 0.f);
          F2 incl = x;
#pragma unroll 1
          for (int o = 1; o < 32; o <<= 1) {
            const F2 y = shfl_up_f2(incl, o);
            if (lane >= o) incl = f2_add(incl, y);
          }
          const F2 before = f2_add(base_g, f2_sub(incl, x));
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, k < nch && f2_gt(f2_add(before, x), t));
          const unsigned pos = __ballot_sync(0xFFFFFFFFu, k < nch && x.hi > 0.f);
          const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
          if (L >= 0) {
            kstar = 32 * gstar + L;
            base_k = shfl_f2(before, L);
          }
        }
        if (kstar < 0) kstar = 0, base_k = s_base;
        k_first = kstar;
        base = base_k;
      }
      for (int k = k_first; k < nch && !found; ++k) {
        const int v = c0 + 32 * k + lane;
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = 0.f;
        if (v < c1) weights(v, load_final(v), w, use_q);
        float lsum = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          lsum += w[e];
          if (w[e] > 0.f) last_pos = v * VEC + e;
        }
        const float incl = warp_incl_scan_f(lsum);
        const F2 before = f2_add(base, incl - lsum);
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, f2_gt(f2_add(before, lsum), t));
        if (hit) {
          const int L = __ffs(hit) - 1;
          if (lane == L) {
            F2 cum = before;
            int j = -1, lastp = -1;
            for (int e = 0; e < VEC; ++e) {
              if (w[e] <= 0.f) continue;
              const F2 prev = cum;
              cum = f2_add(cum, w[e]);
              lastp = v * VEC + e;
              if (f2_gt(cum, t)) {
                j = v * VEC + e;
                near = (f2_val(f2_sub(t, prev)) < kNearTieF) || (f2_val(f2_sub(cum, t)) < kNearTieF);
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
        base = f2_add(base, __shfl_sync(0xFFFFFFFFu, incl, 31));
        if (keep_chunks && !found) break;  // rounding: t fell past the chunk's end
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
    // no CTA leaves while a peer may still read its slice totals
    if (C > 1) cluster_wait();
  }
  if (p.commit) {
    if (commit_L >= 0)
      commit_path_slice(p.cm, b, commit_L, s_path, commit_count, rank, C);
    else if (tid == 0 && rank == 0)
      set_status(p.status, SV_DEV_BAD_PREFIX);
  }
  __syncthreads();

  if (tid == 0 && writer) {
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
    if (p.out_near_ties)
      p.out_near_ties[b] = (uint32_t)(s_nd + nuc_near) + (uint32_t)s_snear * kSampleTie;
    if (p.commit && commit_L >= 0) p.cm.prefix_len[b] = commit_L + commit_count;
  }
}

template <typename T, bool GREEDY, bool TOPK, bool RING>
__global__ void __launch_bounds__(kSelThreads) accept_select_kernel(const AcceptParams p) {
  const unsigned C = cluster_size(), rank = cluster_rank();
  // (select_seq waits for the statistics kernel once it has read its other inputs)
  select_seq<T, GREEDY, TOPK, RING, kSelThreads>(p, blockIdx.x / (int)C, rank, C);
}


// CTAs per sequence for the final sample: the most (a power of two, at most 16) that keep
// the select grid within one CTA per SM, so that its CTAs can start as the statistics
// kernel's last CTAs leave (the pass over two rows per sequence is split among them).
// With top-k, two per SM: its pass reads only the p row, at a few loads per vector.
int select_cluster(int B, int num_sms, bool topk) {
  const long long slots = (long long)num_sms * (topk ? 2 : 1);
  int C = 1;
  while (C < kMaxCluster && (long long)B * C * 2 <= slots) C *= 2;
  return C;
}

// Launch of one select kernel instantiation: C CTAs per sequence (clusters above 8 CTAs
// need the non-portable size, else C = 8), dyn bytes of dynamic shared memory.
template <typename T, bool GREEDY, bool TOPK, bool RING>
cudaError_t launch_select_kernel(AcceptParams pl, int C, cudaStream_t s) {
  auto kern = accept_select_kernel<T, GREEDY, TOPK, RING>;
  int dev = 0;
  cudaGetDevice(&dev);
  const bool dev_ok = dev >= 0 && dev < 64;
  if (C > 8) {
    // per device: 0 untried, 1 allowed, 2 refused (atomic: host threads may launch at once)
    static std::atomic<int> big_ok[64];
    if (dev_ok && big_ok[dev].load() == 0) {
      const bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                      cudaSuccess;
      cudaGetLastError();
      big_ok[dev].store(ok ? 1 : 2);
    }
    if (!dev_ok || big_ok[dev].load() != 1) C = 8;
  }
  size_t dyn = 0;
  if constexpr (RING) {
    // as many stages as one CTA's slice fills, at most kRingStages
    const int nvec = pl.V / Elem<T>::kVec;
    const int per_cta = ((nvec + C - 1) / C + 31) / 32 * 32;
    pl.ring_stages = std::max(1, std::min(kRingStages, (per_cta + kRingVec - 1) / kRingVec));
    dyn = (size_t)pl.ring_stages * ring_stage_bytes<T>(pl.q_kind == SV_Q_PROBS_F32);
    static std::atomic<bool> attr_ok[64];
    if (!dev_ok || !attr_ok[dev].load()) {
      const cudaError_t e = cudaFuncSetAttribute(
          kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
          (int)((size_t)kRingStages * ring_stage_bytes<T>(true)));
      if (e != cudaSuccess) return e;
      if (dev_ok) attr_ok[dev].store(true);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.B * C));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // its launch and prologue overlap the statistics kernel's tail
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, pl);
}

// Select kernel of a call: the ring variant (final sample streamed through shared
// memory) when each CTA's slice of the vocabulary is long, else the register variant
// (short slices are latency-bound; it keeps the dynamic shared memory at zero, so that its
// CTAs can start beside the statistics kernel's last CTAs).
template <typename T, bool GREEDY, bool TOPK>
cudaError_t launch_select(const AcceptParams &p, int num_sms, cudaStream_t s) {
  const int C = GREEDY ? 1 : select_cluster(p.B, num_sms, TOPK);
  AcceptParams pl = p;
  pl.ring_stages = 0;
  if constexpr (!GREEDY && !TOPK) {
    const int nvec = p.V / Elem<T>::kVec;
    const int per_cta = ((nvec + C - 1) / C + 31) / 32 * 32;
    if (per_cta >= kRingMinVec) return launch_select_kernel<T, GREEDY, TOPK, true>(pl, C, s);
  }
  return launch_select_kernel<T, GREEDY, TOPK, false>(pl, C, s);
}

// Kernel 1 alone: the statistics of every target row, then of every q row (q logits).
template <typename T>
cudaError_t launch_stats_typed(const AcceptParams &p, cudaStream_t s) {
  const bool greedy = p.mode == SV_GREEDY;
  const bool topk = !greedy && p.top_k > 0 && p.top_k < p.V;
  const int rows = p.B * p.N + ((!greedy && p.q_kind == SV_Q_LOGITS) ? p.B * p.Dq : 0);
  if (greedy)
    accept_stats_kernel<T, true, false><<<rows, stat_threads<false>(), 0, s>>>(p);
  else if (topk)
    accept_stats_kernel<T, false, true><<<rows, stat_threads<true>(), 0, s>>>(p);
  else
    accept_stats_kernel<T, false, false><<<rows, stat_threads<false>(), 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const AcceptParams &p, int num_sms, cudaStream_t s) {
  const bool greedy = p.mode == SV_GREEDY;
  const bool topk = !greedy && p.top_k > 0 && p.top_k < p.V;
  if (p.typical) {
    // the target rows' statistics with their entropy, then the greedy-form select kernel
    // taking the typical decisions (the emitted token after the path is the argmax)
    accept_stats_kernel<T, false, false, true><<<p.B * p.N, stat_threads<false>(), 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_select<T, true, false>(p, num_sms, s);
  }
  cudaError_t e = launch_stats_typed<T>(p, s);
  if (e != cudaSuccess) return e;
  if (greedy) return launch_select<T, true, false>(p, num_sms, s);
  return topk ? launch_select<T, false, true>(p, num_sms, s)
              : launch_select<T, false, false>(p, num_sms, s);
}

}  // namespace

size_t accept_ws_bytes(int B, int N, int Dq) {
  return (size_t)B * (size_t)(N + Dq) * sizeof(RowStat);
}

cudaError_t launch_accept(sv_dtype dt, const AcceptParams &p, int num_sms, cudaStream_t s) {
  return dt == SV_F32 ? launch_typed<float>(p, num_sms, s) : launch_typed<bf16>(p, num_sms, s);
}

cudaError_t launch_accept_stats(sv_dtype dt, const AcceptParams &p, cudaStream_t s) {
  return dt == SV_F32 ? launch_stats_typed<float>(p, s) : launch_stats_typed<bf16>(p, s);
}

// The target rows' statistics are already in place (the LM-head projection's epilogue
// wrote them; no top-k): the statistics kernel over the q rows only when q comes as
// logits, then the select kernel (its wait for the previous grid then covers either).
template <typename T>
cudaError_t launch_given_typed(const AcceptParams &p, int num_sms, cudaStream_t s) {
  const bool greedy = p.mode == SV_GREEDY;
  if (!greedy && p.q_kind == SV_Q_LOGITS && p.B * p.Dq > 0) {
    AcceptParams pq = p;
    pq.stat_row0 = p.B * p.N;
    accept_stats_kernel<T, false, false><<<p.B * p.Dq, stat_threads<false>(), 0, s>>>(pq);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (greedy) return launch_select<T, true, false>(p, num_sms, s);
  return launch_select<T, false, false>(p, num_sms, s);
}

cudaError_t launch_accept_given_target_stats(sv_dtype dt, const AcceptParams &p, int num_sms,
                                             cudaStream_t s) {
  return dt == SV_F32 ? launch_given_typed<float>(p, num_sms, s) : launch_given_typed<bf16>(p, num_sms, s);
}

}  // namespace sv
