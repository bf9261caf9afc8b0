// Exact tree acceptance with the siblings of a node tried in turn (sm_103a).
//
// Method (hncyxsy.com sections 2.1-2.2: after a rejected candidate the target becomes the
// residual norm([p - q]+); the jennyma11 blog, section "Medusa", separates this lossless
// tree verification from typical acceptance).  From the root, the children of the current
// node are tried in row (rank) order: child c is accepted iff u_acc(b, c) < r(x_c) / q(x_c),
// where r starts as the node's effective target distribution p and, after each rejected
// sibling, becomes the residual norm([r - q]+) (kept as it was, and counted as a near tie,
// when that residual has no mass); q is the effective draft distribution of the children's
// depth.  An accepted child becomes the current node.  When every child is rejected the
// next token is drawn with u_smp(b, node) from norm([r - q]+) of the last r; a leaf draws
// the bonus token from its p.  With one child per node this is the chain procedure.
//
// The residual after k rejections has a closed form: r_k = [p - c_k q]+ / N_k with
// c_0 = 0, N_0 = 1, c_k = c_{k-1} + N_{k-1} and N_k = sum_j [p_j - c_k q_j]+ (because
// [p - c q]+ / N - q is positive only where p - c q > N q >= 0, and there equals
// (p - (c + N) q) / N).  So each rejection costs one reduction pass over the vocabulary
// of the current node's target row and the depth's q row, and the final sample is one
// inverse-CDF pass over w = [p - c q]+.
//
// A thread-block cluster of C CTAs per sequence walks the tree, every CTA alike: thread 0
// of each takes each decision in double from the two logits at the candidate and the
// rows' statistics (kernel 1 of the acceptance), so all CTAs follow the same path.  Each
// CTA owns a slice of the vocabulary: a residual mass is the sum of the CTAs' slice sums
// (entries formed in float, summed exactly as float pairs, then in double), exchanged
// through distributed shared memory and added in rank order, identically in every CTA.
// The final sample: per-chunk sums of w in each slice, the slice holding u * sum(w) found
// from the slice totals, then in that CTA the chunk (a scan of its chunk sums) and the
// token inside it (warp-wide inclusive scans in token order).  The cluster barriers are
// reached by every CTA (their branches depend only on values all CTAs compute alike); no
// other wait: every loop is bounded by the vocabulary or the tree size.
#include <atomic>

#include "row_stat.cuh"
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kRecThreads = 512;
constexpr int kRecWarps = kRecThreads / 32;
constexpr int kRecMaxChunks = 1024;  // chunk sums kept by a CTA
constexpr int kRecMaxCluster = 16;   // CTAs per sequence
constexpr double kRecNearTie = 1e-6;
// Error bound of a residual mass formed here, in units of the target's probabilities:
// each entry [p_j - c q_j]+ is formed in float from p_j and q_j that carry a few float
// roundings each, so the sum over the vocabulary is off by at most about
// kRecEntryErr * (1 + c) (the entries' magnitudes sum to 1 + c).  After rejections the
// residual mass n can be small, and the relative error of anything divided by n grows
// as (1 + c) / n: the near-tie windows widen by that bound where it exceeds 1e-6.
constexpr double kRecEntryErr = 4.0 * 1.1920928955078125e-7;  // 4 float epsilons

// One sequence's view of the current node's target row and the depth's q row.
template <typename T>
struct RowPair {
  const T *zt;        // target logits of the current node
  const T *zq;        // q logits of the children's depth (q logits), else NULL
  const float *qp;    // q probabilities of that depth (q probabilities), else NULL
  RowStat sa, sq;     // statistics of the two rows (sq: q logits only)
  float c_log2;       // log2(e) / T
  float inv_sa, inv_sq;
};

// w_j = [p_j - c q_j]+ of entry j, in float (c == 0: p_j, the q row is not read).
template <typename T>
__device__ __forceinline__ float w_at(const RowPair<T> &r, int j, float c) {
  const float z = Elem<T>::load(r.zt + j);
  const float pj = kept<T>(z, j, r.sa) ? exp2f((z - r.sa.zmax) * r.c_log2) * r.inv_sa : 0.f;
  if (c == 0.f) return pj;
  float qj;
  if (r.zq != nullptr) {
    const float zq = Elem<T>::load(r.zq + j);
    qj = kept<T>(zq, j, r.sq) ? exp2f((zq - r.sq.zmax) * r.c_log2) * r.inv_sq : 0.f;
  } else {
    qj = r.qp[j];
  }
  return fmaxf(pj - c * qj, 0.f);
}

// The 8 entries w_j = [p_j - c q_j]+ of group g (entries 8g .. 8g+7), each formed in
// float exactly as w_at forms it, from 16-byte loads of the two rows.
template <typename T>
__device__ __forceinline__ void w_group(const RowPair<T> &r, int g, float c, float w[8]) {
  constexpr int kv = Elem<T>::kVec;  // entries per 16-byte vector
  float z[8], zq[8];
#pragma unroll
  for (int i = 0; i < 8 / kv; ++i)
    Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(r.zt + (size_t)g * 8) + i), z + i * kv);
  if (c != 0.f) {
    if (r.zq != nullptr) {
#pragma unroll
      for (int i = 0; i < 8 / kv; ++i)
        Elem<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(r.zq + (size_t)g * 8) + i), zq + i * kv);
    } else {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(r.qp + (size_t)g * 8));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(r.qp + (size_t)g * 8) + 1);
      zq[0] = a.x, zq[1] = a.y, zq[2] = a.z, zq[3] = a.w;
      zq[4] = b.x, zq[5] = b.y, zq[6] = b.z, zq[7] = b.w;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = g * 8 + i;
    const float pj = kept<T>(z[i], j, r.sa) ? exp2f((z[i] - r.sa.zmax) * r.c_log2) * r.inv_sa : 0.f;
    if (c == 0.f) {
      w[i] = pj;
      continue;
    }
    float qj;
    if (r.zq != nullptr)
      qj = kept<T>(zq[i], j, r.sq) ? exp2f((zq[i] - r.sq.zmax) * r.c_log2) * r.inv_sq : 0.f;
    else
      qj = zq[i];
    w[i] = fmaxf(pj - c * qj, 0.f);
  }
}

// A running sum carried as hi + lo of two floats: each addition is exact up to the
// final rounding of hi + lo (Knuth's TwoSum), so the sum of float entries is as good as
// a double accumulation, without the part's slow FP64 adds.
struct SumF2 {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float s = hi + x;
    const float bb = s - hi;
    lo += (hi - (s - bb)) + (x - bb);
    hi = s;
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// This thread's sum of w over groups g0, g0 + stride, ... below g_end, two groups'
// loads in flight at a time.
template <typename T>
__device__ __forceinline__ double w_sum(const RowPair<T> &r, int g0, int g_end, int stride, float c) {
  SumF2 acc;
  int g = g0;
  for (; g + stride < g_end; g += 2 * stride) {
    float a[8], b[8];
    w_group<T>(r, g, c, a);
    w_group<T>(r, g + stride, c, b);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc.add(a[i]);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc.add(b[i]);
  }
  if (g < g_end) {
    float a[8];
    w_group<T>(r, g, c, a);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc.add(a[i]);
  }
  return acc.value();
}

__device__ __forceinline__ unsigned rec_cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned rec_cluster_size() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void rec_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ double ld_peer_d(const double *local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ void st_peer_i(int *local, unsigned rank, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// The cluster-wide sum of one double per thread (v): each warp's sum goes to
// parts[k & 1][warp]; after one cluster barrier warp 0 of every CTA reads all C ranks'
// warp sums (lane r those of rank r, added in warp order) and sums the ranks in a fixed
// order, so every CTA gets the same total; lane r of warp 0 also gets rank r's total in
// *lane_val.  The slots alternate with k (and so does the broadcast), so that a slot is
// rewritten only after the next cluster barrier, which every peer reaches after its reads.
__device__ double cluster_sum(double v, double (*parts)[kRecWarps], double *bcast, int k, unsigned C,
                              double *lane_val) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) parts[k & 1][warp] = v;
  rec_cluster_sync();  // (also orders this CTA's writes of parts before warp 0's reads)
  if (warp == 0) {
    double x = 0.0;
    if (lane < (int)C)
      for (int w = 0; w < kRecWarps; ++w) x += ld_peer_d(&parts[k & 1][w], (unsigned)lane);
    if (lane_val) *lane_val = x;
    const double t = warp_sum_d(x);
    if (lane == 0) bcast[k & 1] = t;
  }
  __syncthreads();
  return bcast[k & 1];
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// What the decision on candidate child ch of the current node needs, in double: p(x) and
// q(x) of its token x, and u_acc(b, ch).  Computed for all children of a node at once (one
// thread each); flags: bit 0 the token is out of range, bit 1 q(x) = 0.
struct ChildIn {
  double px, qx, u;
  int flags;
};
template <typename T>
__device__ ChildIn child_inputs(const AcceptParams &p, const RowPair<T> &r, int b, int ch, bool logits) {
  ChildIn ci{0.0, 0.0, 1.0, 0};
  const int x = p.tokens[(size_t)b * p.tok_stride + ch - p.tok_offset];
  if (x < 0 || x >= p.V) {
    ci.flags = 1;
    return ci;
  }
  const double temp = (double)p.temperature;
  const float zp = Elem<T>::load(r.zt + x);
  ci.px = kept<T>(zp, x, r.sa) ? exp(((double)zp - (double)r.sa.zmax) / temp) / (double)r.sa.S : 0.0;
  if (logits) {
    const float zq = Elem<T>::load(r.zq + x);
    ci.qx = kept<T>(zq, x, r.sq) ? exp(((double)zq - (double)r.sq.zmax) / temp) / (double)r.sq.S : 0.0;
  } else {
    ci.qx = (double)r.qp[x];
  }
  if (!(ci.qx > 0.0)) ci.flags |= 2;
  uint32_t k_acc = 0u, k_smp = 0u;
  verify_uniform_ints(p.seed, p.round, b, ch, &k_acc, &k_smp);
  ci.u = ((double)k_acc + 0.5) * (1.0 / 16777216.0);
  return ci;
}

// The decision on a child against the current residual [p - c q]+ / n (thread 0):
// ratio = [p(x) - c q(x)]+ / (n q(x)).  Returns bit 0: accepted, bit 1: near tie.
__device__ int decide_child(const AcceptParams &p, const ChildIn &ci, double c, double n) {
  if (ci.flags & 1) {
    set_status(p.status, SV_DEV_BAD_TOKEN);
    return 0;
  }
  const double rx = fmax(ci.px - c * ci.qx, 0.0) / n;
  double ratio;
  if (ci.qx > 0.0) {
    ratio = rx / ci.qx;
  } else {
    set_status(p.status, SV_DEV_ZERO_DRAFT_PROB);
    ratio = rx > 0.0 ? INFINITY : 0.0;
  }
  // after a rejection (c > 0) the ratio divides by the float-formed residual mass n
  const double win =
      kRecNearTie + (c > 0.0 ? kRecEntryErr * (1.0 + c) / n * fmax(ratio, 1.0) : 0.0);
  return (ci.u < ratio ? 1 : 0) | (fabs(ci.u - ratio) < win ? 2 : 0);
}

template <typename T>
__global__ void __launch_bounds__(kRecThreads) accept_recursive_kernel(const AcceptParams p) {
  __shared__ double s_chunk[kRecMaxChunks];
  __shared__ double s_parts[2][kRecWarps], s_bcast[2];
  __shared__ int s_dec[2], s_tok, s_near;
  int ndec = 0;  // decisions so far (parity of the s_dec slot)
  __shared__ ChildIn s_cin[kMaxNodes];

  const unsigned C = rec_cluster_size(), rank = rec_cluster_rank();
  const int b = blockIdx.x / (int)C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.tree.N, V = p.V;
  const bool logits = p.q_kind == SV_Q_LOGITS;
  const RowStat *tstat = p.stats + (size_t)b * N;
  const RowStat *qstat = p.stats + (size_t)p.B * N + (size_t)b * p.Dq;

  // this CTA's slice of the vocabulary: chunks [ch_lo, ch_hi) of CH entries (whole 256-entry
  // warp steps; at most kRecMaxChunks per CTA), in 8-entry groups [g_lo, g_hi)
  const int ng = V / 8;
  const int per_cta = (V + (int)C - 1) / (int)C;
  const int CH = max(256, ((per_cta + kRecMaxChunks - 1) / kRecMaxChunks + 255) / 256 * 256);
  const int CHG = CH / 8;
  const int nch_all = (V + CH - 1) / CH;
  const int ch_per = (nch_all + (int)C - 1) / (int)C;
  const int ch_lo = min(nch_all, (int)rank * ch_per), ch_hi = min(nch_all, ch_lo + ch_per);
  const int nloc = ch_hi - ch_lo;
  const int g_lo = ch_lo * CHG, g_hi = min(ng, ch_hi * CHG);
  int xk = 0;  // cluster exchanges so far (slot parity)

  // sequence b's tree (the shared one, or its own row, checked: a malformed row or a node
  // deeper than the q rows leaves the root alone, which draws the bonus from its p)
  __shared__ int s_par[kMaxNodes], s_dep[kMaxNodes];
  bool bad = false;
  if (tid < kMaxNodes) {
    int v = -1;
    if (tid < N) {
      v = tree_parent(p.tree, b, tid);
      bad = tid == 0 ? v != -1 : (v < 0 || v >= tid);
      if (bad) v = tid == 0 ? -1 : 0;
    }
    s_par[tid] = v;
  }
  __syncthreads();
  if (tid < N) {
    uint64_t anc_unused;
    int d = 0;
    tree_walk(s_par, tid, &anc_unused, &d);
    s_dep[tid] = d;
    if (d > p.Dq) bad = true;
  }
  const bool seq_bad = __syncthreads_or(bad) != 0;
  if (seq_bad && tid == 0 && rank == 0) set_status(p.status, SV_DEV_BAD_TREE);
  const int Nw = seq_bad ? 1 : N;  // nodes walked: the root alone for a bad tree

  // thread 0's running counts: near ties that can change a decision (near decisions,
  // empty residuals handed to a sibling; nucleus cuts) and those of the final sample
  unsigned near = 0u, near_smp = 0u;
  bool nuc = false;

  RowPair<T> r;
  r.c_log2 = p.c_log2;
  r.zq = nullptr;
  r.qp = nullptr;
  r.inv_sq = 0.f;
  int node = 0;
  double c = 0.0, n = 1.0;    // the current residual: [p - c q]+ / n
  double c_fin = 0.0;         // the final sample's w = [p - c_fin q]+
  for (int steps = 0; steps < N; ++steps) {
    // the children of the node: rows after it whose parent it is (the same in every thread)
    int first = -1, last = -1;
    for (int ch = node + 1; ch < Nw; ++ch)
      if (s_par[ch] == node) {
        if (first < 0) first = ch;
        last = ch;
      }
    r.zt = reinterpret_cast<const T *>(p.target) + ((size_t)b * N + node) * V;
    r.sa = load_stat(tstat + node);
    r.inv_sa = 1.f / r.sa.S;
    if (tid == 0) nuc |= (r.sa.flags & 1u) != 0u;
    c = 0.0;
    n = 1.0;
    if (first < 0) {  // a leaf: the bonus token from its p
      c_fin = 0.0;
      break;
    }
    const int drow = s_dep[node];  // q row of the children's depth (depth - 1)
    if (logits) {
      r.zq = reinterpret_cast<const T *>(p.q) + ((size_t)b * p.Dq + drow) * V;
      r.sq = load_stat(qstat + drow);
      r.inv_sq = 1.f / r.sq.S;
      if (tid == 0) nuc |= (r.sq.flags & 1u) != 0u;
    } else {
      r.qp = static_cast<const float *>(p.q) + ((size_t)b * p.Dq + drow) * V;
    }
    // every child's p(x), q(x) and u at once, one thread each
    if (tid >= first && tid <= last && s_par[tid] == node) s_cin[tid] = child_inputs<T>(p, r, b, tid, logits);
    __syncthreads();
    int next = -1;
    for (int ch = first; ch <= last; ++ch) {
      if (s_par[ch] != node) continue;
      if (tid == 0) {
        const int d = decide_child(p, s_cin[ch], c, n);
        near += (unsigned)(d >> 1);
        s_dec[ndec & 1] = d & 1;
      }
      __syncthreads();
      // (two slots: a slot is rewritten two decisions later, past another barrier)
      const int acc = s_dec[ndec & 1];
      ++ndec;
      if (acc) {
        next = ch;
        break;
      }
      if (ch == last) break;
      // the next sibling sees the residual [p - (c + n) q]+ / its mass
      const double c1 = c + n;
      const float c1f = (float)c1;
      const double tot = cluster_sum(w_sum<T>(r, g_lo + tid, g_hi, kRecThreads, c1f), s_parts, s_bcast,
                                     xk++, C, nullptr);
      if (tot > kRecEntryErr * (1.0 + c1)) {
        c = c1;
        n = tot;
      } else if (tid == 0) {
        // no mass left, or less than the rounding error of its sum: the residual stays
        // as it was (a near tie: in exact arithmetic it may hold a little mass)
        ++near;
      }
    }
    if (next >= 0) {
      node = next;
      continue;
    }
    c_fin = c + n;  // every child rejected: sample from the last residual's residual
    break;
  }

  // ---- final sample: inverse CDF of w = [p - c_fin q]+ in token order, with u_smp(b, node)
  float cf = (float)c_fin;
  // the 1e-6 window in units of the normalised residual, or the rounding bound of the
  // float-formed w (kRecEntryErr per unit of the entries' magnitudes) when that is wider
  const double tol = fmax(kRecNearTie * n, kRecEntryErr * (1.0 + c_fin));
  double total = 0.0, slice_tot = 0.0;  // slice_tot: rank `lane`'s slice total (warp 0)
  for (int attempt = 0; attempt < 2; ++attempt) {
    double wpart = 0.0;  // this warp's chunks (every lane holds it)
    for (int k = warp; k < nloc; k += kRecWarps) {
      const int kg = ch_lo + k;
      const double sk = warp_sum_d(w_sum<T>(r, kg * CHG + lane, min(ng, (kg + 1) * CHG), 32, cf));
      if (lane == 0) s_chunk[k] = sk;
      wpart += sk;
    }
    total = cluster_sum(lane == 0 ? wpart : 0.0, s_parts, s_bcast, xk++, C, &slice_tot);
    if (total > kRecEntryErr * (1.0 + (double)cf) || attempt == 1) break;
    // the residual has no mass: sample from the last residual itself
    if (tid == 0) ++near_smp;
    cf = (float)c;
    __syncthreads();  // s_chunk is rewritten by the second attempt
  }

  if (warp == 0) {
    uint32_t k_acc = 0u, k_smp = 0u;
    verify_uniform_ints(p.seed, p.round, b, node, &k_acc, &k_smp);
    const double u = ((double)k_smp + 0.5) * (1.0 / 16777216.0);
    // the slice holding u * sum(w): lane r holds rank r's slice total (the same in every
    // CTA); the sum is the scan's end, as the prefixes are
    const double sincl = warp_incl_scan_d(slice_tot);
    const double t = u * __shfl_sync(0xFFFFFFFFu, sincl, 31);
    unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < (int)C && sincl > t);
    if (hit == 0u) {  // t at or past the end (rounding): the last slice with mass
      const unsigned m = __ballot_sync(0xFFFFFFFFu, lane < (int)C && slice_tot > 0.0);
      hit = m != 0u ? 1u << (31 - __clz(m)) : 1u;
    }
    const int owner = __ffs(hit) - 1;
    const double sbase = __shfl_sync(0xFFFFFFFFu, sincl - slice_tot, owner);
    if ((int)rank == owner) {
      // lane l owns local chunks [l * per, (l + 1) * per): its sum, then a scan over the lanes
      const int per = (nloc + 31) / 32;
      const int k0 = min(nloc, lane * per), k1 = min(nloc, k0 + per);
      double ls = 0.0;
      for (int k = k0; k < k1; ++k) ls += s_chunk[k];
      const double incl = sbase + warp_incl_scan_d(ls);
      unsigned hit2 = __ballot_sync(0xFFFFFFFFu, k1 > k0 && incl > t);
      if (hit2 == 0u) {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, ls > 0.0);
        hit2 = m != 0u ? 1u << (31 - __clz(m)) : 1u;
      }
      const int L = __ffs(hit2) - 1;
      // lane L finds its first chunk whose end passes t (else its last chunk)
      int my_start = k1 - 1;
      double my_base = incl - ls;
      if (lane == L) {
        for (int k = k0; k < k1; ++k) {
          if (my_base + s_chunk[k] > t) {
            my_start = k;
            break;
          }
          if (k + 1 < k1) my_base += s_chunk[k];
        }
      }
      const int start = max(0, __shfl_sync(0xFFFFFFFFu, my_start, L));
      const double base = __shfl_sync(0xFFFFFFFFu, my_base, L);
      // the token: warp-wide scans in token order from the start chunk to the slice end
      const int j_end = min(V, g_hi * 8);
      int tok = -1, last_pos = -1, nearf = 0;
      double run = base;
      for (int j0 = (ch_lo + start) * CH; j0 < j_end; j0 += 32) {
        const int j = j0 + lane;
        const double w = j < j_end ? (double)w_at<T>(r, j, cf) : 0.0;
        const double ci = warp_incl_scan_d(w);
        const double cum = run + ci, prev = cum - w;
        const unsigned h = __ballot_sync(0xFFFFFFFFu, w > 0.0 && cum > t);
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, w > 0.0);
        if (h != 0u) {
          const int lh = __ffs(h) - 1;
          const int nr = (t - prev < tol || cum - t < tol) ? 1 : 0;
          nearf = __shfl_sync(0xFFFFFFFFu, nr, lh);
          tok = j0 + lh;
          break;
        }
        if (pos != 0u) last_pos = j0 + 31 - __clz(pos);
        run += __shfl_sync(0xFFFFFFFFu, ci, 31);
      }
      if (tok < 0) {  // rounding put u * sum(w) at or past the end: the last token with mass
        tok = last_pos >= 0 ? last_pos : 0;
        nearf = 1;
      }
      if (lane == 0) {  // to rank 0, which writes the outputs
        st_peer_i(&s_tok, 0u, tok);
        st_peer_i(&s_near, 0u, nearf);
      }
    }
  }
  rec_cluster_sync();  // the token is in rank 0's shared memory

  if (tid == 0 && rank == 0) {
    near += nuc ? 1u : 0u;
    near_smp += (unsigned)s_near;
    const int W = p.tree.Dmax + 1;
    const int D = s_dep[node];
    int32_t *pn = p.out_path_nodes ? p.out_path_nodes + (size_t)b * W : nullptr;
    int32_t *tk = p.out_tokens + (size_t)b * W;
    for (int i = 0; i < W; ++i) {
      if (pn) pn[i] = -1;
      tk[i] = -1;
    }
    int i = D;
    for (int a = node; a >= 0 && i >= 0; a = s_par[a], --i) {
      if (pn) pn[i] = a;
      if (i >= 1) tk[i - 1] = p.tokens[(size_t)b * p.tok_stride + a - p.tok_offset];
    }
    tk[D] = s_tok;
    p.out_num_emitted[b] = D + 1;
    p.out_num_accepted[b] = D;
    if (p.out_near_ties) p.out_near_ties[b] = near + near_smp * 65536u;
  }
}

// CTAs per sequence: the largest power of two up to kRecMaxCluster that keeps the grid
// within one CTA per SM and each CTA's slice at least 2048 entries.
int recursive_cluster(int B, int V, int num_sms) {
  int C = 1;
  while (C < kRecMaxCluster && (long long)B * C * 2 <= num_sms && V / (C * 2) >= 2048) C *= 2;
  return C;
}

template <typename T>
cudaError_t launch_recursive_typed(const AcceptParams &p, cudaStream_t s) {
  auto kern = accept_recursive_kernel<T>;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int C = recursive_cluster(p.B, p.V, sms);
  if (C > 8) {
    static std::atomic<int> big_ok[64];  // 0 untried, 1 allowed, 2 refused
    const bool dev_ok = dev >= 0 && dev < 64;
    if (dev_ok && big_ok[dev].load() == 0) {
      const bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                      cudaSuccess;
      cudaGetLastError();
      big_ok[dev].store(ok ? 1 : 2);
    }
    if (!dev_ok || big_ok[dev].load() != 1) C = 8;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * C));
  cfg.blockDim = dim3(kRecThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_accept_recursive(sv_dtype dt, const AcceptParams &p, cudaStream_t s) {
  cudaError_t e = launch_accept_stats(dt, p, s);
  if (e != cudaSuccess) return e;
  return dt == SV_F32 ? launch_recursive_typed<float>(p, s) : launch_recursive_typed<bf16>(p, s);
}

}  // namespace sv
