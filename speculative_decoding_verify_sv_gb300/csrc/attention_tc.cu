// Tree attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA), sm_103a.
//
// What it computes is the tree attention of attention.cu: for sequence b, node n and
// query head h the keys are the prefix [0, L_b) plus the tree nodes on n's root path
// (the ancestor mask of "推测解码技术详解", section "Tree Attention验证").
//
// Work unit = (sequence b, kv head, group of 128*MT query rows); its rows are the
// (node, group-head) pairs, so the tree and the GQA group form the M side of one MMA.
// A unit's keys are tiles of BN: tile 0 = the tree nodes (masked by ancestor bits),
// tiles 1.. = the prefix.  The flattened (unit, tile) space is split evenly over one
// persistent CTA per SM (stream-K); a unit cut by a CTA boundary is written as fp32
// partials by the CTAs holding its later tiles, and the CTA holding its first tiles merges
// them with log-sum-exp weights in the same launch (cooperative, so all CTAs are resident).
//
// Per CTA, warp roles:
//   producer warp   TMA loads of Q (per piece, QBUF buffers) and K/V tiles into rings
//                   of STAGES K and VST V stages (a single M tile with one P buffer
//                   spends the second P buffer's room on a third V stage -- V is held
//                   until P V completes, K only until S = Q K^T does -- or on a
//                   second Q buffer);
//   MMA warp        one thread issues P V as soon as P is written and keeps S = Q K^T
//                   two tiles ahead (S in TMEM, double buffered; O accumulates in TMEM);
//   4*MT softmax warps, one thread per query row: read S from TMEM, mask, online
//                   softmax in log2 units, write P (bf16, 128B-swizzled, PBUF
//                   buffers) to shared memory, rescale O in TMEM only when the running
//                   max grows by more than 2^8, and write the normalised row at the end.
// When all query rows fit in 128/CP lanes (CP = 2 or 4 row copies), the rows are
// loaded CP times into the A tile so that every TMEM lane quarter, and so every SM
// sub-partition's exponential unit, holds a copy; the copies split each tile's columns.
//
// Two M tiles (129..256 rows) run as a ping-pong instead: each M tile m has one S region
// in TMEM, and its softmax warps write P (bf16) over that S in TMEM, from where P V takes
// its A operand; S[m] is free again once P V of m has completed.  The tensor pipe then
// alternates between the M tiles (Q K^T of one while the other's softmax runs), no P
// passes through shared memory, and the keys come in tiles of 128, so that Q (both M
// tiles, 64 KB at D = 128) is read by the tensor core once per 128 keys.
#include <atomic>
#include <cudaTypedefs.h>

#include <cfloat>

#include "sv_common.cuh"
#include "sv_internal.h"
#include "tc_primitives.cuh"

namespace sv {

namespace {

using namespace tc;

constexpr int kRows = 128;                // rows per MMA (one M tile)
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr unsigned kPollSleepNs = 32;     // MMA issuer's back-off between idle polls
// Slots of the flattened work space that stand for the start of a unit (its Q load,
// the previous piece's O readout and, for a cut unit, the merge).  Charged only when a
// CTA holds few units (then the number of unit starts per CTA varies by one or two and
// decides which CTA finishes last); with many units per CTA the costs average out.
constexpr int kUnitStartSlots = 4;

// 2^x by the hardware's approximate exponential (one MUFU op; 2^-inf = +0).  P is
// rounded to bf16 for the tensor core, far coarser than this instruction's error.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int MT, int CP, int BN, int STAGES, int QBUF, int PBUF>
struct TcLayout {
  static constexpr int KB = D / 64;                      // 64-element column blocks of Q/K/V
  static constexpr int Q_BLOCK = MT * kRows * 128;       // one column block of Q
  static constexpr int Q_BYTES = KB * Q_BLOCK;
  static constexpr int KV_BLOCK = BN * 128;              // one column block of a K/V tile
  static constexpr int KV_BYTES = KB * KV_BLOCK;
  static constexpr int PB = BN / 64;                     // 64-key column blocks of P
  static constexpr int P_BLOCK = kRows * 128;
  static constexpr int P_TILE = PB * P_BLOCK;            // P of one M tile
  // two M tiles keep P in TMEM (over S): no P buffers in shared memory
  static constexpr bool PT = MT == 2;
  static constexpr int P_BYTES = PT ? 0 : MT * P_TILE;   // one P buffer (PBUF are used)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QBUF * Q_BYTES;
  // V stages: one more than K's when a single M tile keeps one P buffer and one Q buffer
  static constexpr int VST = (MT == 1 && PBUF == 1 && QBUF == 1) ? STAGES + 1 : STAGES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + VST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + PBUF * P_BYTES;
  // k_full[S], k_empty[S], v_full[VST], v_empty[VST], s_full[2], s_free[2], p_full[2], p_free[2], o_free, drain,
  // xch_full[2], xl_full, pub, q_full[QBUF], q_empty[QBUF], stage_full (one M tile only)
  static constexpr int NBAR = 2 * STAGES + 2 * VST + 14 + 2 * QBUF + (MT == 1 ? 1 : 0);
  // row copies exchange partial row maxima [2][4][32] and row sums [4][32] (f32)
  static constexpr int OFF_XCH = OFF_BAR + NBAR * 8;
  static constexpr int OFF_XL = OFF_XCH + (CP > 1 ? 2 * 4 * 32 * 4 : 0);
  static constexpr int OFF_MISC = OFF_XL + (CP > 1 ? 4 * 32 * 4 : 0);
  static constexpr int OFF_RED = OFF_MISC + 16;  // [16] i64 scratch of the work split
  static constexpr int OFF_ANC = OFF_RED + 16 * 8;
  static constexpr int OFF_PAR = OFF_ANC + kMaxNodes * 8;
  static constexpr int BYTES = OFF_PAR + kMaxNodes * 4;
  static constexpr int SMEM = BYTES;  // the dynamic window starts 1024-aligned (checked)
  // S: two buffers per M tile, or (P in TMEM) one region per M tile
  static constexpr int S_COLS = (PT ? 1 : 2) * MT * BN;
  static constexpr int NEED_COLS = S_COLS + MT * D;
  static constexpr uint32_t TMEM_COLS = NEED_COLS <= 256 ? 256 : 512;
  static constexpr int NSW = 4 * MT;  // softmax warps
  static constexpr int THREADS = 32 * (NSW + 2);
  static_assert(NEED_COLS <= 512, "TMEM columns");
};

// Byte offset of 16-byte unit `rem` (of the KB * 8 in a row) of row r of a K/V tile, before
// the swizzle.  Plain layout: one block of BN rows x 128 bytes per 64-column half.  Grouped
// layout (pages loaded with both halves in one copy; D = 128): 8-row groups of 2 KB, each
// holding the 8 rows of the first half, then of the second.
template <class Lay>
__device__ __forceinline__ int kv_unit_offset(bool grouped, int r, int rem) {
  return grouped ? (r >> 3) * (Lay::KB * 1024) + (rem >> 3) * 1024 + (r & 7) * 128 + (rem & 7) * 16
                 : (rem >> 3) * Lay::KV_BLOCK + r * 128 + (rem & 7) * 16;
}

// Iterator over the pieces (unit, tile range) of one CTA's share of the work.
struct PieceIter {
  long long f, end;
  int b, ul, t, T;
};
struct Piece {
  int b, kvh, mg, t0, t1, T;
  long long unit, fs;  // unit index, flattened index of the piece's first tile
};

__device__ __forceinline__ int clamp_len(const TcParams &p, int b) {
  int L = p.prefix_len[b];
  return L < 0 ? 0 : (L > p.cap ? p.cap : L);
}

// tiles of each unit of sequence b: the tree tile, then the prefix in tiles of bn keys
__device__ __forceinline__ int unit_tiles(const TcParams &p, int b) {
  return 1 + (clamp_len(p, b) + p.bn - 1) / p.bn;
}

// Each unit occupies vt + T slots of the flattened space: vt empty slots that stand for
// the fixed cost of starting a unit (the CTA that holds a unit's start is charged for
// it and gets that many fewer tiles), then its T tiles.  it.t runs over the slots;
// pieces are reported in tile coordinates and pieces without tiles are skipped.
__device__ __forceinline__ bool piece_next(PieceIter &it, const TcParams &p, Piece &pc) {
  while (it.f < it.end) {
    const int span = it.T + p.vt;
    const int s0 = it.t;
    const int s1 = (int)min((long long)span, (long long)it.t + (it.end - it.f));
    const long long f_s0 = it.f;
    pc.b = it.b;
    pc.kvh = it.ul / p.m_groups;
    pc.mg = it.ul % p.m_groups;
    pc.T = it.T;
    pc.unit = (long long)it.b * p.upb + it.ul;
    it.f += s1 - s0;
    it.t = s1;
    if (it.t == span) {
      it.t = 0;
      if (++it.ul == p.upb) {
        it.ul = 0;
        ++it.b;
        if (it.f < it.end) it.T = unit_tiles(p, it.b);
      }
    }
    pc.t0 = max(0, s0 - p.vt);
    pc.t1 = max(0, s1 - p.vt);
    if (pc.t1 > pc.t0) {
      pc.fs = f_s0 + (pc.t0 + p.vt - s0);  // flattened index of tile t0
      return true;
    }
  }
  return false;
}

// Flattened tile at which CTA c of P starts (CTA P starts at W: the end).
__device__ __forceinline__ long long cta_first(long long W, int c, int P) { return W * c / P; }

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *a) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long *a, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

// Block-wide inclusive scan of one value per thread (warp totals in red[0..nwarps)).
__device__ __forceinline__ long long block_scan(long long x, long long *red, long long &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  long long before = 0;
  total = 0;
  for (int w = 0; w < nw; ++w) {
    const long long t = red[w];
    if (w < warp) before += t;
    total += t;
  }
  __syncthreads();
  return before + x;
}

// One piece (n tiles from tile counter g, the piece's index qi in this CTA) of a softmax
// warp whose rows are all padding.  It reads no S and writes no P or O, but takes its part
// in every barrier and in zeroing the V rows past the prefix end.  Each arrival waits for
// the previous phase of its barrier to be complete, since no write of this warp orders
// it (with P in TMEM the wait for S of M tile mt orders it).  Kept out of line so that
// the row loop's code stays small.  False if a wait gave up.
template <class Lay, int BN, int PBUF>
__device__ __noinline__ bool idle_piece(int N, int t0, int n, bool publish, int g, int qi, int L,
                                        bool grouped, int mt,
                                        uint64_t *s_full, uint64_t *s_free, uint64_t *v_full,
                                        uint64_t *p_full, uint64_t *o_free, uint64_t *pub, uint8_t *sV,
                                        volatile int *abort_flag, unsigned long long wlim) {
  const int lane = threadIdx.x & 31;
  for (int k = 0; k < n; ++k) {
    const int gk = g + k, j = gk & 1, s = gk % Lay::VST, t = t0 + k, pb = gk % PBUF;
    if constexpr (Lay::PT) {
      if (!mbar_wait(&s_full[mt], gk & 1, abort_flag, wlim)) return false;
    } else {
      if (!mbar_wait(&s_full[j], (gk >> 1) & 1, abort_flag, wlim)) return false;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[j]);
    }
    const int nvalid = t == 0 ? N : min(BN, L - (t - 1) * BN);
    // this warp's share of zeroing the V tail (see the row loop)
    if (t != 0 && nvalid < BN && (!Lay::PT || mt == 0)) {
      if (!mbar_wait(&v_full[s], (gk / Lay::VST) & 1, abort_flag, wlim)) return false;
      uint8_t *vt = sV + s * Lay::KV_BYTES;
      constexpr int per_row = Lay::KB * 8;
      constexpr int stride = 32 * (Lay::PT ? 4 : Lay::NSW);
      for (int i = threadIdx.x; i < (BN - nvalid) * per_row; i += stride) {
        const int r = nvalid + i / per_row, rem = i % per_row;
        *reinterpret_cast<uint4 *>(vt + kv_unit_offset<Lay>(grouped, r, rem)) = make_uint4(0, 0, 0, 0);
      }
    }
    if (!Lay::PT && gk >= PBUF && !mbar_wait(&p_full[pb], ((gk / PBUF) - 1) & 1, abort_flag, wlim))
      return false;
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&p_full[Lay::PT ? mt : pb]);
  }
  if (publish) {  // (nothing written: the arrival only completes the barrier)
    __syncwarp();
    if (lane == 0) mbar_arrive(pub);
  }
  if (qi > 0 && !mbar_wait(o_free, (qi - 1) & 1, abort_flag, wlim)) return false;
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(o_free);
  return true;
}

template <int D, int MT, int CP, int BN, int STAGES, int QBUF, int PBUF>
__global__ void __launch_bounds__(TcLayout<D, MT, CP, BN, STAGES, QBUF, PBUF>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p) {
  static_assert(CP == 1 || MT == 1, "row copies need a single M tile");
  static_assert(PBUF == 1 || PBUF == 2, "P buffers");
  using Lay = TcLayout<D, MT, CP, BN, STAGES, QBUF, PBUF>;
  constexpr int NSW = Lay::NSW;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  const int P = gridDim.x;
  // Completion counting: every CTA reads the call's epoch first and then counts itself
  // out; the last one to do so advances the workspace's generation for the next call.
  unsigned long long *gen = p.hdr;
  unsigned int *done = reinterpret_cast<unsigned int *>(p.hdr + 1);
  const unsigned long long epoch = *reinterpret_cast<volatile unsigned long long *>(gen) + 1ull;
  auto finish = [&]() {
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(done, 1u) == (unsigned)P - 1u) {
        *reinterpret_cast<volatile unsigned int *>(done) = 0u;
        __threadfence();
        *reinterpret_cast<volatile unsigned long long *>(gen) = epoch;
      }
    }
  };
  if (smem_u32(sm) & 1023u) {  // 128B-swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, SV_DEV_LAYOUT);
    __syncthreads();
    finish();
    return;
  }
  // the limit of every wait for progress (copies, MMAs, other CTAs' pieces); the waits
  // for work already in flight to land after an abort keep the fixed kWaitLimitNs
  const unsigned long long wlim = p.wait_ns;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::OFF_BAR);
  uint64_t *k_full = bars;
  uint64_t *k_empty = bars + STAGES;
  constexpr int VST = Lay::VST;
  uint64_t *v_full = bars + 2 * STAGES;
  uint64_t *v_empty = bars + 2 * STAGES + VST;
  uint64_t *s_full = bars + 2 * STAGES + 2 * VST;
  uint64_t *s_free = s_full + 2;
  uint64_t *p_full = s_free + 2;
  uint64_t *p_free = p_full + 2;
  uint64_t *o_free = p_free + 2;
  uint64_t *drain = o_free + 1;
  uint64_t *xch_full = drain + 1;
  uint64_t *xl_full = xch_full + 2;
  uint64_t *pub = xl_full + 1;
  uint64_t *q_full = pub + 1;
  uint64_t *q_empty = q_full + QBUF;
  uint64_t *stage_full = q_empty + QBUF;  // a head piece's first producer, staged
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + Lay::OFF_MISC + 4);
  uint64_t *sAnc = reinterpret_cast<uint64_t *>(sm + Lay::OFF_ANC);
  int *sPar = reinterpret_cast<int *>(sm + Lay::OFF_PAR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long *red = reinterpret_cast<long long *>(sm + Lay::OFF_RED);

  // ---- this CTA's share of the flattened (unit, tile) space: an equal split of the
  // total W, computed alike by every CTA from the prefix lengths; then the sequence
  // holding its first slot f0 (b_start) and the slots before that sequence (base_start)
  long long W, f0, f1;
  int b_start = 0;
  long long base_start = 0;
  if (p.B <= (int)blockDim.x) {
    // one scan: thread b holds sequence b
    const int b = threadIdx.x;
    long long w = 0;
    if (b < p.B) {
      if (blockIdx.x == 0) {
        const int L = p.prefix_len[b];
        if (L < 0 || L > p.cap) set_status(p.status, SV_DEV_BAD_PREFIX);
      }
      w = (long long)(unit_tiles(p, b) + p.vt) * p.upb;
    }
    long long total;
    const long long incl = block_scan(w, red, total);
    W = total;
    f0 = cta_first(W, blockIdx.x, P);
    f1 = cta_first(W, blockIdx.x + 1, P);
    if (b < p.B && incl - w <= f0 && f0 < incl) {
      red[14] = b;
      red[15] = incl - w;
    }
    __syncthreads();
  } else {
    long long part = 0;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      if (blockIdx.x == 0) {
        const int L = p.prefix_len[b];
        if (L < 0 || L > p.cap) set_status(p.status, SV_DEV_BAD_PREFIX);
      }
      part += unit_tiles(p, b) + p.vt;
    }
    long long total;
    block_scan(part, red, total);
    W = total * p.upb;
    f0 = cta_first(W, blockIdx.x, P);
    f1 = cta_first(W, blockIdx.x + 1, P);
    long long carry = 0;
    bool found = f0 >= f1;
    for (int b0 = 0; b0 < p.B && !found; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      const long long w = b < p.B ? (long long)(unit_tiles(p, b) + p.vt) * p.upb : 0;
      const long long incl = block_scan(w, red, total);
      const long long excl = carry + incl - w;
      if (b < p.B && excl <= f0 && f0 < excl + w) {
        red[14] = b;
        red[15] = excl;
      }
      __syncthreads();
      carry += total;
      found = carry > f0;
    }
  }
  if (f0 >= f1) {  // no work for this CTA (uniform)
    finish();
    return;
  }
  b_start = (int)red[14];
  base_start = red[15];

  if (threadIdx.x < kMaxNodes)
    sPar[threadIdx.x] = threadIdx.x < p.tree.N ? (int)p.tree.parent[threadIdx.x] : -1;
  if (threadIdx.x == 0) {
    for (int i = 0; i < VST; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    // with P in TMEM, index j is the M tile: S[j] full and free (its P V done) are MMA
    // commits, P[j] written is the arrival of that M tile's four softmax warps
    for (int j = 0; j < 2; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&s_free[j], Lay::PT ? 1 : NSW);
      mbar_init(&p_full[j], Lay::PT ? 4 : NSW);
      mbar_init(&p_free[j], 1);
      mbar_init(&xch_full[j], NSW);
    }
    mbar_init(o_free, NSW);
    mbar_init(drain, 1);
    mbar_init(xl_full, NSW);
    mbar_init(pub, NSW);
    if (MT == 1) mbar_init(stage_full, 32);
    for (int i = 0; i < QBUF; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, Lay::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == NSW && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_kt);
    prefetch_tmap(&p.tm_vt);
    prefetch_tmap(&p.tm_kc);
    prefetch_tmap(&p.tm_vc);
  }
  __syncthreads();
  if (threadIdx.x < kMaxNodes) {
    uint64_t m = 0;
    if (threadIdx.x < p.tree.N)
      for (int a = threadIdx.x; a >= 0; a = sPar[a]) m |= 1ull << a;
    sAnc[threadIdx.x] = m;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // this CTA has read the epoch: count it out now (the count only advances the generation
  // for the next call, which starts after this grid has ended); with two M tiles at the end
  if (MT == 1) finish();

  PieceIter it;
  it.f = f0;
  it.end = f1;
  it.b = b_start;
  it.T = unit_tiles(p, b_start);
  it.ul = (int)((f0 - base_start) / (it.T + p.vt));
  it.t = (int)((f0 - base_start) % (it.T + p.vt));

  uint8_t *const sQ = sm + Lay::OFF_Q;
  uint8_t *const sK = sm + Lay::OFF_K;
  uint8_t *const sV = sm + Lay::OFF_V;
  uint8_t *const sP = sm + Lay::OFF_P;

  if (warp == NSW) {
    // ------------------------------------------------------------- producer
    // K of a tile is released as soon as its S = Q K^T completes, V only when its P V
    // does; so K runs one tile ahead of V: the load of V(g-1) is issued after K(g).
    // Paged tiles use the whole warp: lane i reads the block-table entry of the tile's
    // page i (one tile ahead, so the read overlaps the waits) and copies that page.
    struct Src {
      int kind;  // 0 tree nodes, 1 contiguous cache, 2 paged cache
      int kvh, row, npg, pos0, blk;  // blk, pos0: this lane's page (paged)
    };
    int g = 0, gv = 0, nq = 0;  // K tiles, V tiles and Q pieces issued
    bool ok = true;
    // the cache is streamed once: its lines go first when L2 needs room, which keeps
    // the partial outputs of cut units resident until they are merged
    const uint64_t stream_policy = l2_policy_evict_first();
    // lane 0 waits; the outcome is shared with the warp
    auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
      int r = 1;
      if (lane == 0) r = mbar_wait(bar, parity, abort_flag, wlim) ? 1 : 0;
      return __shfl_sync(0xFFFFFFFFu, r, 0) != 0;
    };
    auto load = [&](const Src &src, int gi, bool is_v) -> bool {
      const int NS = is_v ? VST : STAGES;
      const int s = gi % NS;
      uint64_t *full = is_v ? &v_full[s] : &k_full[s];
      if (gi >= NS &&
          !wait_all(is_v ? &v_empty[s] : &k_empty[s], ((gi / NS) - 1) & 1))
        return false;
      uint8_t *dst = (is_v ? sV : sK) + s * Lay::KV_BYTES;
      const CUtensorMap *map =
          src.kind == 0 ? (is_v ? &p.tm_vt : &p.tm_kt) : (is_v ? &p.tm_vc : &p.tm_kc);
      if (src.kind != 2) {
        if (lane == 0) {
          mbar_expect_tx(full, Lay::KV_BYTES);
          for (int kb = 0; kb < Lay::KB; ++kb) {
            if (src.kind == 0)
              tma_load_3d(dst + kb * Lay::KV_BLOCK, map, kb * 64, src.kvh, src.row, full);
            else
              tma_load_3d_hint(dst + kb * Lay::KV_BLOCK, map, kb * 64, src.kvh, src.row, full,
                               stream_policy);
          }
        }
      } else {
        const bool mine = lane < src.npg;
        const bool valid = mine && src.blk >= 0 && src.blk < p.num_blocks;
        if (mine && !valid && !is_v) set_status(p.status, SV_DEV_BAD_BLOCK);
        const unsigned nvalid = __popc(__ballot_sync(0xFFFFFFFFu, valid));
        if (lane == 0)
          mbar_expect_tx(full, nvalid * (uint32_t)Lay::KB * (uint32_t)p.page_rows * 128u);
        __syncwarp();
        if (valid) {
          const int pos = src.pos0 + lane * p.page_rows;
          const int prow = src.blk * p.block_size + pos % p.block_size;
          if (p.pg_grouped) {
            // both halves of the page in one copy: rows prow .. prow + page_rows (a multiple
            // of 8) land as page_rows / 8 groups of 2 KB
            tma_load_5d_hint(dst + lane * p.page_rows * (Lay::KB * 128), is_v ? &p.tm_vc5 : &p.tm_kc5,
                             0, 0, 0, prow >> 3, src.kvh, full, stream_policy);
          } else {
            for (int kb = 0; kb < Lay::KB; ++kb)
              tma_load_3d_hint(dst + kb * Lay::KV_BLOCK + lane * p.page_rows * 128, map, kb * 64,
                               src.kvh, prow, full, stream_policy);
          }
        }
      }
      return true;
    };
    // description of tile t of piece pc; a paged tile's block-table read is issued here
    // and consumed at the tile's load
    auto make_src = [&](const Piece &pc, int t) -> Src {
      Src src;
      src.kvh = pc.kvh;
      src.npg = 0;
      src.pos0 = 0;
      src.blk = -1;
      src.row = 0;
      if (t == 0) {
        src.kind = 0;
        src.row = pc.b * p.N;
      } else if (!p.paged) {
        src.kind = 1;
        src.row = pc.b * p.Lmax + (t - 1) * BN;
      } else {
        src.kind = 2;
        src.pos0 = (t - 1) * BN;
        const int rows = min(BN, clamp_len(p, pc.b) - src.pos0);
        src.npg = (rows + p.page_rows - 1) / p.page_rows;
        if (lane < src.npg)
          src.blk = __ldg(p.block_table + (size_t)pc.b * p.max_blocks +
                          (src.pos0 + lane * p.page_rows) / p.block_size);
      }
      return src;
    };
    Src pend;
    bool have_pend = false;
    Piece pc;
    // per piece: K of its first tile and the previous tile's V go out before the wait
    // for the Q buffer (held until the previous piece's last S completes)
    Piece last;
    bool have_last = false;
    while (ok && piece_next(it, p, pc)) {
      if constexpr (MT == 1) {
        last = pc;
        have_last = true;
      }
      bool q_pending = true;
      Src nxt = make_src(pc, pc.t0);
      for (int t = pc.t0; t < pc.t1; ++t) {
        const Src src = nxt;
        if (t + 1 < pc.t1) nxt = make_src(pc, t + 1);
        if (!load(src, g, false)) {
          ok = false;
          break;
        }
        ++g;
        if (have_pend) {
          if (!load(pend, gv, true)) {
            ok = false;
            break;
          }
          ++gv;
        }
        pend = src;
        have_pend = true;
        if (q_pending) {
          const int qb = nq % QBUF;
          if (nq >= QBUF && !wait_all(&q_empty[qb], ((nq / QBUF) - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(&q_full[qb], Lay::Q_BYTES);
            for (int cp = 0; cp < CP; ++cp)  // the same rows in each of the CP row copies
              for (int kb = 0; kb < Lay::KB; ++kb)
                tma_load_3d(sQ + qb * Lay::Q_BYTES + kb * Lay::Q_BLOCK + cp * (kRows / CP) * 128,
                            &p.tm_q, kb * 64, pc.kvh * p.G,
                            pc.b * p.N + pc.mg * (MT * kRows / p.G), &q_full[qb]);
          }
          ++nq;
          q_pending = false;
        }
      }
    }
    if (ok && have_pend && load(pend, gv, true)) ++gv;
    // The CTA's last piece is a head (it holds the first tiles of a unit that later CTAs
    // continue; one M tile): once the first of those CTAs has published its partial
    // result and the last S has freed the K stages and Q, this warp copies that partial
    // O into the K area (the layout the merge reads) and its row maxima and sums into
    // the Q area, while the softmax warps finish the last tile.
    if constexpr (MT == 1) {
      if (ok && have_last && last.t0 == 0 && last.t1 < last.T) {
        const long long U_end = last.fs - last.t0 + last.T;
        long long sl0 = -1;
        for (int c2 = blockIdx.x + 1; c2 < P; ++c2) {
          const long long fa = cta_first(W, c2, P);
          if (fa >= U_end) break;
          if (fa == cta_first(W, c2 + 1, P)) continue;
          sl0 = last.unit + c2;
          break;
        }
        if (sl0 >= 0) {
          int r = 1;
          if (lane == 0) {
            const unsigned long long t0 = global_ns();
            while (ld_acquire_u64(p.flags + sl0) != epoch) {
              if (*abort_flag || global_ns() - t0 > wlim) {
                *abort_flag = 1;
                r = 0;
                break;
              }
            }
            if (r && !mbar_wait(&k_empty[(g - 1) % STAGES], ((g - 1) / STAGES) & 1, abort_flag, wlim)) r = 0;
            if (r && !mbar_wait(&q_empty[(nq - 1) % QBUF], ((nq - 1) / QBUF) & 1, abort_flag, wlim)) r = 0;
          }
          if (__shfl_sync(0xFFFFFFFFu, r, 0)) {
            (void)ld_acquire_u64(p.flags + sl0);  // each lane's own acquire of the published rows
            float4 *stage = reinterpret_cast<float4 *>(sK);
            float2 *mls = reinterpret_cast<float2 *>(sQ);
            static_assert(MT > 1 || kRows * D * 4 <= STAGES * Lay::KV_BYTES, "staging room");
            for (int row = lane; row < kRows; row += 32) {
              // 16-byte unit i of row r at r * (D / 4) + (i ^ (r % (D / 4))): a warp reading
              // one unit of 32 rows meets no bank conflict
              // (partial O is stored by 16-byte unit: unit i of all rows, then unit i + 1)
              const float4 *src = reinterpret_cast<const float4 *>(p.part_o) + (size_t)sl0 * (D / 4) * kRows + row;
              for (int i = 0; i < D / 4; ++i)
                cp_async_16(stage + (size_t)row * (D / 4) + (i ^ (row % (D / 4))), src + (size_t)i * kRows, true);
              cp_async_8(mls + row, p.part_ml + ((size_t)sl0 * kRows + row) * 2);
            }
            cp_async_mbar_arrive(stage_full);
          }
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // let copies already in flight land before the CTA retires
      const unsigned long long t0 = global_ns();
      auto settle = [&](uint64_t *bars_, int n, int depth) {
        for (int i = max(0, n - depth); i < n; ++i)
          while (!mbar_try_wait(&bars_[i % depth], (i / depth) & 1) &&
                 global_ns() - t0 < kWaitLimitNs) {
          }
      };
      settle(k_full, g, STAGES);
      settle(v_full, gv, VST);
      settle(q_full, nq, QBUF);
    }
    // this lane's staging copies (a split unit's partial rows) land before the CTA retires,
    // also when the consumer gave up waiting for them
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == NSW + 1) {
    // -------------------------------------------------------------- MMA issue
    // One thread polls both kinds of work and issues whichever is ready, P V first:
    // P V of a tile as soon as its P is written, and S = Q K^T up to two tiles ahead of
    // P V (S is double buffered), across piece boundaries.  A late K never holds back
    // a P V that is ready.  Two M tiles (P in TMEM) take the ping-pong order below.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kRows, BN, 0, 0);
      constexpr uint32_t idO = idesc_bf16(kRows, D, 0, 1);
      // descriptors of each buffer's start; offsets inside shared memory (< 256 KB) are
      // added in 16-byte units to the start-address field without carrying out of it
      const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dp = sdesc_sw128(smem_u32(sP), 16, 1024);
      const uint64_t dv = sdesc_sw128(smem_u32(sV), Lay::KV_BLOCK, 1024);
      // the grouped layout of paged prefix tiles: 8-row groups 2 KB apart, the second
      // 64-column half 1 KB after the first
      const uint64_t dk_g = sdesc_sw128(smem_u32(sK), 16, Lay::KB * 1024);
      const uint64_t dv_g = sdesc_sw128(smem_u32(sV), 1024, Lay::KB * 1024);
      // the idle poll: gives up after the wait limit (or when another role gave up)
      unsigned long long idle_t0 = 0;
      uint32_t idle_n = 0;
      auto idle = [&]() -> bool {
        if ((++idle_n & 63u) == 0) {
          if (*abort_flag) return false;
          const unsigned long long now = global_ns();
          if (idle_n == 64) idle_t0 = now;
          else if (now - idle_t0 > wlim) {
            *abort_flag = 1;
            return false;
          }
        }
        // a short sleep keeps the poll from taking issue slots from the softmax warps
        // that share this SM sub-partition
        __nanosleep(kPollSleepNs);
        return true;
      };
      if constexpr (Lay::PT) {
        // Ping-pong of the two M tiles, in a fixed order: S[0] and S[1] of the first tile,
        // then per tile k: P V of M tile 0, S[0] of tile k+1 (once that P V has completed:
        // P lives over S[0]), P V of M tile 1, S[1] of tile k+1.  One M tile's Q K^T and
        // P V run while the other M tile's softmax works.  Each step waits on its own
        // barrier (a blocking wait wakes as soon as the phase completes).
        PieceIter its = it;
        Piece pcs;
        struct TileInfo {
          bool first, last, grp;
          int qi;
        };
        int s_qi = -1, s_rem = 0;
        bool first_flag = false;
        auto next_tile = [&](TileInfo &ti) -> bool {
          if (s_rem == 0) {
            if (!piece_next(its, p, pcs)) return false;
            ++s_qi;
            s_rem = pcs.t1 - pcs.t0;
            first_flag = true;
          }
          ti.first = first_flag;
          first_flag = false;
          ti.qi = s_qi;
          // tile pcs.t1 - s_rem of its unit; tile 0 holds the tree nodes (plain layout)
          ti.grp = p.pg_grouped && pcs.t1 - s_rem != 0;
          ti.last = s_rem == 1;
          --s_rem;
          return true;
        };
        auto issue_qk = [&](const TileInfo &ti, int gk, int m) -> bool {
          const int s = gk % STAGES, qb = ti.qi % QBUF;
          if (m == 0 && ti.first && !mbar_wait(&q_full[qb], (ti.qi / QBUF) & 1, abort_flag, wlim))
            return false;
          if (m == 0 && !mbar_wait(&k_full[s], (gk / STAGES) & 1, abort_flag, wlim)) return false;
          if (gk > 0 && !mbar_wait(&s_free[m], (gk - 1) & 1, abort_flag, wlim)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = dq + (uint64_t)((qb * Lay::Q_BYTES + (kk >> 2) * Lay::Q_BLOCK +
                                                 m * kRows * 128 + (kk & 3) * 32) >> 4);
            const uint64_t bd =
                ti.grp ? dk_g + (uint64_t)((s * Lay::KV_BYTES + (kk >> 2) * 1024 + (kk & 3) * 32) >> 4)
                       : dk + (uint64_t)((s * Lay::KV_BYTES + (kk >> 2) * Lay::KV_BLOCK + (kk & 3) * 32) >> 4);
            umma_bf16(tmem + (uint32_t)(m * BN), a, bd, idS, kk > 0);
          }
          umma_commit(&s_full[m]);
          if (m == MT - 1) {
            umma_commit(&k_empty[s]);
            if (ti.last) umma_commit(&q_empty[qb]);
          }
          return true;
        };
        auto issue_pv = [&](const TileInfo &ti, int gk, int m) -> bool {
          const int s = gk % VST;
          if (!mbar_wait(&p_full[m], gk & 1, abort_flag, wlim)) return false;
          // the first P V of a piece overwrites O: the previous piece's readout is done
          if (m == 0 && ti.first && ti.qi > 0 && !mbar_wait(o_free, (ti.qi - 1) & 1, abort_flag, wlim))
            return false;
          if (m == 0 && !mbar_wait(&v_full[s], (gk / VST) & 1, abort_flag, wlim)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd =
                ti.grp ? dv_g + (uint64_t)((s * Lay::KV_BYTES + kk * 2 * (Lay::KB * 1024)) >> 4)
                       : dv + (uint64_t)((s * Lay::KV_BYTES + kk * 16 * 128) >> 4);
            // 16 keys of P per MMA: 8 TMEM columns of bf16 pairs
            umma_bf16_ts(tmem + (uint32_t)(Lay::S_COLS + m * D), tmem + (uint32_t)(m * BN + kk * 8), bd,
                         idO, (!ti.first || kk > 0) ? 1u : 0u);
          }
          umma_commit(&s_free[m]);
          if (m == MT - 1) umma_commit(&v_empty[s]);
          return true;
        };
        TileInfo cur, nxt;
        bool have = next_tile(cur);
        bool ok = !have || (issue_qk(cur, 0, 0) && issue_qk(cur, 0, 1));
        for (int gk = 0; ok && have; ++gk) {
          const bool more = next_tile(nxt);
          ok = issue_pv(cur, gk, 0) && (!more || issue_qk(nxt, gk + 1, 0)) && issue_pv(cur, gk, 1) &&
               (!more || issue_qk(nxt, gk + 1, 1));
          cur = nxt;
          have = more;
        }
      } else {
        PieceIter its = it;  // S side of the walk over this CTA's tiles
        Piece pcs;
        int s_qi = -1, s_rem = 0, gs = 0, gp = 0;
        bool s_first = false, s_done = false;
        uint8_t m_first[4], m_grp[4];
        int m_qi[4];
        while (true) {
          bool prog = false;
          if (gp < gs) {
            const int gk = gp, s = gk % VST, pb = gk % PBUF;
            const bool first = m_first[gk & 3];
            const bool grp = m_grp[gk & 3];
            const int qi = m_qi[gk & 3];
            if (mbar_test(&p_full[pb], (gk / PBUF) & 1) &&
                (!first || qi == 0 || mbar_test(o_free, (qi - 1) & 1)) &&
                mbar_test(&v_full[s], (gk / VST) & 1)) {
              tc_fence_after();
#pragma unroll
              for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                  const uint64_t a = dp + (uint64_t)((pb * Lay::P_BYTES + m * Lay::P_TILE +
                                                       (kk >> 2) * Lay::P_BLOCK + (kk & 3) * 32) >> 4);
                  const uint64_t bd =
                      grp ? dv_g + (uint64_t)((s * Lay::KV_BYTES + kk * 2 * (Lay::KB * 1024)) >> 4)
                          : dv + (uint64_t)((s * Lay::KV_BYTES + kk * 16 * 128) >> 4);
                  umma_bf16(tmem + (uint32_t)(Lay::S_COLS + m * D), a, bd, idO,
                            (!first || kk > 0) ? 1u : 0u);
                }
              }
              umma_commit(&v_empty[s]);
              umma_commit(&p_free[pb]);
              ++gp;
              prog = true;
            }
          }
          if (!s_done && gs < gp + 2) {
            if (s_rem == 0) {
              if (piece_next(its, p, pcs)) {
                ++s_qi;
                s_rem = pcs.t1 - pcs.t0;
                s_first = true;
              } else {
                s_done = true;
              }
            }
            const int gk = gs, s = gk % STAGES, j = gk & 1, qb = s_qi % QBUF;
            if (!s_done && (!s_first || mbar_test(&q_full[qb], (s_qi / QBUF) & 1)) &&
                mbar_test(&k_full[s], (gk / STAGES) & 1) &&
                (gk < 2 || mbar_test(&s_free[j], ((gk >> 1) - 1) & 1))) {
              tc_fence_after();
              // tile pcs.t1 - s_rem of its unit; tile 0 holds the tree nodes (plain layout)
              const bool grp = p.pg_grouped && pcs.t1 - s_rem != 0;
#pragma unroll
              for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint64_t a = dq + (uint64_t)((qb * Lay::Q_BYTES + (kk >> 2) * Lay::Q_BLOCK +
                                                       m * kRows * 128 + (kk & 3) * 32) >> 4);
                  const uint64_t bd =
                      grp ? dk_g + (uint64_t)((s * Lay::KV_BYTES + (kk >> 2) * 1024 + (kk & 3) * 32) >> 4)
                          : dk + (uint64_t)((s * Lay::KV_BYTES + (kk >> 2) * Lay::KV_BLOCK + (kk & 3) * 32) >> 4);
                  umma_bf16(tmem + (uint32_t)((j * MT + m) * BN), a, bd, idS, kk > 0);
                }
              }
              umma_commit(&s_full[j]);
              umma_commit(&k_empty[s]);
              if (s_rem == 1) umma_commit(&q_empty[qb]);
              m_first[gk & 3] = s_first;
              m_grp[gk & 3] = grp;
              m_qi[gk & 3] = s_qi;
              s_first = false;
              --s_rem;
              ++gs;
              prog = true;
            }
          }
          if (s_done && gp == gs) break;
          if (prog) {
            idle_n = 0;
            continue;
          }
          // nothing ready: give up after the wait limit (or when another role gave up)
          if (!idle()) break;
        }
      }
      // every MMA issued must complete before TMEM is released
      umma_commit(drain);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    // Warp w reads TMEM lane quarter w&3 of M tile w>>2.  With CP > 1 row copies the
    // warps of copy c take columns [c*CW, (c+1)*CW) of each tile, combine their partial
    // row maxima through shared memory and write their slice of the one P row; copy 0's
    // warps own the O rows (lanes 0 .. 128/CP-1).  Columns go in chunks of 32: a first
    // pass over TMEM finds the row maximum, a second forms P.
    constexpr int CW = BN / CP;   // columns per warp
    constexpr int QPC = 4 / CP;   // lane quarters per copy
    constexpr int CH = CW < 32 ? CW : 32;  // columns per TMEM read
    constexpr int NCH = CW / CH;
    const int mt = warp >> 2, wq = warp & 3;
    const int copy = wq / QPC;
    const int row = (wq % QPC) * 32 + lane;  // row of the M tile (lane of copy 0)
    const int col0 = copy * CW;
    const bool owner = copy == 0;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    float *xch = reinterpret_cast<float *>(sm + Lay::OFF_XCH);
    float *xl = reinterpret_cast<float *>(sm + Lay::OFF_XL);
    const int tid_sm = threadIdx.x;  // 0 .. 128*MT-1
    const float sc = p.scale_log2;
    int g = 0, qi = 0;
    Piece pc;
    bool ok = true;
    auto read_chunk = [&](uint32_t ta, float (&v)[CH]) {
      if constexpr (CH == 32) {
        tmem_ld32(ta, v);
      } else {
        tmem_ld16(ta, v);
      }
      tmem_wait_ld();
    };
    while (ok && piece_next(it, p, pc)) {
      const int n = pc.t1 - pc.t0;
      const int R_local = mt * kRows + row;
      const int R = pc.mg * (MT * kRows) + R_local;
      const bool valid_row = R < p.M;
      const int node = valid_row ? R / p.G : 0;
      // the node's ancestor mask: the shared tree's, or a walk of sequence b's own row
      uint64_t anc = 0ull;
      if (valid_row) {
        if (p.tree.rows) {
          int dep;
          if (!tree_walk_seq(p.tree, pc.b, node, &anc, &dep)) set_status(p.status, SV_DEV_BAD_TREE);
        } else {
          anc = sAnc[node];
        }
      }
      const bool warp_idle = CP == 1 && __all_sync(0xFFFFFFFFu, !valid_row);
      const int L = clamp_len(p, pc.b);
      if (warp_idle) {  // every row of this warp is padding: barriers only
        if (!idle_piece<Lay, BN, PBUF>(p.N, pc.t0, n, pc.t0 > 0, g, qi, L, p.pg_grouped != 0, mt,
                                              s_full, s_free, v_full,
                                              p_full, o_free, pub, sV, abort_flag, wlim)) {
          ok = false;
          break;
        }
        g += n;
        ++qi;
        continue;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int k = 0; k < n; ++k) {
        const int gk = g + k, j = gk & 1, s = gk % VST, t = pc.t0 + k, pb = gk % PBUF;
        const bool tree = t == 0;
        const int nvalid = tree ? p.N : min(BN, L - (t - 1) * BN);
        // S of this tile: buffer j, or (P in TMEM) this M tile's region, one phase per tile
        if (!(Lay::PT ? mbar_wait(&s_full[mt], gk & 1, abort_flag, wlim)
                      : mbar_wait(&s_full[j], (gk >> 1) & 1, abort_flag, wlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // V rows past the prefix end may hold anything: zero them so that 0 * V stays 0.
        // Done by all softmax threads once V has landed, before P is published.  With P in
        // TMEM, by the warps of M tile 0, whose P V is issued first.
        auto zero_v_tail = [&]() -> bool {
          if (tree || nvalid >= BN || (Lay::PT && mt != 0)) return true;
          if (!mbar_wait(&v_full[s], (gk / VST) & 1, abort_flag, wlim)) return false;
          uint8_t *vt = sV + s * Lay::KV_BYTES;
          constexpr int per_row = Lay::KB * 8;
          constexpr int stride = 32 * (Lay::PT ? 4 : NSW);
          const bool grouped = p.pg_grouped != 0;  // (a prefix tile)
          for (int i = tid_sm; i < (BN - nvalid) * per_row; i += stride) {
            const int r = nvalid + i / per_row, rem = i % per_row;
            *reinterpret_cast<uint4 *>(vt + kv_unit_offset<Lay>(grouped, r, rem)) = make_uint4(0, 0, 0, 0);
          }
          return true;
        };
        // visible columns of this warp's slice: tree tile -> ancestor bits, prefix
        // tile -> columns before the prefix end
        const uint64_t anc_s = (tree && valid_row && col0 < 64) ? (anc >> col0) : 0ull;
        const int nv_rel = (tree || !valid_row) ? 0 : nvalid - col0;
        const bool full = !tree && valid_row && nv_rel >= CW;
        const uint32_t ta0 = t_lane + (uint32_t)(((Lay::PT ? 0 : j * MT) + mt) * BN + col0);

        // bit c of visible(h) <=> column h*CH + c of this warp's slice is a key the row sees.
        // Padding rows (past the unit's rows) see every column: their results are never
        // used, and this keeps a warp that mixes real and padding rows on one code path.
        constexpr uint32_t kAll = CH == 32 ? 0xFFFFFFFFu : (1u << CH) - 1u;
        auto visible = [&](int h) -> uint32_t {
          if (full || !valid_row) return kAll;
          const int sh = h * CH;
          if (tree) return sh < 64 ? (uint32_t)(anc_s >> sh) & kAll : 0u;
          const int r = nv_rel - sh;
          return r <= 0 ? 0u : (r >= CH ? kAll : (1u << r) - 1u);
        };

        // the row maximum over chunk h's visible columns
        auto chunk_max = [&](int h, const float (&v)[CH]) -> float {
          const uint32_t km = visible(h);
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
          if (km == kAll) {
#pragma unroll
            for (int c = 0; c < CH; c += 2) mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], v[c], v[c + 1]);
          } else {
#pragma unroll
            for (int c = 0; c < CH; ++c) mx[c & 7] = fmaxf(mx[c & 7], ((km >> c) & 1u) ? v[c] : -INFINITY);
          }
          return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        };
        // The row's columns are read from TMEM twice (max, then P), 32 at a time, and S is
        // released with P: releasing it early lets the next S take the tensor pipe ahead
        // of this tile's P V, which costs more than it gains.  (With P in TMEM, P goes over
        // columns already read in the second pass, and S is free once P V has completed.)
        constexpr bool kOnePass = false;
        float vs[kOnePass ? CW : 1];
        auto vchunk = [&](int h) -> float (&)[CH] { return *reinterpret_cast<float(*)[CH]>(vs + h * CH); };
        float pmax = -INFINITY;
        if constexpr (kOnePass) {
#pragma unroll
          for (int h = 0; h < NCH; ++h) {
            if constexpr (CH == 32) tmem_ld32(ta0 + h * CH, vchunk(h));
            else tmem_ld16(ta0 + h * CH, vchunk(h));
          }
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NCH; ++h) pmax = fmaxf(pmax, chunk_max(h, vchunk(h)));
        } else {
#pragma unroll 1
          for (int h = 0; h < NCH; ++h) {
            float v[CH];
            read_chunk(ta0 + h * CH, v);
            pmax = fmaxf(pmax, chunk_max(h, v));
          }
        }
        if constexpr (CP > 1) {
          // the row's maximum over all copies' columns
          float *xb = xch + (gk & 1) * 4 * 32;
          xb[wq * 32 + lane] = pmax;
          __syncwarp();
          if (lane == 0) mbar_arrive(&xch_full[gk & 1]);
          if (!mbar_wait(&xch_full[gk & 1], (gk >> 1) & 1, abort_flag, wlim)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int c2 = 0; c2 < CP; ++c2) pmax = fmaxf(pmax, xb[(c2 * QPC + (wq % QPC)) * 32 + lane]);
        }
        // raw maximum times the (positive) scale = maximum in log2 units
        const float tmax = sc * pmax;
        float alpha = 1.f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = tmax;
        } else if (tmax > m_ref + kRescaleThreshold) {
          alpha = ex2(m_ref - tmax);
          m_ref = tmax;
          rescale = true;
        }
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;

        // O is rescaled in place only when the running max jumped: all earlier P V of
        // this piece must have finished first (P V runs in order, so waiting for the
        // previous tile's buffer release is enough; with P in TMEM, this tile's S was
        // computed only after the previous P V of this M tile completed)
        if (owner && __any_sync(0xFFFFFFFFu, rescale)) {
          if (!Lay::PT &&
              !mbar_wait(&p_free[(gk - 1) % PBUF], ((gk - 1) / PBUF) & 1, abort_flag, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float o[32];
            const uint32_t ta = t_lane + (uint32_t)(Lay::S_COLS + mt * D + ch * 32);
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] *= alpha;
            tmem_st32(ta, o);
          }
          tmem_wait_st();
        }
        // P buffer gk&1 is free once the P V of tile gk-2 has finished
        if (!Lay::PT && gk >= PBUF && !mbar_wait(&p_free[pb], ((gk / PBUF) - 1) & 1, abort_flag, wlim)) {
          ok = false;
          break;
        }
        // 2^(s*scale - max) of a whole chunk, the scale and the subtraction on fp32 pairs;
        // partial row sums in rs (pairs of lanes 0/1 and 2/3)
        auto exp_pairs = [&](float (&v)[CH], float (&rs)[4]) {
          const float2 sc2 = make_float2(sc, sc), nmu2 = make_float2(-mu, -mu);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < CH; c += 2) {
            const float2 x = __ffma2_rn(make_float2(v[c], v[c + 1]), sc2, nmu2);
            v[c] = ex2(x.x);
            v[c + 1] = ex2(x.y);
            if ((c >> 1) & 1) acc1 = __fadd2_rn(acc1, make_float2(v[c], v[c + 1]));
            else acc0 = __fadd2_rn(acc0, make_float2(v[c], v[c + 1]));
          }
          rs[0] += acc0.x;
          rs[1] += acc0.y;
          rs[2] += acc1.x;
          rs[3] += acc1.y;
        };
        // P = 2^(s*scale - max) in bf16 into this warp's slice of the P row
        uint8_t *ptile = sP + pb * Lay::P_BYTES + mt * Lay::P_TILE;
        auto chunk_exp = [&](int h, float (&v)[CH]) -> float {
          const uint32_t km = visible(h);
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
          if (km == kAll) {
            exp_pairs(v, rs);
          } else {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
              v[c] = ((km >> c) & 1u) ? ex2(fmaf(v[c], sc, -mu)) : 0.f;
              rs[c & 3] += v[c];
            }
          }
#pragma unroll
          for (int c8 = 0; c8 < CH / 8; ++c8) {
            const int a = (col0 + h * CH) / 8 + c8;  // 8-key chunk index in the row
            uint4 w;
            w.x = pack_bf16x2(v[c8 * 8 + 0], v[c8 * 8 + 1]);
            w.y = pack_bf16x2(v[c8 * 8 + 2], v[c8 * 8 + 3]);
            w.z = pack_bf16x2(v[c8 * 8 + 4], v[c8 * 8 + 5]);
            w.w = pack_bf16x2(v[c8 * 8 + 6], v[c8 * 8 + 7]);
            *reinterpret_cast<uint4 *>(ptile + (a >> 3) * Lay::P_BLOCK +
                                       sw128_offset((uint32_t)row, (uint32_t)(a & 7))) = w;
          }
          return (rs[0] + rs[1]) + (rs[2] + rs[3]);
        };
        // With P in TMEM: P of chunk h as bf16 pairs over TMEM columns [h*CH/2, (h+1)*CH/2)
        // of this row's S region, which hold S columns of chunks h/2 and earlier, already read
        auto chunk_exp_tmem = [&](int h, float (&v)[CH]) -> float {
          static_assert(CH == 32, "P in TMEM takes 32-column chunks");
          const uint32_t km = visible(h);
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
          if (km == kAll) {
            exp_pairs(v, rs);
          } else {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
              v[c] = ((km >> c) & 1u) ? ex2(fmaf(v[c], sc, -mu)) : 0.f;
              rs[c & 3] += v[c];
            }
          }
          float pw[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pw[c] = __uint_as_float(pack_bf16x2(v[2 * c], v[2 * c + 1]));
          tmem_st16(ta0 + (uint32_t)(h * 16), pw);
          return (rs[0] + rs[1]) + (rs[2] + rs[3]);
        };
        float rsum = 0.f;
        if constexpr (kOnePass) {
#pragma unroll
          for (int h = 0; h < NCH; ++h) rsum += chunk_exp(h, vchunk(h));
        } else {
#pragma unroll 1
          for (int h = 0; h < NCH; ++h) {
            float v[CH];
            read_chunk(ta0 + h * CH, v);
            if constexpr (Lay::PT) rsum += chunk_exp_tmem(h, v);
            else rsum += chunk_exp(h, v);
          }
        }
        l = l * alpha + rsum;
        if (!zero_v_tail()) {
          ok = false;
          break;
        }
        if constexpr (Lay::PT) tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (!kOnePass && !Lay::PT) mbar_arrive(&s_free[j]);
          mbar_arrive(&p_full[Lay::PT ? mt : pb]);
        }
      }
      if (!ok) break;

      // end of the piece: the row sum over all copies, then O of every row (copy 0)
      const int gl = g + n - 1;
      if constexpr (CP > 1) {
        xl[wq * 32 + lane] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(xl_full);
        if (!mbar_wait(xl_full, qi & 1, abort_flag, wlim)) break;
        if (owner) {
          l = 0.f;
#pragma unroll
          for (int c2 = 0; c2 < CP; ++c2) l += xl[(c2 * QPC + (wq % QPC)) * 32 + lane];
        }
      }
      // A unit cut by CTA boundaries: each later piece (t0 > 0, always the first piece
      // of its CTA) leaves (max, sum, O) in fp32 and publishes it; the CTA holding the
      // unit's first tiles (its last piece) merges them into the output.
      const bool whole = pc.t0 == 0 && pc.t1 == pc.T;
      const bool head = pc.t0 == 0 && !whole;
      const long long U_end = pc.fs - pc.t0 + pc.T;
      constexpr int ROWS = MT * kRows;
      if (owner && !warp_idle) {
        // the piece's last P V has completed (with P in TMEM: that of this M tile)
        if (!(Lay::PT ? mbar_wait(&s_free[mt], gl & 1, abort_flag, wlim)
                      : mbar_wait(&p_free[gl % PBUF], (gl / PBUF) & 1, abort_flag, wlim)))
          break;
        tc_fence_after();
        const int hq = pc.kvh * p.G + (valid_row ? R % p.G : 0);
        bf16 *dst = static_cast<bf16 *>(p.out) + (((size_t)pc.b * p.N + node) * p.Hq + hq) * D;
        float w_own = 1.f, inv = l > 0.f ? 1.f / l : 0.f;
        // producers of a head piece: the later CTAs c2 whose share overlaps the unit; the
        // first kPre are kept in registers (slot and weight) and the first one's partial
        // O is prefetched a chunk ahead; any further ones are read in place
        constexpr int kPre = 4;
        int np = 0;
        long long pslot[kPre];
        float pw[kPre];
        auto for_producers = [&](auto &&fn) {
          int j = 0;
          for (int c2 = blockIdx.x + 1; c2 < P; ++c2) {
            const long long fa = cta_first(W, c2, P);
            if (fa >= U_end) break;
            if (fa == cta_first(W, c2 + 1, P)) continue;
            if (!fn(j++, pc.unit + c2)) break;
          }
        };
        if (head && valid_row) {
          // wait for the later pieces, then weigh every piece by 2^(m_piece - M)
          float M = m_ref;
          float pm[kPre], pl[kPre];
          for_producers([&](int j, long long sl) -> bool {
            float2 ml;
            if (MT == 1 && j == 0) {
              // staged by the producer warp (after it saw the flag)
              if (!mbar_wait(stage_full, 0, abort_flag, wlim)) return false;
              ml = reinterpret_cast<const float2 *>(sQ)[R_local];
            } else {
              const unsigned long long *flag = p.flags + sl;
              const unsigned long long t0 = global_ns();
              while (ld_acquire_u64(flag) != epoch) {
                if (*abort_flag || global_ns() - t0 > wlim) {
                  *abort_flag = 1;
                  return false;
                }
              }
              ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + ((size_t)sl * ROWS + R_local) * 2));
            }
#pragma unroll
            for (int k = 0; k < kPre; ++k)
              if (k == j) pslot[k] = sl, pm[k] = ml.x, pl[k] = ml.y;
            M = fmaxf(M, ml.x);
            np = j + 1;
            return true;
          });
          if (*abort_flag) break;
          w_own = m_ref == -INFINITY ? 0.f : exp2f(m_ref - M);
          float L = l * w_own;
#pragma unroll
          for (int k = 0; k < kPre; ++k) {
            pw[k] = 0.f;
            if (k < np && pm[k] != -INFINITY) {
              pw[k] = exp2f(pm[k] - M);
              L += pw[k] * pl[k];
            }
          }
          if (np > kPre)
            for_producers([&](int j, long long sl) -> bool {
              if (j < kPre) return true;
              const float2 ml =
                  __ldcg(reinterpret_cast<const float2 *>(p.part_ml + ((size_t)sl * ROWS + R_local) * 2));
              if (ml.x != -INFINITY) L += exp2f(ml.x - M) * ml.y;
              return true;
            });
          inv = L > 0.f ? 1.f / L : 0.f;
          m_ref = M;  // the weights below are 2^(m_piece - M)
        }
        // The first producer's partial rows were staged in shared memory by the producer
        // warp (one M tile only); 16-byte unit i of row r at r * (D / 4) + (i ^ (r % (D / 4))).
        float4 *stage = nullptr;
        if (MT == 1 && head && valid_row && np > 0)
          stage = reinterpret_cast<float4 *>(sK) + (size_t)R_local * (D / 4);
        __syncwarp();  // tcgen05.ld below is warp-collective
        const long long slot = pc.unit + blockIdx.x;
        // partial O by 16-byte unit (unit i of all ROWS rows, then unit i + 1): a warp's
        // stores and loads of one unit cover 32 consecutive rows, 512 contiguous bytes
        float4 *pdst = reinterpret_cast<float4 *>(p.part_o) + (size_t)slot * (D / 4) * ROWS + R_local;
        auto punit = [&](long long sl, int i) -> const float4 * {
          return reinterpret_cast<const float4 *>(p.part_o) + ((size_t)sl * (D / 4) + i) * ROWS + R_local;
        };
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float4 cur[8];
          if (stage) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) cur[c4] = stage[(ch * 8 + c4) ^ (R_local % (D / 4))];
          }
          float o[32];
          tmem_ld32(t_lane + (uint32_t)(Lay::S_COLS + mt * D + ch * 32), o);
          tmem_wait_ld();
          if (!valid_row) continue;
          if (pc.t0 > 0) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              pdst[(size_t)(ch * 8 + c4) * ROWS] = make_float4(o[c4 * 4], o[c4 * 4 + 1], o[c4 * 4 + 2], o[c4 * 4 + 3]);
            continue;
          }
          if (head) {
            auto add = [&](float w2, const float4 *src) {
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4) {
                const float4 x = src[c4];
                o[c4 * 4 + 0] += w2 * x.x;
                o[c4 * 4 + 1] += w2 * x.y;
                o[c4 * 4 + 2] += w2 * x.z;
                o[c4 * 4 + 3] += w2 * x.w;
              }
            };
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] *= w_own;
            if (stage) add(pw[0], cur);
#pragma unroll
            for (int k = stage ? 1 : 0; k < kPre; ++k) {
              if (k < np) {
                float4 x[8];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) x[c4] = __ldcg(punit(pslot[k], ch * 8 + c4));
                add(pw[k], x);
              }
            }
            if (np > kPre)
              for_producers([&](int j, long long sl) -> bool {
                if (j < kPre) return true;
                const size_t row = (size_t)sl * ROWS + R_local;
                const float m2 = __ldcg(p.part_ml + row * 2);
                if (m2 == -INFINITY) return true;
                float4 x[8];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) x[c4] = __ldcg(punit(sl, ch * 8 + c4));
                add(exp2f(m2 - m_ref), x);
                return true;
              });
          }
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint4 v;
            v.x = pack_bf16x2(o[c8 * 8 + 0] * inv, o[c8 * 8 + 1] * inv);
            v.y = pack_bf16x2(o[c8 * 8 + 2] * inv, o[c8 * 8 + 3] * inv);
            v.z = pack_bf16x2(o[c8 * 8 + 4] * inv, o[c8 * 8 + 5] * inv);
            v.w = pack_bf16x2(o[c8 * 8 + 6] * inv, o[c8 * 8 + 7] * inv);
            *reinterpret_cast<uint4 *>(dst + ch * 32 + c8 * 8) = v;
          }
        }
        if (valid_row && pc.t0 > 0) {
          float *ml = p.part_ml + ((size_t)slot * ROWS + R_local) * 2;
          ml[0] = m_ref;
          ml[1] = l;
        }
      }
      // O has been read out of TMEM: the next piece's P V may overwrite it (before the
      // publication below, which touches global memory only)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      if (pc.t0 > 0) {
        // publish this piece once every softmax warp has written its rows: the arrivals
        // (release, CTA scope) order each warp's writes before thread 0's wait, and thread
        // 0's fence and release store make them visible with the flag (cumulatively)
        __syncwarp();
        if (lane == 0) mbar_arrive(pub);
        if (threadIdx.x == 0 && mbar_wait(pub, 0, abort_flag, wlim)) {
          __threadfence();
          st_release_u64(p.flags + pc.unit + blockIdx.x, epoch);
        }
      }
      g += n;
      ++qi;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, Lay::TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, SV_DEV_TIMEOUT);
  if (MT == 2) finish();
}

template <int D, int MT, int CP, int BN, int STAGES, int QBUF, int PBUF>
cudaError_t launch_tc_typed(const TcParams &p, int grid, cudaStream_t s) {
  using Lay = TcLayout<D, MT, CP, BN, STAGES, QBUF, PBUF>;
  static_assert(Lay::SMEM <= 232448, "shared memory layout exceeds 227 KB");
  static std::atomic<bool> attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, MT, CP, BN, STAGES, QBUF, PBUF>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr[dev].store(true);
  }
  // all CTAs must be resident together: a CTA may wait for pieces of later CTAs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Lay::THREADS);
  cfg.dynamicSmemBytes = Lay::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, MT, CP, BN, STAGES, QBUF, PBUF>, p);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D bf16 view (D, heads, rows) with a (64, box1, box2) box, 128-byte swizzle.
bool map3d(CUtensorMap *m, const void *base, int D, int heads, long long rows, int box1,
           int box2) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * heads};
  cuuint32_t box[3] = {64u, (cuuint32_t)box1, (cuuint32_t)box2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// The pages of a paged cache as a 5-D bf16 view (64 columns, 8 rows, 2 column halves,
// groups of 8 rows, heads) with a (64, 8, 2, page_rows / 8, 1) box, 128-byte swizzle: one
// copy brings both 64-column halves of a page, as page_rows / 8 groups of 2 KB (the grouped
// tile layout).  D = 128 only.  rows must be a multiple of 8.
bool map5d_pages(CUtensorMap *m, const void *base, int heads, long long rows, int page_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc || rows % 8 != 0 || page_rows % 8 != 0 || page_rows / 8 > 256) return false;
  const cuuint64_t row_bytes = (cuuint64_t)128 * 2 * heads;  // one position, all heads
  cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)(rows / 8), (cuuint64_t)heads};
  cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, 256};
  cuuint32_t box[5] = {64u, 8u, 2u, (cuuint32_t)(page_rows / 8), 1u};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool tc_eligible(sv_dtype dt, int N, int Hq, int Hkv, int D, int paged_block_size) {
  if (dt != SV_BF16 || (D != 64 && D != 128) || N > 64 || Hkv < 1 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  if (G < 1 || G > 128 || 128 % G != 0) return false;
  if (paged_block_size > 0) {
    // a tile's rows must be whole pages or whole 128-row spans of a page
    const int bs = paged_block_size;
    if (!(bs == 16 || bs == 32 || bs == 64 || (bs >= 128 && bs % 128 == 0))) return false;
  }
  return encoder() != nullptr;
}

TcPlan tc_plan(int B, int N, int Hq, int Hkv, int D, int num_sms) {
  TcPlan pl{};
  const int G = Hq / Hkv;
  const int M = N * G;
  pl.MT = M > kRows ? 2 : 1;
  // row copies spread a small M over all four TMEM lane quarters (see the kernel)
  pl.CP = 1;
  if (pl.MT == 1 && M <= 32 && 32 % G == 0) pl.CP = 4;
  else if (pl.MT == 1 && M <= 64 && 64 % G == 0) pl.CP = 2;
  pl.BN = 128;  // keys per tile
  pl.m_groups = (M + pl.MT * kRows - 1) / (pl.MT * kRows);
  pl.grid = num_sms > 0 ? num_sms : 152;
  const long long units = (long long)B * Hkv * pl.m_groups;
  const long long slots = units + pl.grid;
  const int rows = pl.MT * kRows;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  pl.off_hdr = 0;
  pl.off_flags = 256;
  pl.off_ml = pl.off_flags + up((size_t)slots * 8);
  pl.off_o = pl.off_ml + up((size_t)slots * rows * 2 * 4);
  pl.ws_bytes = pl.off_o + up((size_t)slots * rows * D * 4);
  return pl;
}

cudaError_t launch_attention_tc(const AttnParams &a, const TcPlan &pl, void *ws, cudaStream_t s) {
  TcParams p{};
  const int G = a.G;
  const int rows_q = pl.MT * kRows / pl.CP;  // query rows per TMA box (one row copy)
  const int BN = pl.BN;
  if (!map3d(&p.tm_q, a.q, a.D, a.Hq, (long long)a.B * a.N, G, rows_q / G) ||
      !map3d(&p.tm_kt, a.k_tree, a.D, a.Hkv, (long long)a.B * a.N, 1, BN) ||
      !map3d(&p.tm_vt, a.v_tree, a.D, a.Hkv, (long long)a.B * a.N, 1, BN))
    return cudaErrorInvalidValue;
  if (a.block_table == nullptr) {
    const long long rows = (long long)a.B * (a.Lmax > 0 ? a.Lmax : 1);
    if (!map3d(&p.tm_kc, a.cache_k, a.D, a.Hkv, rows, 1, BN) ||
        !map3d(&p.tm_vc, a.cache_v, a.D, a.Hkv, rows, 1, BN))
      return cudaErrorInvalidValue;
    p.paged = 0;
    p.page_rows = BN;
  } else {
    p.page_rows = a.block_size < BN ? a.block_size : BN;
    const long long rows = (long long)a.num_blocks * a.block_size;
    if (!map3d(&p.tm_kc, a.cache_k, a.D, a.Hkv, rows, 1, p.page_rows) ||
        !map3d(&p.tm_vc, a.cache_v, a.D, a.Hkv, rows, 1, p.page_rows))
      return cudaErrorInvalidValue;
    p.paged = 1;
    // pages shorter than a tile: one copy per page (both column halves) instead of two,
    // into the grouped layout; the plain layout stays when the 5-D view is not available
    p.pg_grouped = a.D == 128 && p.page_rows < BN &&
                   map5d_pages(&p.tm_kc5, a.cache_k, a.Hkv, rows, p.page_rows) &&
                   map5d_pages(&p.tm_vc5, a.cache_v, a.Hkv, rows, p.page_rows);
  }
  uint8_t *w = static_cast<uint8_t *>(ws);
  p.hdr = reinterpret_cast<unsigned long long *>(w + pl.off_hdr);
  p.flags = reinterpret_cast<unsigned long long *>(w + pl.off_flags);
  p.part_ml = reinterpret_cast<float *>(w + pl.off_ml);
  p.part_o = reinterpret_cast<float *>(w + pl.off_o);
  p.prefix_len = a.prefix_len;
  p.block_table = a.block_table;
  p.out = a.out;
  p.status = a.status;
  p.B = a.B;
  p.N = a.N;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.M = a.N * G;
  p.m_groups = pl.m_groups;
  p.upb = a.Hkv * pl.m_groups;
  p.bn = BN;
  p.vt = (long long)a.B * p.upb <= 2LL * pl.grid ? kUnitStartSlots : 0;
  p.Lmax = a.Lmax;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.cap = a.cap;
  p.scale_log2 = a.scale_log2;
  p.tree = a.tree;
  p.wait_ns = a.wait_ns;
  if (a.D == 128) {
    // One M tile: one P buffer, its room spent on a third V stage (ragged-paged 763 us
    // against 775 with two P buffers) or, with two row copies, on a second Q buffer, so
    // that the next piece's Q is loaded before the current piece ends (medusa-t64 66.7
    // us against 68.2 with the third V stage; ragged-paged, four row copies, 774 against
    // 764 the other way round).
    if (pl.MT == 2) return launch_tc_typed<128, 2, 1, 128, 2, 1, 1>(p, pl.grid, s);
    if (pl.CP == 4) return launch_tc_typed<128, 1, 4, 128, 2, 1, 1>(p, pl.grid, s);
    if (pl.CP == 2) return launch_tc_typed<128, 1, 2, 128, 2, 2, 1>(p, pl.grid, s);
    return launch_tc_typed<128, 1, 1, 128, 2, 1, 1>(p, pl.grid, s);
  }
  if (pl.MT == 2) return launch_tc_typed<64, 2, 1, 128, 4, 2, 1>(p, pl.grid, s);
  if (pl.CP == 4) return launch_tc_typed<64, 1, 4, 128, 3, 2, 2>(p, pl.grid, s);
  if (pl.CP == 2) return launch_tc_typed<64, 1, 2, 128, 3, 2, 2>(p, pl.grid, s);
  return launch_tc_typed<64, 1, 1, 128, 3, 2, 2>(p, pl.grid, s);
}

}  // namespace sv
