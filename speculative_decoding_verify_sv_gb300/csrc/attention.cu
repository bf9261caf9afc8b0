// Tree attention of a flattened candidate tree against the KV prefix (sm_103a).
//
// For every sequence b, node n and query head h (KV head g = h / (Hq/Hkv)) the keys are
// the prefix positions [0, L_b) plus the tree nodes on n's root path (the ancestor
// bitmask of the tree-attention section of "推测解码技术详解"; a node's context is its
// root path, lpnh.cn Medusa walkthrough section 3.2).
//
// bf16 path: one CTA per (64 query rows, prefix split, kv head, sequence).  The query
// rows of a KV head are the (node, group head) pairs, so the GQA group and the tree's
// nodes form the M side of a dense contraction; K/V tiles of 64 keys stream through a
// cp.async pipeline and both products run on bf16 tensor cores with fp32 accumulators
// and an online softmax.  Splits of the prefix merge in a second kernel by
// log-sum-exp weights.
#include <atomic>
#include <cfloat>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kTileKeys = 64;
constexpr int kRowsPerCta = 64;
constexpr int kStages = 3;
constexpr int kThreads = 128;

template <int D>
constexpr size_t attn_smem_bytes() {
  return (size_t)(kRowsPerCta + 2 * kStages * kTileKeys) * (D + 8) * sizeof(bf16) +
         kMaxNodes * sizeof(uint64_t) + kMaxNodes * sizeof(int);
}

// Cache row of prefix position pos of sequence b, or -1 if its block is invalid.
__device__ __forceinline__ long long cache_row(const AttnParams &p, int b, int pos) {
  if (p.block_table == nullptr) return (long long)b * p.Lmax + pos;
  const int blk = p.block_table[(size_t)b * p.max_blocks + pos / p.block_size];
  if (blk < 0 || blk >= p.num_blocks) return -1;
  return (long long)blk * p.block_size + pos % p.block_size;
}

__device__ __forceinline__ int clamp_prefix(const AttnParams &p, int b) {
  int L = p.prefix_len[b];
  if (L < 0 || L > p.cap) {
    set_status(p.status, SV_DEV_BAD_PREFIX);
    L = L < 0 ? 0 : p.cap;
  }
  return L;
}

template <int D>
__global__ void __launch_bounds__(kThreads) attn_mma_kernel(const AttnParams p) {
  constexpr int LDS = D + 8;  // padded row stride (elements): conflict-free ldmatrix
  constexpr int CH = D / 8;   // 16-byte chunks per row
  extern __shared__ __align__(16) unsigned char smem[];
  bf16 *sQ = reinterpret_cast<bf16 *>(smem);
  bf16 *sK = sQ + kRowsPerCta * LDS;
  bf16 *sV = sK + kStages * kTileKeys * LDS;
  uint64_t *sAnc = reinterpret_cast<uint64_t *>(sV + kStages * kTileKeys * LDS);
  int *sPar = reinterpret_cast<int *>(sAnc + kMaxNodes);

  const bf16 *gq = static_cast<const bf16 *>(p.q);
  const bf16 *gkt = static_cast<const bf16 *>(p.k_tree);
  const bf16 *gvt = static_cast<const bf16 *>(p.v_tree);
  const bf16 *gkc = static_cast<const bf16 *>(p.cache_k);
  const bf16 *gvc = static_cast<const bf16 *>(p.cache_v);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x % p.m_tiles, split = blockIdx.x / p.m_tiles;
  const int kvh = blockIdx.y, b = blockIdx.z;

  const int L = clamp_prefix(p, b);
  const int k_begin = split * p.chunk;
  const int k_end = min(L, k_begin + p.chunk);
  const int n_pref = k_end > k_begin ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;
  const int has_tree = split == 0 ? 1 : 0;
  const int n_tiles = n_pref + has_tree;

  // sequence b's tree (shared, or its own row): ancestor masks of its nodes
  if (tid < kMaxNodes) sPar[tid] = tid < p.tree.N ? tree_parent(p.tree, b, tid) : -1;
  __syncthreads();
  if (tid < kMaxNodes) {
    uint64_t m = 0;
    int d;
    if (tid < p.tree.N && !tree_walk(sPar, tid, &m, &d) && split == 0 && kvh == 0 && mt == 0)
      set_status(p.status, SV_DEV_BAD_TREE);
    sAnc[tid] = m;
  }

  // query rows of this tile: row R = mt*64 + r -> node R / G, head kvh*G + R % G
  for (int c = tid; c < kRowsPerCta * CH; c += kThreads) {
    const int r = c / CH, col = c % CH, R = mt * kRowsPerCta + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (R < p.M) {
      const int n = R / p.G, hq = kvh * p.G + R % p.G;
      v = *reinterpret_cast<const uint4 *>(gq + (((size_t)b * p.N + n) * p.Hq + hq) * D + col * 8);
    }
    *reinterpret_cast<uint4 *>(sQ + r * LDS + col * 8) = v;
  }

  auto load_tile = [&](int t, int stage) {
    const bool tree = has_tree && t == 0;
    const int base = k_begin + (t - has_tree) * kTileKeys;
    bf16 *dk = sK + stage * kTileKeys * LDS;
    bf16 *dv = sV + stage * kTileKeys * LDS;
    for (int c = tid; c < kTileKeys * CH; c += kThreads) {
      const int r = c / CH, col = c % CH;
      bool valid;
      const bf16 *sk, *sv;
      if (tree) {
        valid = r < p.N;
        const size_t off = (((size_t)b * p.N + (valid ? r : 0)) * p.Hkv + kvh) * D + col * 8;
        sk = gkt + off;
        sv = gvt + off;
      } else {
        const int pos = base + r;
        valid = pos < k_end;
        long long row = 0;
        if (valid) {
          row = cache_row(p, b, pos);
          if (row < 0) {
            if (col == 0) set_status(p.status, SV_DEV_BAD_BLOCK);
            valid = false;
            row = 0;
          }
        }
        const size_t off = ((size_t)row * p.Hkv + kvh) * D + col * 8;
        sk = gkc + off;
        sv = gvc + off;
      }
      cp_async_16(dk + r * LDS + col * 8, sk, valid);
      cp_async_16(dv + r * LDS + col * 8, sv, valid);
    }
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_tiles) load_tile(s, s);
    cp_async_commit();
  }
  __syncthreads();  // sQ, sAnc ready

  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    ldmatrix_x4(qf[ks], sQ + (warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LDS + ks * 16 +
                            (lane >> 4) * 8);

  // the two query rows this thread accumulates (fragment rows g and g+8)
  const int r_lo = warp * 16 + (lane >> 2);
  uint64_t anc[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int R = mt * kRowsPerCta + r_lo + 8 * i;
    anc[i] = R < p.M ? sAnc[R / p.G] : 0ull;
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int tn = t + kStages - 1;
      if (tn < n_tiles) load_tile(tn, tn % kStages);
      cp_async_commit();
    }
    const int stage = t % kStages;
    const bf16 *tk = sK + stage * kTileKeys * LDS;
    const bf16 *tv = sV + stage * kTileKeys * LDS;
    const bool tree = has_tree && t == 0;
    const int base = k_begin + (t - has_tree) * kTileKeys;

    float sc[kTileKeys / 8][4];
#pragma unroll
    for (int i = 0; i < kTileKeys / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < kTileKeys / 16; ++np) {
        uint32_t kf[4];
        ldmatrix_x4(kf, tk + (np * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + ks * 16 +
                            ((lane >> 3) & 1) * 8);
        mma_bf16_16816(sc[2 * np], qf[ks], kf[0], kf[1]);
        mma_bf16_16816(sc[2 * np + 1], qf[ks], kf[2], kf[3]);
      }
    }

    // mask, scale to log2 units, online softmax per row
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kTileKeys / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = nt * 8 + 2 * (lane & 3) + e;
          const bool ok = tree ? ((anc[i] >> kk) & 1ull) != 0 : (base + kk < k_end);
          const float x = ok ? sc[nt][2 * i + e] * p.scale_log2 : -INFINITY;
          sc[nt][2 * i + e] = x;
          mx = fmaxf(mx, x);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run[i], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_run[i] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int nt = 0; nt < kTileKeys / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pe = exp2f(sc[nt][2 * i + e] - m_use);
          sc[nt][2 * i + e] = pe;
          rs += pe;
        }
      }
      l_run[i] = l_run[i] * alpha + rs;
      m_run[i] = m_new;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        o[dt][2 * i] *= alpha;
        o[dt][2 * i + 1] *= alpha;
      }
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < kTileKeys / 16; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
      a[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
      a[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      a[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t vf[4];
        ldmatrix_x4_trans(vf, tv + (kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LDS +
                                  dp * 16 + (lane >> 4) * 8);
        mma_bf16_16816(o[2 * dp], a, vf[0], vf[1]);
        mma_bf16_16816(o[2 * dp + 1], a, vf[2], vf[3]);
      }
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xFFFFFFFFu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xFFFFFFFFu, l_run[i], 2);
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int R = mt * kRowsPerCta + r_lo + 8 * i;
    if (p.splits == 1) {
      if (R >= p.M) continue;
      const int n = R / p.G, hq = kvh * p.G + R % p.G;
      bf16 *dst = static_cast<bf16 *>(p.out) + (((size_t)b * p.N + n) * p.Hq + hq) * D;
      const float inv = l_run[i] > 0.f ? 1.f / l_run[i] : 0.f;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        const int col = dt * 8 + 2 * (lane & 3);
        *reinterpret_cast<uint32_t *>(dst + col) = pack_bf16x2(o[dt][2 * i] * inv, o[dt][2 * i + 1] * inv);
      }
    } else {
      const size_t row = (((size_t)b * p.Hkv + kvh) * p.splits + split) * p.Mpad + R;
      float *dst = p.part_o + row * D;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        const int col = dt * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2 *>(dst + col) = make_float2(o[dt][2 * i], o[dt][2 * i + 1]);
      }
      if ((lane & 3) == 0) {
        p.part_ml[row * 2] = m_run[i];
        p.part_ml[row * 2 + 1] = l_run[i];
      }
    }
  }
}

// Merge the prefix splits of one query row: weights 2^(m_s - max m) (log2 units).
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const AttnParams p) {
  const int R = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const size_t row0 = (((size_t)b * p.Hkv + kvh) * p.splits) * p.Mpad + R;
  float mx = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, p.part_ml[(row0 + (size_t)s * p.Mpad) * 2]);
  float acc = 0.f, den = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const size_t row = row0 + (size_t)s * p.Mpad;
    const float m = p.part_ml[row * 2];
    if (m == -INFINITY) continue;
    const float w = exp2f(m - mx);
    den += w * p.part_ml[row * 2 + 1];
    acc += w * p.part_o[row * D + d];
  }
  const int n = R / p.G, hq = kvh * p.G + R % p.G;
  bf16 *dst = static_cast<bf16 *>(p.out) + (((size_t)b * p.N + n) * p.Hq + hq) * D;
  dst[d] = __float2bfloat16(den > 0.f ? acc / den : 0.f);
}

// fp32 path (FFMA, no tensor cores): one warp per query row (node, query head), the
// kThreads / 32 rows of a CTA sharing one kv head.  The keys go in chunks of 32 -- the
// prefix, then the tree nodes -- copied by the whole CTA with cp.async into a ring of
// f32_stages() shared-memory stages, so that that many chunks are in flight at once (a short
// prefix arrives in one round trip).  Lane j scores key j of the chunk (rows of K padded to
// D + 4 floats: conflict-free 16-byte reads); online softmax in fp32 per row: chunk maximum
// and sum by warp reductions, then P V with lane i holding dimensions i, i + 32, ... and
// each key's weight broadcast by a shuffle.
constexpr int kF32Keys = 32;  // keys per chunk: one per lane
// stages of the ring: 8 (132 KB) at D = 64, 6 (198 KB) at D = 128
template <int D>
__host__ __device__ constexpr int f32_stages() { return D == 64 ? 8 : 6; }

template <int D>
__host__ __device__ constexpr size_t f32_stage_floats() { return (size_t)kF32Keys * (D + 4) + (size_t)kF32Keys * D; }

template <int D>
__global__ void __launch_bounds__(kThreads) attn_f32_kernel(const AttnParams p) {
  constexpr int KC = kF32Keys, ST = f32_stages<D>();
  constexpr int KS = D + 4;                 // K row stride in shared memory (floats)
  constexpr int PL = D / 32;                // dimensions per lane in P V
  constexpr int NW = kThreads / 32;         // rows per CTA
  constexpr int F4 = KC * D / 4;            // float4 per chunk of K (and of V)
  constexpr int PER = F4 / kThreads;        // float4 of K (and of V) per thread per chunk
  static_assert(F4 % kThreads == 0, "whole float4 per thread");
  extern __shared__ __align__(16) float f32_ring[];  // ST x { K [KC][KS], V [KC][D] }
  __shared__ __align__(16) float sQ[NW][D];
  __shared__ uint8_t sValid[ST][KC];        // key j of a stage exists (block id checked)
  __shared__ int sPar[kMaxNodes];
  __shared__ uint64_t sAnc[kMaxNodes];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, b = blockIdx.z;
  // sequence b's tree (shared, or its own row): ancestor masks of its nodes
  if (tid < kMaxNodes) sPar[tid] = tid < p.tree.N ? tree_parent(p.tree, b, tid) : -1;
  __syncthreads();
  if (tid < kMaxNodes) {
    uint64_t m = 0;
    int d;
    if (tid < p.tree.N && !tree_walk(sPar, tid, &m, &d) && blockIdx.x == 0 && kvh == 0)
      set_status(p.status, SV_DEV_BAD_TREE);
    sAnc[tid] = m;
  }
  const float *gq = static_cast<const float *>(p.q);
  const float *gkt = static_cast<const float *>(p.k_tree);
  const float *gvt = static_cast<const float *>(p.v_tree);
  const float *gkc = static_cast<const float *>(p.cache_k);
  const float *gvc = static_cast<const float *>(p.cache_v);
  const int L = clamp_prefix(p, b);
  // this warp's row: query rows of the kv head are (node, group head), node-major
  const int R = blockIdx.x * NW + warp;
  const bool live = R < p.M;
  const int n = live ? R / p.G : 0, hq = kvh * p.G + (live ? R % p.G : 0);

  // chunk c: prefix positions [32c, 32c + 32) for c < nP, then tree nodes from 32 (c - nP)
  const int nP = (L + KC - 1) / KC, nT = (p.N + KC - 1) / KC, nC = nP + nT;
  auto stage_k = [&](int st) { return f32_ring + (size_t)st * f32_stage_floats<D>(); };
  auto stage_v = [&](int st) { return f32_ring + (size_t)st * f32_stage_floats<D>() + KC * KS; };
  auto issue = [&](int c, int st) {
    float *sk = stage_k(st), *sv = stage_v(st);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int f = tid + k * kThreads, key = f / (D / 4), d4 = f % (D / 4);
      const float *srck = gkc, *srcv = gvc;  // any valid address when nothing is read
      bool ok = false;
      if (c < nP) {
        const int pos = c * KC + key;
        if (pos < L) {
          const long long row = cache_row(p, b, pos);
          if (row >= 0) {
            const size_t off = ((size_t)row * p.Hkv + kvh) * D + 4 * d4;
            srck = gkc + off;
            srcv = gvc + off;
            ok = true;
          } else if (d4 == 0) {
            set_status(p.status, SV_DEV_BAD_BLOCK);
          }
        }
      } else {
        const int j = (c - nP) * KC + key;
        if (j < p.N) {
          const size_t off = (((size_t)b * p.N + j) * p.Hkv + kvh) * D + 4 * d4;
          srck = gkt + off;
          srcv = gvt + off;
          ok = true;
        }
      }
      cp_async_16(sk + key * KS + 4 * d4, srck, ok);
      cp_async_16(sv + key * D + 4 * d4, srcv, ok);
      if (d4 == 0) sValid[st][key] = ok ? 1 : 0;
    }
  };
  // the first ST chunks in flight together; one commit group per chunk (empty past the end)
#pragma unroll 1
  for (int st = 0; st < ST; ++st) {
    if (st < nC) issue(st, st);
    cp_async_commit();
  }
  // the row's q while the chunks are in flight
  for (int i = lane; i < D; i += 32)
    sQ[warp][i] = live ? gq[(((size_t)b * p.N + n) * p.Hq + hq) * D + i] : 0.f;
  __syncthreads();  // sQ, sAnc
  const uint64_t anc = sAnc[n];
  float m = -INFINITY, l = 0.f, o[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) o[i] = 0.f;
#pragma unroll 1
  for (int c = 0; c < nC; ++c) {
    const int st = c % ST;
    cp_async_wait<ST - 1>();  // chunk c's group has landed (later ones may still be in flight)
    __syncthreads();
    if (live) {
      const float *sk = stage_k(st), *sv = stage_v(st);
      // lane j scores key j of the chunk
      const bool tree_chunk = c >= nP;
      const int j = tree_chunk ? (c - nP) * KC + lane : c * KC + lane;
      bool vis = sValid[st][lane] != 0;
      if (tree_chunk) vis = vis && ((anc >> j) & 1ull);
      const float4 *kr = reinterpret_cast<const float4 *>(sk + lane * KS);
      const float4 *qr = reinterpret_cast<const float4 *>(sQ[warp]);
      float dot = 0.f;
#pragma unroll 8
      for (int d4 = 0; d4 < D / 4; ++d4) {
        const float4 kv = kr[d4], qv = qr[d4];
        dot = fmaf(qv.x, kv.x, dot);
        dot = fmaf(qv.y, kv.y, dot);
        dot = fmaf(qv.z, kv.z, dot);
        dot = fmaf(qv.w, kv.w, dot);
      }
      const float sc = vis ? dot * p.scale : -INFINITY;
      float cm = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, off));
      const float m_new = fmaxf(m, cm);
      if (m_new != -INFINITY) {
        const float alpha = m == -INFINITY ? 0.f : expf(m - m_new);
        const float pe = vis ? expf(sc - m_new) : 0.f;
        float ps = pe;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, off);
        l = l * alpha + ps;
#pragma unroll
        for (int i = 0; i < PL; ++i) o[i] *= alpha;
#pragma unroll 8
        for (int jj = 0; jj < KC; ++jj) {
          const float w = __shfl_sync(0xFFFFFFFFu, pe, jj);
#pragma unroll
          for (int i = 0; i < PL; ++i) o[i] = fmaf(w, sv[jj * D + lane + 32 * i], o[i]);
        }
        m = m_new;
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
    if (c + ST < nC) issue(c + ST, st);
    cp_async_commit();
  }
  cp_async_wait<0>();
  if (!live) return;
  float *dst = static_cast<float *>(p.out) + (((size_t)b * p.N + n) * p.Hq + hq) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) dst[lane + 32 * i] = o[i] * inv;
}

template <int D>
cudaError_t launch_f32(const AttnParams &p, cudaStream_t s) {
  const size_t smem = (size_t)f32_stages<D>() * f32_stage_floats<D>() * sizeof(float);
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev].load()) {
    const cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true);
  }
  dim3 grid((p.M + kThreads / 32 - 1) / (kThreads / 32), p.Hkv, p.B);
  attn_f32_kernel<D><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_mma(const AttnParams &p, cudaStream_t s) {
  const size_t smem = attn_smem_bytes<D>();
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true);
  }
  dim3 grid(p.m_tiles * p.splits, p.Hkv, p.B);
  attn_mma_kernel<D><<<grid, kThreads, smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  attn_combine_kernel<D><<<dim3(p.M, p.Hkv, p.B), D, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

AttnPlan attn_plan(sv_dtype dt, int B, int N, int Hq, int Hkv, int D, int max_prefix,
                   int num_sms) {
  AttnPlan pl{};
  const int G = Hq / Hkv;
  const int M = N * G;
  pl.m_tiles = (M + kRowsPerCta - 1) / kRowsPerCta;
  pl.Mpad = pl.m_tiles * kRowsPerCta;
  pl.splits = 1;
  pl.chunk = max_prefix > 0 ? max_prefix : kTileKeys;
  if (dt == SV_BF16 && max_prefix > 0) {
    const long long base = (long long)B * Hkv * pl.m_tiles;
    const long long want = 2LL * (num_sms > 0 ? num_sms : 152);
    long long splits = (want + base - 1) / base;
    const long long max_splits = (max_prefix + 511) / 512;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int chunk = (int)((max_prefix + splits - 1) / splits);
    chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
    pl.chunk = chunk;
    pl.splits = (max_prefix + chunk - 1) / chunk;
  }
  pl.ws_bytes = pl.splits > 1
                    ? (size_t)B * Hkv * pl.splits * pl.Mpad * (size_t)(D + 2) * sizeof(float)
                    : 0;
  return pl;
}

cudaError_t launch_attention(sv_dtype dt, const AttnParams &p, cudaStream_t s) {
  if (dt == SV_F32) return p.D == 64 ? launch_f32<64>(p, s) : launch_f32<128>(p, s);
  return p.D == 64 ? launch_mma<64>(p, s) : launch_mma<128>(p, s);
}

}  // namespace sv
