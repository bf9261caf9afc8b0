// The LM-head projection on the 5th-generation tensor cores, with the acceptance's row
// statistics in its epilogue (sm_103a).
//
// What it computes ("推测解码技术详解", section "Medusa Heads": the original LM head and
// the Medusa heads read the backbone's last hidden states; lpnh.cn walkthrough, section
// 3.1: a head is a Linear(H, V) from h_t to V logits): z[r, v] = sum_k h[r, k] w[v, k],
// h [R, Dm] and w [V, Dm] bf16 (both K-major), fp32 accumulation, z stored in bf16.  The
// epilogue also takes, per (row, 256-column tile), the tile's maximum, its lowest argmax
// and the Kahan sum of 2^((z - max) c) over the stored (bf16-rounded) logits, c =
// log2(e) / T; a merge kernel turns them into the row's statistics (max, argmax, softmax
// sum) -- what the acceptance's statistics kernel would compute by reading the logits
// back.  The stored logits remain the input of the final sample (the chosen row is known
// only after every row's normaliser), so they are still written.
//
// One persistent CTA per SM, 192 threads: warp 0 issues the TMA loads of H and W tiles
// into a 4-stage ring, warp 1 owns TMEM and one of its threads issues the MMAs
// (128 x 256 x 16 each, accumulating in TMEM), warps 2..5 run the epilogue (warp w
// reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, one output row per thread).  Two TMEM
// accumulators of 256 columns let the epilogue of one tile overlap the MMAs of the next.
// Tiles are numbered rows-fastest, so the CTAs that read the same W tile run at the same
// time and W comes from HBM about once.  Every wait is bounded (SV_DEV_TIMEOUT).
#include <atomic>
#include <cudaTypedefs.h>

#include <cfloat>
#include <climits>

#include "sv_common.cuh"
#include "sv_internal.h"
#include "tc_primitives.cuh"

namespace sv {

namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB: 128 rows of 64 bf16 (128-byte swizzle)
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kBarBytes = 256;
constexpr int kSmem = kStages * kStageBytes + kBarBytes;

__device__ __forceinline__ bool better_idx(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kThreads, 1) lm_head_kernel(const __grid_constant__ LmHeadParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *empty = full + kStages;
  uint64_t *acc_full = empty + kStages;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0u) {  // swizzled stages need a 1024-aligned window
    if (threadIdx.x == 0) set_status(p.status, SV_DEV_LAYOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&p.tm_h);
    prefetch_tmap(&p.tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int T = p.mtiles * p.ntiles, KB = (p.Dm + kBK - 1) / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
        const int m = t % p.mtiles, n = t / p.mtiles;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int s = (int)(g % kStages);
          if (g >= kStages && !mbar_wait(&empty[s], (uint32_t)(((g / kStages) - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *a = smem + s * kStageBytes;
          mbar_expect_tx(&full[s], kStageBytes);
          tma_load_3d(a, &p.tm_h, kb * kBK, 0, m * kBM, &full[s]);
          tma_load_3d(a + kABytes, &p.tm_w, kb * kBK, 0, n * kBN, &full[s]);
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA retires
        const unsigned long long t0 = global_ns();
        for (long long i = g - kStages < 0 ? 0 : g - kStages; i < g; ++i)
          while (!mbar_try_wait(&full[i % kStages], (uint32_t)((i / kStages) & 1)) &&
                 global_ns() - t0 < kWaitLimitNs) {
          }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN, 0, 0);
      long long g = 0;
      int i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += gridDim.x, ++i) {
        const int acc = i & 1;
        if (i >= 2 && !mbar_wait(&acc_empty[acc], (uint32_t)(((i >> 1) - 1) & 1), abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int s = (int)(g % kStages);
          if (!mbar_wait(&full[s], (uint32_t)((g / kStages) & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * kStageBytes), b0 = a0 + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t a = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(b0 + kk * 32, 16, 1024);
            umma_bf16(tmem + (uint32_t)(acc * kBN), a, b, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (ok) umma_commit(&acc_full[acc]);
      }
      // every MMA issued must complete before TMEM is released
      umma_commit(drain);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const float c = p.c_log2;
    int i = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
      const int acc = i & 1, m = t % p.mtiles, n = t / p.mtiles;
      if (!mbar_wait(&acc_full[acc], (uint32_t)((i >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      const int row = m * kBM + q * 32 + lane;
      const bool live = row < p.R;
      bf16 *zrow = static_cast<bf16 *>(p.z) + (size_t)(live ? row : 0) * p.V;
      float zm = -INFINITY;  // running maximum of the tile's stored logits
      int am = INT_MAX;
      KahanF ks;             // sum of 2^((z - zm) c), rescaled when zm grows
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN + c0), v);
        tmem_wait_ld();
        const int j0 = n * kBN + c0;
        const int nval = min(32, p.V - j0);  // columns of this chunk inside the vocabulary
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[k], v[k + 1]);
          pk[k / 2] = *reinterpret_cast<const uint32_t *>(&h2);
          v[k] = __low2float(h2);  // the stored logits from here on
          v[k + 1] = __high2float(h2);
        }
        if (!live || nval <= 0) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(zrow + j0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (8 * k < nval) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        float cm = -INFINITY;
        int ci = INT_MAX;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k < nval && v[k] > cm) cm = v[k], ci = j0 + k;  // lowest index among equals
        if (better_idx(cm, ci, zm, am)) {
          if (cm > zm && zm != -INFINITY && c > 0.f) {
            const float sc = ex2_approx((zm - cm) * c);
            ks.s *= sc;
            ks.c *= sc;
          }
          if (cm > zm) zm = cm;
          am = ci;
        }
        if (c > 0.f) {
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nval) s4[k & 3] += ex2_approx((v[k] - zm) * c);
          ks.add((s4[0] + s4[1]) + (s4[2] + s4[3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (live && p.part)
        p.part[(size_t)row * p.ntiles + n] = make_float4(zm, ks.value(), __int_as_float(am), 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, SV_DEV_TIMEOUT);
}

// One warp per row: the row's maximum and its lowest argmax over the tiles, and
// S = sum_t s_t 2^((m_t - zmax) c) (m_t, s_t: a tile's maximum and sum), each term in
// float (as the statistics kernel forms its terms) and the sum in double.
__global__ void lm_head_merge_kernel(const float4 *part, int R, int ntiles, float c_log2,
                                     RowStat *stats) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= R) return;
  const float4 *pr = part + (size_t)row * ntiles;
  float m = -INFINITY;
  int a = INT_MAX;
  for (int t = lane; t < ntiles; t += 32) {
    const float4 e = __ldcg(pr + t);
    const int ea = __float_as_int(e.z);
    if (better_idx(e.x, ea, m, a)) m = e.x, a = ea;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const int oa = __shfl_xor_sync(0xFFFFFFFFu, a, o);
    if (better_idx(om, oa, m, a)) m = om, a = oa;
  }
  double S = 0.0;
  if (c_log2 > 0.f) {
    for (int t = lane; t < ntiles; t += 32) {
      const float4 e = __ldcg(pr + t);
      if (e.x != -INFINITY) S += (double)(e.y * ex2_approx((e.x - m) * c_log2));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
  }
  if (lane == 0) {
    RowStat st;
    st.zmax = m;
    st.argmax = a;
    st.key_k = 0u;       // no top-k: every entry is kept
    st.idx_k = INT_MAX;
    st.S = (float)S;
    st.flags = 0u;
    st.H = 0.f;
    st.pad = 0u;
    stats[row] = st;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
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

// A row-major bf16 matrix [rows, cols] as a (cols, 1, rows) view with a (64, 1, box_rows)
// box, 128-byte swizzle: one box is box_rows rows of 64 columns, the K-major operand layout.
bool kmajor_map(CUtensorMap *m, const void *base, int cols, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, 1, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2};
  cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t lm_head_part_bytes(int R, int V) {
  const int ntiles = (V + kBN - 1) / kBN;
  return (size_t)R * (size_t)ntiles * sizeof(float4);
}

cudaError_t launch_lm_head(const void *hidden, const void *weight, int R, int Dm, int V,
                           float c_log2, void *z, void *part, RowStat *stats, unsigned int *status,
                           int num_sms, cudaStream_t s) {
  LmHeadParams p{};
  if (!kmajor_map(&p.tm_h, hidden, Dm, R, kBM) || !kmajor_map(&p.tm_w, weight, Dm, V, kBN))
    return cudaErrorInvalidValue;
  p.z = z;
  p.part = static_cast<float4 *>(part);
  p.status = status;
  p.R = R;
  p.V = V;
  p.Dm = Dm;
  p.mtiles = (R + kBM - 1) / kBM;
  p.ntiles = (V + kBN - 1) / kBN;
  p.c_log2 = c_log2;
  static std::atomic<bool> attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr[dev].load()) {
    const cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr[dev].store(true);
  }
  const int tiles = p.mtiles * p.ntiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  lm_head_kernel<<<grid, kThreads, kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || stats == nullptr) return e;
  constexpr int kRowsPerCta = 2;  // many small CTAs: the rows are few and short
  lm_head_merge_kernel<<<(R + kRowsPerCta - 1) / kRowsPerCta, 32 * kRowsPerCta, 0, s>>>(
      p.part, R, p.ntiles, c_log2, stats);
  return cudaGetLastError();
}

}  // namespace sv
