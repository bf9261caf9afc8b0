// KV commit of the accepted path (sm_103a).
//
// qwbw.cn sections 3.1.4 and 6.3, hncyxsy.com section 4.3: after verification only the
// KV of the root and the accepted candidates is kept; rejected candidates are dropped
// by not advancing the valid length over them.  One CTA per sequence copies the tree
// K/V rows of the path nodes (root first, depth order) to positions
// prefix_len[b] + i with 16-byte vectors, then advances prefix_len[b].
#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const CommitParams p) {
  const int b = blockIdx.x;
  __shared__ int s_L, s_n;
  if (threadIdx.x == 0) {
    s_L = p.prefix_len[b];
    s_n = p.num_accepted[b];
  }
  __syncthreads();
  const int L = s_L, n_acc = s_n;
  const size_t row_vec = (size_t)p.Hkv * p.D * p.esize / 16;  // 16-byte vectors per row
  const uint4 *kt = static_cast<const uint4 *>(p.k_tree);
  const uint4 *vt = static_cast<const uint4 *>(p.v_tree);
  uint4 *ck = static_cast<uint4 *>(p.cache_k);
  uint4 *cv = static_cast<uint4 *>(p.cache_v);
  const int count = n_acc + 1;
  const bool ok_n = n_acc >= 0 && n_acc < p.path_stride && L >= 0;
  if (ok_n) {
    for (size_t i = threadIdx.x; i < (size_t)count * row_vec; i += kCommitThreads) {
      const int k = (int)(i / row_vec);
      const size_t e = i % row_vec;
      const int node = p.path_nodes[(size_t)b * p.path_stride + k];
      if (node < 0 || node >= p.N) {
        set_status(p.status, SV_DEV_BAD_TOKEN);
        continue;
      }
      const int pos = L + k;
      long long dst_row;
      if (p.block_table) {
        const int bi = pos / p.block_size;
        const int blk = bi < p.max_blocks ? p.block_table[(size_t)b * p.max_blocks + bi] : -1;
        if (blk < 0 || blk >= p.num_blocks) {
          if (e == 0) set_status(p.status, SV_DEV_BAD_BLOCK);
          continue;
        }
        dst_row = (long long)blk * p.block_size + pos % p.block_size;
      } else {
        if (pos >= p.Lmax) {
          if (e == 0) set_status(p.status, SV_DEV_BAD_PREFIX);
          continue;
        }
        dst_row = (long long)b * p.Lmax + pos;
      }
      const size_t src = ((size_t)b * p.N + node) * row_vec + e;
      const size_t dst = (size_t)dst_row * row_vec + e;
      ck[dst] = kt[src];
      cv[dst] = vt[src];
    }
  } else if (threadIdx.x == 0) {
    set_status(p.status, SV_DEV_BAD_PREFIX);
  }
  __syncthreads();
  if (threadIdx.x == 0 && ok_n) p.prefix_len[b] = L + count;
}

}  // namespace

cudaError_t launch_commit(const CommitParams &p, cudaStream_t s) {
  commit_kernel<<<p.B, kCommitThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sv
