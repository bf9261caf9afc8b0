// Device helpers shared by the verify-step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sv.h"
#include "sv_internal.h"

namespace sv {

typedef __nv_bfloat16 bf16;

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void set_status(unsigned int *status, unsigned int bits) {
  if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------------ trees

// Parent of node c (< N) of sequence b: the shared tree's, or the sequence's own row.
__device__ __forceinline__ int tree_parent(const Tree &t, int b, int c) {
  return t.rows ? __ldg(t.rows + (size_t)b * t.stride + c) : (int)t.parent[c];
}

// Walk from node c to the root over a parent array par[] (BFS order): the ancestor mask
// (bit j set iff j is c or one of its ancestors) and the depth.  False when the chain is
// not that of a BFS-ordered tree (a parent outside [0, i), or par[0] != -1): the walk stops
// there, with the bits and depth gathered so far.  Per-sequence trees come from device
// memory unchecked, so every kernel walks them this way; a shared tree was checked on the
// host and always walks to the root.
template <typename P>
__device__ __forceinline__ bool tree_walk(const P *par, int c, uint64_t *anc, int *depth) {
  uint64_t m = 0;
  int d = 0, a = c;
  for (int s = 0; s < kMaxNodes; ++s) {
    m |= 1ull << a;
    if (a == 0) {
      *anc = m;
      *depth = d;
      return (int)par[0] == -1;
    }
    const int pa = (int)par[a];
    if (pa < 0 || pa >= a) break;
    a = pa;
    ++d;
  }
  *anc = m;
  *depth = d;
  return false;
}

// The same walk reading sequence b's parents straight from the tree descriptor.
__device__ __forceinline__ bool tree_walk_seq(const Tree &t, int b, int c, uint64_t *anc,
                                              int *depth) {
  uint64_t m = 0;
  int d = 0, a = c;
  for (int s = 0; s < kMaxNodes; ++s) {
    m |= 1ull << a;
    if (a == 0) {
      *anc = m;
      *depth = d;
      return tree_parent(t, b, 0) == -1;
    }
    const int pa = tree_parent(t, b, a);
    if (pa < 0 || pa >= a) break;
    a = pa;
    ++d;
  }
  *anc = m;
  *depth = d;
  return false;
}

// ------------------------------------------------------------ element access

// Widen 8 packed bf16 (one 16-byte vector) to float; element i at bits [16i, 16i+16).
__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename T>
struct Elem;

template <>
struct Elem<bf16> {
  static constexpr int kVec = 8;  // elements per 16-byte vector
  __device__ static __forceinline__ void unpack(const uint4 &v, float f[8]) { unpack_bf16x8(v, f); }
  __device__ static __forceinline__ float load(const bf16 *p) { return __bfloat162float(*p); }
  // Order-preserving integer key: a larger key is a larger value.
  __device__ static __forceinline__ uint32_t key(float f) {
    uint32_t h = __float_as_uint(f) >> 16;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  }
  static constexpr int kKeyBits = 16;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;  // two bf16 -inf
};

template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ static __forceinline__ void unpack(const uint4 &v, float f[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ float load(const float *p) { return *p; }
  __device__ static __forceinline__ uint32_t key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  static constexpr int kKeyBits = 32;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
};

// 2^x by the hardware's approximate exponential (one MUFU op, subnormal results
// flushed to zero); relative error about 2^-22.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of f32 (one instruction for both lanes; each lane rounds as the scalar
// instruction would).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " sub.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Lane-wise maximum of two pairs of bf16 (a NaN lane yields the other operand).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------ Philox

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32->64
// multiplies by the Philox multipliers, mixing with the other two words and the key;
// the key advances by the two Weyl increments after every round.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t a = c[0], b = c[2];
    const uint32_t hi0 = __umulhi(0xD2511F53u, a), lo0 = 0xD2511F53u * a;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, b), lo1 = 0xCD9E8D57u * b;
    const uint32_t n0 = hi1 ^ c[1] ^ k0;
    const uint32_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// Uniforms of (sequence b, node c): u_acc from word 0, u_smp from word 1, each
// ((w >> 8) + 0.5) * 2^-24, exact in double.
__device__ __forceinline__ void verify_uniforms(uint64_t seed, uint64_t round, int b, int c,
                                                double *u_acc, double *u_smp) {
  uint32_t ctr[4] = {(uint32_t)c, (uint32_t)b, (uint32_t)round, (uint32_t)(round >> 32)};
  philox4x32_10(ctr, (uint32_t)seed, (uint32_t)(seed >> 32));
  *u_acc = ((double)(ctr[0] >> 8) + 0.5) * (1.0 / 16777216.0);
  *u_smp = ((double)(ctr[1] >> 8) + 0.5) * (1.0 / 16777216.0);
}

// The same uniforms as their 24-bit integers k: u = (k + 0.5) * 2^-24.
__device__ __forceinline__ void verify_uniform_ints(uint64_t seed, uint64_t round, int b, int c,
                                                    uint32_t *k_acc, uint32_t *k_smp) {
  uint32_t ctr[4] = {(uint32_t)c, (uint32_t)b, (uint32_t)round, (uint32_t)(round >> 32)};
  philox4x32_10(ctr, (uint32_t)seed, (uint32_t)(seed >> 32));
  *k_acc = ctr[0] >> 8;
  *k_smp = ctr[1] >> 8;
}

// --------------------------------------------------------- warp reductions

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Kahan-compensated accumulation.
struct KahanF {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ float value() const { return s - c; }
};

// ------------------------------------------------------ async copies, MMA

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte cp.async; when !valid nothing is read and the destination is zero-filled.
__device__ __forceinline__ void cp_async_16(void *smem, const void *gmem, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(n));
}
// 8-byte cp.async (cached in L1).
__device__ __forceinline__ void cp_async_8(void *smem, const void *gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
// Arrive on an mbarrier once all of this thread's earlier cp.async copies have landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t r[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace sv
