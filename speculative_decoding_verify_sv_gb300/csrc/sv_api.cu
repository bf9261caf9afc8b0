// C ABI of the verify step: argument validation, planning and launches.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "sv_common.cuh"
#include "sv_internal.h"

#define SV_VERSION_STRING "sv 0.1.0 (sm_103a)"

// Sticky device status word (SV_DEV_* bits); kernels get its address as a parameter.
__device__ unsigned int g_sv_status;

namespace sv {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace sv

namespace {

thread_local std::string g_last_error;

sv_status fail(sv_status code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

sv_status cuda_fail(cudaError_t e, const char *what) {
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

// The tensor-core attention kernel's limit on a wait for progress (sv_set_wait_limit_ns).
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

// Launch failures injected on the host (sv_inject_launch_failures): the next n launch
// requests report cudaErrorLaunchFailure instead of launching.
std::atomic<int> g_injected_failures{0};
bool take_injected_failure() {
  int n = g_injected_failures.load(std::memory_order_relaxed);
  while (n > 0)
    if (g_injected_failures.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
  return false;
}

// An NVTX range named after the entry point for the duration of the host call, so that a
// profiler's timeline (and ncu's --nvtx filters) show which call enqueued which kernels.
// Without a profiler attached a push or a pop costs a few nanoseconds.
struct CallRange {
  explicit CallRange(const char *name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange &) = delete;
  CallRange &operator=(const CallRange &) = delete;
};

// Device address of the status word on the current device (looked up once per device;
// threads that race on the first lookup store the same address, atomically).
unsigned int *status_word() {
  static std::atomic<unsigned int *> addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int *a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sv_status) != cudaSuccess) return nullptr;
    a = static_cast<unsigned int *>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

int num_sms() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;
  }
  if (!sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    sms[dev] = n;
  }
  return sms[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validate a BFS-ordered parent array and fill the tree descriptor.
sv_status make_tree(int N, const int32_t *parent, sv::Tree *t) {
  if (parent == nullptr) return fail(SV_ERR_INVALID_ARG, "parent is NULL");
  if (N < 1 || N > SV_MAX_TREE_NODES)
    return fail(N < 1 ? SV_ERR_INVALID_ARG : SV_ERR_UNSUPPORTED,
                "tree has %d nodes (supported 1..%d)", N, SV_MAX_TREE_NODES);
  if (parent[0] != -1) return fail(SV_ERR_INVALID_ARG, "parent[0] must be -1 (the root)");
  memset(t, 0, sizeof *t);
  t->N = N;
  t->parent[0] = -1;
  for (int i = 1; i < N; ++i) {
    if (parent[i] < 0 || parent[i] >= i)
      return fail(SV_ERR_INVALID_ARG, "parent[%d] = %d is not in [0, %d)", i, parent[i], i);
    t->parent[i] = (int8_t)parent[i];
    t->depth[i] = (int8_t)(t->depth[parent[i]] + 1);
    t->has_child[parent[i]] = 1;
    if (t->depth[i] > t->Dmax) t->Dmax = t->depth[i];
  }
  for (int i = N; i < SV_MAX_TREE_NODES; ++i) t->parent[i] = -1;
  return SV_OK;
}

// The tree argument of the tree entry points: parent_stride == 0 -> a host array [N]
// shared by the batch (checked here); parent_stride >= N -> a device array [B,stride], one
// tree per sequence (checked by the kernels, which report SV_DEV_BAD_TREE); outputs then
// have N columns (the deepest possible path).
sv_status tree_arg(int N, const int32_t *parent, int parent_stride, sv::Tree *t) {
  if (parent_stride == 0) return make_tree(N, parent, t);
  if (parent == nullptr) return fail(SV_ERR_INVALID_ARG, "parent is NULL");
  if (N < 1 || N > SV_MAX_TREE_NODES)
    return fail(N < 1 ? SV_ERR_INVALID_ARG : SV_ERR_UNSUPPORTED,
                "tree has %d nodes (supported 1..%d)", N, SV_MAX_TREE_NODES);
  if (parent_stride < N)
    return fail(SV_ERR_INVALID_ARG, "parent_stride = %d (0 for a shared tree, >= N = %d per sequence)",
                parent_stride, N);
  if ((reinterpret_cast<uintptr_t>(parent) & 3u) != 0)
    return fail(SV_ERR_INVALID_ARG, "per-sequence parent rows must be 4-byte aligned");
  // the shared fields hold a chain (a valid tree) that no kernel reads for these calls
  int32_t chain[SV_MAX_TREE_NODES];
  for (int i = 0; i < N; ++i) chain[i] = i - 1;
  make_tree(N, chain, t);
  t->Dmax = N - 1;
  t->rows = parent;
  t->stride = parent_stride;
  return SV_OK;
}

int max_prefix_of(const sv_kv_cache &c) {
  return c.block_table ? c.max_blocks * c.block_size : c.Lmax;
}

sv_status check_cache(const sv_kv_cache &c, bool writable, int B) {
  (void)writable;
  if (B > 0 && (!c.k || !c.v || !c.prefix_len))
    return fail(SV_ERR_INVALID_ARG, "cache k, v or prefix_len is NULL");
  if (!aligned16(c.k) || !aligned16(c.v)) return fail(SV_ERR_INVALID_ARG, "cache k/v not 16-byte aligned");
  if (c.block_table) {
    if (c.block_size < 1 || c.max_blocks < 1 || c.num_blocks < 1)
      return fail(SV_ERR_INVALID_ARG, "paged cache needs block_size, max_blocks, num_blocks >= 1");
  } else if (c.Lmax < 0) {
    return fail(SV_ERR_INVALID_ARG, "Lmax < 0");
  }
  return SV_OK;
}

}  // namespace

extern "C" {

const char *sv_last_error(void) { return g_last_error.c_str(); }

const char *sv_version(void) { return SV_VERSION_STRING; }

uint64_t sv_kernel_launches(void) { return sv::g_launches.load(std::memory_order_relaxed); }

void sv_inject_launch_failures(int n) { g_injected_failures.store(n > 0 ? n : 0, std::memory_order_relaxed); }

void sv_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns, std::memory_order_relaxed);
}

uint64_t sv_get_wait_limit_ns(void) { return g_wait_limit_ns.load(std::memory_order_relaxed); }

sv_status sv_tree_prepare(int N, const int32_t *parent, uint64_t *anc, int32_t *depth) {
  sv::Tree t;
  sv_status st = make_tree(N, parent, &t);
  if (st != SV_OK) return st;
  for (int n = 0; n < N; ++n) {
    uint64_t m = 0;
    for (int a = n; a >= 0; a = t.parent[a]) m |= 1ull << a;
    if (anc) anc[n] = m;
    if (depth) depth[n] = t.depth[n];
  }
  return SV_OK;
}

sv_status sv_read_device_status(uint32_t *host_out, void *stream) {
  if (!host_out) return fail(SV_ERR_INVALID_ARG, "host_out is NULL");
  unsigned int *w = status_word();
  if (!w) return fail(SV_ERR_CUDA, "device status word unavailable");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, w, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *host_out = v;
  return SV_OK;
}

// ------------------------------------------------------------------ attention

size_t sv_tree_attention_workspace_size(sv_dtype dt, int B, int N, int Hq, int Hkv, int D,
                                        int max_prefix) {
  if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || max_prefix < 0)
    return 0;
  size_t ws = sv::attn_plan(dt, B, N, Hq, Hkv, D, max_prefix, num_sms()).ws_bytes;
  if (dt == SV_BF16 && (D == 64 || D == 128)) {
    const size_t tc = sv::tc_plan(B, N, Hq, Hkv, D, num_sms()).ws_bytes;
    if (tc > ws) ws = tc;
  }
  return ws;
}

int sv_tree_attention_path(sv_dtype dt, int N, int Hq, int Hkv, int D, int block_size) {
  if ((dt != SV_F32 && dt != SV_BF16) || N < 1 || N > SV_MAX_TREE_NODES || Hq < 1 || Hkv < 1 ||
      Hq % Hkv != 0 || (D != 64 && D != 128) || block_size < 0)
    return -1;
  return sv::tc_eligible(dt, N, Hq, Hkv, D, block_size) ? 1 : 0;
}

sv_status sv_tree_attention(sv_dtype dt, int B, int N, int Hq, int Hkv, int D, const void *q,
                            const void *k_tree, const void *v_tree, sv_kv_cache cache,
                            const int32_t *parent, int parent_stride, float scale, void *out,
                            void *workspace, size_t workspace_bytes, void *stream) {
  const CallRange range("sv_tree_attention");
  if (dt != SV_F32 && dt != SV_BF16) return fail(SV_ERR_UNSUPPORTED, "dtype %d not supported", (int)dt);
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(SV_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d", B, Hq, Hkv);
  if (D != 64 && D != 128) return fail(SV_ERR_UNSUPPORTED, "head dim %d (supported 64, 128)", D);
  sv::Tree tree;
  sv_status st = tree_arg(N, parent, parent_stride, &tree);
  if (st != SV_OK) return st;
  if (B > 0 && (!q || !k_tree || !v_tree || !out))
    return fail(SV_ERR_INVALID_ARG, "q, k_tree, v_tree or out is NULL");
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(out))
    return fail(SV_ERR_INVALID_ARG, "q, k_tree, v_tree and out must be 16-byte aligned");
  if ((st = check_cache(cache, false, B)) != SV_OK) return st;
  if (!std::isfinite(scale)) return fail(SV_ERR_INVALID_ARG, "scale is not finite");
  if (B == 0) return SV_OK;
  const int max_prefix = max_prefix_of(cache);
  const sv::AttnPlan plan = sv::attn_plan(dt, B, N, Hq, Hkv, D, max_prefix, num_sms());
  const bool use_tc = sv::tc_eligible(dt, N, Hq, Hkv, D, cache.block_table ? cache.block_size : 0);
  const sv::TcPlan tplan = use_tc ? sv::tc_plan(B, N, Hq, Hkv, D, num_sms()) : sv::TcPlan{};
  const size_t ws_need = use_tc ? tplan.ws_bytes : plan.ws_bytes;
  if (ws_need > 0) {
    if (!workspace || workspace_bytes < ws_need)
      return fail(SV_ERR_WORKSPACE, "attention workspace %zu bytes, need %zu", workspace_bytes,
                  ws_need);
    if (!aligned16(workspace)) return fail(SV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  }
  unsigned int *status = status_word();
  if (!status) return fail(SV_ERR_CUDA, "no CUDA device");

  sv::AttnParams p{};
  p.q = q;
  p.k_tree = k_tree;
  p.v_tree = v_tree;
  p.cache_k = cache.k;
  p.cache_v = cache.v;
  p.prefix_len = cache.prefix_len;
  p.block_table = cache.block_table;
  p.out = out;
  p.status = status;
  p.B = B;
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = D;
  p.Lmax = cache.Lmax;
  p.block_size = cache.block_size;
  p.max_blocks = cache.max_blocks;
  p.num_blocks = cache.num_blocks;
  p.cap = max_prefix;
  p.M = N * p.G;
  p.m_tiles = plan.m_tiles;
  p.Mpad = plan.Mpad;
  p.splits = plan.splits;
  p.chunk = plan.chunk;
  p.scale = scale;
  p.scale_log2 = scale * sv::kLog2e;
  p.tree = tree;
  p.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  cudaError_t e;
  if (use_tc) {
    e = take_injected_failure() ? cudaErrorLaunchFailure
                                  : sv::launch_attention_tc(p, tplan, workspace, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) sv::count_launches(1);
  } else {
    if (plan.ws_bytes > 0) {
      p.part_o = static_cast<float *>(workspace);
      p.part_ml = p.part_o + (size_t)B * Hkv * plan.splits * plan.Mpad * D;
    }
    e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_attention(dt, p, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) sv::count_launches(dt == SV_BF16 && plan.splits > 1 ? 2 : 1);
  }
  if (e != cudaSuccess) return cuda_fail(e, "tree attention launch");
  return SV_OK;
}

// ----------------------------------------------------------------- acceptance

size_t sv_accept_workspace_size(int B, int N, int V, int Dq) {
  (void)V;
  if (B <= 0 || N <= 0 || Dq < 0) return 0;
  return sv::accept_ws_bytes(B, N, Dq);
}

namespace {

sv_status accept_common(sv_mode mode, sv_dtype dt, int B, int V, const void *target,
                        const void *q, sv_q_kind q_kind, float temperature, int top_k,
                        float top_p, int32_t *out_tokens, int32_t *out_num_emitted,
                        int32_t *out_num_accepted, bool *greedy) {
  if (mode != SV_GREEDY && mode != SV_EXACT) return fail(SV_ERR_INVALID_ARG, "mode %d", (int)mode);
  if (dt != SV_F32 && dt != SV_BF16) return fail(SV_ERR_UNSUPPORTED, "logit dtype %d", (int)dt);
  if (B < 0) return fail(SV_ERR_INVALID_ARG, "B < 0");
  if (V < 8 || V % 8 != 0) return fail(SV_ERR_UNSUPPORTED, "V = %d must be a positive multiple of 8", V);
  if (!(temperature >= 0.f) || !std::isfinite(temperature))
    return fail(SV_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if (top_k < 0 || top_k > SV_MAX_TOP_K)
    return fail(SV_ERR_INVALID_ARG, "top_k = %d (0..%d)", top_k, SV_MAX_TOP_K);
  if (!(top_p > 0.f && top_p <= 1.f))
    return fail(SV_ERR_INVALID_ARG, "top_p must lie in (0, 1]");
  *greedy = mode == SV_GREEDY || temperature == 0.f;
  if (!*greedy && top_p < 1.f && !(top_k > 0 && top_k < V))
    return fail(SV_ERR_UNSUPPORTED, "top_p < 1 is applied within top-k: needs 0 < top_k < V");
  if (B > 0 && !target) return fail(SV_ERR_INVALID_ARG, "target_logits is NULL");
  if (!aligned16(target)) return fail(SV_ERR_INVALID_ARG, "target_logits not 16-byte aligned");
  if (!*greedy) {
    if (q_kind != SV_Q_PROBS_F32 && q_kind != SV_Q_LOGITS && q_kind != SV_Q_DRAFT_ONEHOT)
      return fail(SV_ERR_INVALID_ARG, "q_kind %d", (int)q_kind);
    if (q_kind != SV_Q_DRAFT_ONEHOT) {  // one-hot drafts have no q rows
      if (B > 0 && !q) return fail(SV_ERR_INVALID_ARG, "q is NULL in exact mode");
      if (!aligned16(q)) return fail(SV_ERR_INVALID_ARG, "q not 16-byte aligned");
    }
  }
  if (B > 0 && (!out_tokens || !out_num_emitted || !out_num_accepted))
    return fail(SV_ERR_INVALID_ARG, "an output pointer is NULL");
  return SV_OK;
}

sv_status accept_launch(sv_dtype dt, sv::AcceptParams &p, bool greedy, void *workspace,
                        size_t workspace_bytes, void *stream) {
  const size_t need = sv::accept_ws_bytes(p.B, p.N, p.Dq);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SV_ERR_WORKSPACE, "acceptance workspace %zu bytes, need %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(SV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  if (p.B == 0) return SV_OK;  // an empty batch: nothing to launch, no device needed
  p.status = status_word();
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  p.mode = greedy ? SV_GREEDY : SV_EXACT;
  p.c_log2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)p.temperature);
  if (p.top_k >= p.V) p.top_k = 0;
  if (greedy) p.top_p = 1.f;
  p.stats = static_cast<sv::RowStat *>(workspace);
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure
                                          : sv::launch_accept(dt, p, num_sms(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "acceptance launch");
  sv::count_launches(2);
  return SV_OK;
}

}  // namespace

namespace {

sv_status chain_params(sv_mode mode, sv_dtype logit_dt, int B, int gamma, int V,
                       const void *target_logits, const void *q, sv_q_kind q_kind,
                       const int32_t *draft_tokens, float temperature, int top_k, float top_p, uint64_t seed,
                       uint64_t round, int32_t *out_tokens, int32_t *out_num_emitted,
                       int32_t *out_num_accepted, uint32_t *out_near_ties, sv::AcceptParams &p,
                       bool *greedy) {
  sv_status st = accept_common(mode, logit_dt, B, V, target_logits, q, q_kind, temperature, top_k,
                               top_p, out_tokens, out_num_emitted, out_num_accepted, greedy);
  if (st != SV_OK) return st;
  if (gamma < 1 || gamma >= SV_MAX_TREE_NODES)
    return fail(SV_ERR_UNSUPPORTED, "gamma = %d (supported 1..%d)", gamma, SV_MAX_TREE_NODES - 1);
  if (B > 0 && !draft_tokens) return fail(SV_ERR_INVALID_ARG, "draft_tokens is NULL");
  int32_t parent[SV_MAX_TREE_NODES];
  for (int i = 0; i <= gamma; ++i) parent[i] = i - 1;
  p = sv::AcceptParams{};
  if ((st = make_tree(gamma + 1, parent, &p.tree)) != SV_OK) return st;
  p.B = B;
  p.N = gamma + 1;
  p.V = V;
  p.Dq = gamma;
  p.q_kind = q_kind;
  p.target = target_logits;
  p.q = q;
  p.tokens = draft_tokens;
  p.tok_stride = gamma;
  p.tok_offset = 1;
  p.chain_end = 1;  // a draft of -1 ends the sequence's chain
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.seed = seed;
  p.round = round;
  p.out_path_nodes = nullptr;
  p.out_tokens = out_tokens;
  p.out_num_emitted = out_num_emitted;
  p.out_num_accepted = out_num_accepted;
  p.out_near_ties = out_near_ties;
  return SV_OK;
}

sv_status tree_params(sv_mode mode, sv_dtype logit_dt, int B, int N, int V, const int32_t *parent,
                      int parent_stride, const int32_t *node_tokens, const void *target_logits, const void *q,
                      sv_q_kind q_kind, int Dq, float temperature, int top_k, float top_p, uint64_t seed,
                      uint64_t round, int32_t *out_path_nodes, int32_t *out_tokens,
                      int32_t *out_num_emitted, int32_t *out_num_accepted,
                      uint32_t *out_near_ties, sv::AcceptParams &p, bool *greedy) {
  sv_status st = accept_common(mode, logit_dt, B, V, target_logits, q, q_kind, temperature, top_k,
                               top_p, out_tokens, out_num_emitted, out_num_accepted, greedy);
  if (st != SV_OK) return st;
  p = sv::AcceptParams{};
  if ((st = tree_arg(N, parent, parent_stride, &p.tree)) != SV_OK) return st;
  if (B > 0 && !node_tokens) return fail(SV_ERR_INVALID_ARG, "node_tokens is NULL");
  if (B > 0 && !out_path_nodes) return fail(SV_ERR_INVALID_ARG, "out_path_nodes is NULL");
  if (!*greedy && !p.tree.rows && Dq < p.tree.Dmax)  // (per-sequence trees: checked on the device)
    return fail(SV_ERR_INVALID_ARG, "q has %d depth rows, the tree is %d deep", Dq, p.tree.Dmax);
  if (!*greedy && p.tree.rows && Dq < 1 && N > 1)
    return fail(SV_ERR_INVALID_ARG, "q has no depth rows");
  if (!*greedy && q_kind == SV_Q_DRAFT_ONEHOT)
    return fail(SV_ERR_UNSUPPORTED, "one-hot draft q is supported for chains only");
  if (Dq < 0) return fail(SV_ERR_INVALID_ARG, "Dq < 0");
  p.B = B;
  p.N = N;
  p.V = V;
  p.Dq = *greedy ? 0 : Dq;
  p.q_kind = q_kind;
  p.target = target_logits;
  p.q = q;
  p.tokens = node_tokens;
  p.tok_stride = N;
  p.tok_offset = 0;
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.seed = seed;
  p.round = round;
  p.out_path_nodes = out_path_nodes;
  p.out_tokens = out_tokens;
  p.out_num_emitted = out_num_emitted;
  p.out_num_accepted = out_num_accepted;
  p.out_near_ties = out_near_ties;
  return SV_OK;
}

// Validation of a commit's cache and tree K/V, shared by sv_commit_kv and the fused
// acceptance + commit calls; fills everything but the path.
sv_status commit_params(sv_dtype dt, int B, int N, int Hkv, int D, const void *k_tree,
                        const void *v_tree, const sv_kv_cache &cache, sv::CommitParams &p) {
  if (dt != SV_F32 && dt != SV_BF16) return fail(SV_ERR_UNSUPPORTED, "dtype %d", (int)dt);
  if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || Hkv < 1 || D < 1)
    return fail(SV_ERR_INVALID_ARG, "bad sizes B=%d N=%d Hkv=%d D=%d", B, N, Hkv, D);
  const int esize = dt == SV_F32 ? 4 : 2;
  if (((size_t)Hkv * D * esize) % 16 != 0)
    return fail(SV_ERR_UNSUPPORTED, "Hkv*D*elem bytes must be a multiple of 16");
  if (B > 0 && (!k_tree || !v_tree)) return fail(SV_ERR_INVALID_ARG, "k_tree or v_tree is NULL");
  if (!aligned16(k_tree) || !aligned16(v_tree)) return fail(SV_ERR_INVALID_ARG, "k_tree/v_tree not 16-byte aligned");
  sv_status st = check_cache(cache, true, B);
  if (st != SV_OK) return st;
  p = sv::CommitParams{};
  p.k_tree = k_tree;
  p.v_tree = v_tree;
  p.cache_k = cache.k;
  p.cache_v = cache.v;
  p.prefix_len = cache.prefix_len;
  p.block_table = cache.block_table;
  p.B = B;
  p.N = N;
  p.Hkv = Hkv;
  p.D = D;
  p.esize = esize;
  p.Lmax = cache.Lmax;
  p.block_size = cache.block_size;
  p.max_blocks = cache.max_blocks;
  p.num_blocks = cache.num_blocks;
  if (B == 0) return SV_OK;  // an empty batch launches nothing: no device needed
  p.status = status_word();
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  return SV_OK;
}

}  // namespace

sv_status sv_accept_chain(sv_mode mode, sv_dtype logit_dt, int B, int gamma, int V,
                          const void *target_logits, const void *q, sv_q_kind q_kind,
                          const int32_t *draft_tokens, float temperature, int top_k, float top_p,
                          uint64_t seed, uint64_t round, int32_t *out_tokens,
                          int32_t *out_num_emitted, int32_t *out_num_accepted,
                          uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                          void *stream) {
  const CallRange range("sv_accept_chain");
  sv::AcceptParams p;
  bool greedy = false;
  sv_status st = chain_params(mode, logit_dt, B, gamma, V, target_logits, q, q_kind, draft_tokens,
                              temperature, top_k, top_p, seed, round, out_tokens, out_num_emitted,
                              out_num_accepted, out_near_ties, p, &greedy);
  if (st != SV_OK) return st;
  return accept_launch(logit_dt, p, greedy, workspace, workspace_bytes, stream);
}

sv_status sv_accept_tree(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                         const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                         const void *target_logits, const void *q, sv_q_kind q_kind, int Dq,
                         float temperature, int top_k, float top_p, uint64_t seed, uint64_t round,
                         int32_t *out_path_nodes, int32_t *out_tokens,
                         int32_t *out_num_emitted, int32_t *out_num_accepted,
                         uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                         void *stream) {
  const CallRange range("sv_accept_tree");
  sv::AcceptParams p;
  bool greedy = false;
  sv_status st = tree_params(mode, logit_dt, B, N, V, parent, parent_stride, node_tokens, target_logits, q,
                             q_kind, Dq, temperature, top_k, top_p, seed, round, out_path_nodes,
                             out_tokens, out_num_emitted, out_num_accepted, out_near_ties, p,
                             &greedy);
  if (st != SV_OK) return st;
  return accept_launch(logit_dt, p, greedy, workspace, workspace_bytes, stream);
}

sv_status sv_accept_tree_recursive(sv_dtype logit_dt, int B, int N, int V, const int32_t *parent,
                                   int parent_stride,
                                   const int32_t *node_tokens, const void *target_logits,
                                   const void *q, sv_q_kind q_kind, int Dq, float temperature,
                                   int top_k, float top_p, uint64_t seed, uint64_t round,
                                   int32_t *out_path_nodes, int32_t *out_tokens,
                                   int32_t *out_num_emitted, int32_t *out_num_accepted,
                                   uint32_t *out_near_ties, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  const CallRange range("sv_accept_tree_recursive");
  sv::AcceptParams p;
  bool greedy = false;
  sv_status st = tree_params(SV_EXACT, logit_dt, B, N, V, parent, parent_stride, node_tokens, target_logits, q,
                             q_kind, Dq, temperature, top_k, top_p, seed, round, out_path_nodes,
                             out_tokens, out_num_emitted, out_num_accepted, out_near_ties, p,
                             &greedy);
  if (st != SV_OK) return st;
  if (greedy)
    return fail(SV_ERR_UNSUPPORTED,
                "siblings tried in turn need temperature > 0 (greedy: sv_accept_tree)");
  const size_t need = sv::accept_ws_bytes(p.B, p.N, p.Dq);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SV_ERR_WORKSPACE, "acceptance workspace %zu bytes, need %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(SV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  if (p.B == 0) return SV_OK;  // an empty batch: nothing to launch, no device needed
  p.status = status_word();
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  p.mode = SV_EXACT;
  p.c_log2 = (float)(1.4426950408889634 / (double)p.temperature);
  if (p.top_k >= p.V) p.top_k = 0;
  p.stats = static_cast<sv::RowStat *>(workspace);
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure
                                          : sv::launch_accept_recursive(logit_dt, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "recursive tree acceptance launch");
  sv::count_launches(2);
  return SV_OK;
}

sv_status sv_accept_typical(sv_dtype logit_dt, int B, int N, int V, const int32_t *parent,
                           int parent_stride, const int32_t *node_tokens,
                           const void *target_logits, float temperature, float epsilon,
                           float delta, int32_t *out_path_nodes, int32_t *out_tokens,
                           int32_t *out_num_emitted, int32_t *out_num_accepted,
                           uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                           void *stream) {
  const CallRange range("sv_accept_typical");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(SV_ERR_INVALID_ARG, "typical acceptance needs a finite temperature > 0");
  if (!(epsilon >= 0.f) || !std::isfinite(epsilon) || !(delta >= 0.f) || !std::isfinite(delta))
    return fail(SV_ERR_INVALID_ARG, "epsilon and delta must be finite and >= 0");
  sv::AcceptParams p;
  bool greedy = false;
  // the greedy form of the parameters (no q rows, no uniforms); the decisions are typical
  sv_status st = tree_params(SV_GREEDY, logit_dt, B, N, V, parent, parent_stride, node_tokens,
                             target_logits, nullptr, SV_Q_LOGITS, 0, temperature, 0, 1.f, 0, 0,
                             out_path_nodes, out_tokens, out_num_emitted, out_num_accepted,
                             out_near_ties, p, &greedy);
  if (st != SV_OK) return st;
  const size_t need = sv::accept_ws_bytes(p.B, p.N, 0);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SV_ERR_WORKSPACE, "acceptance workspace %zu bytes, need %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(SV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  if (p.B == 0) return SV_OK;  // an empty batch: nothing to launch, no device needed
  p.status = status_word();
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  p.mode = SV_GREEDY;
  p.typical = 1;
  p.typ_eps = epsilon;
  p.typ_delta = delta;
  p.temperature = temperature;
  p.c_log2 = (float)(1.4426950408889634 / (double)temperature);
  p.stats = static_cast<sv::RowStat *>(workspace);
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure
                                          : sv::launch_accept(logit_dt, p, num_sms(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "typical acceptance launch");
  sv::count_launches(2);
  return SV_OK;
}

sv_status sv_accept_chain_commit(sv_mode mode, sv_dtype logit_dt, int B, int gamma, int V,
                                 const void *target_logits, const void *q, sv_q_kind q_kind,
                                 const int32_t *draft_tokens, float temperature, int top_k, float top_p,
                                 uint64_t seed, uint64_t round, sv_dtype kv_dt, int Hkv, int D,
                                 const void *k_tree, const void *v_tree, sv_kv_cache cache,
                                 int32_t *out_tokens, int32_t *out_num_emitted,
                                 int32_t *out_num_accepted, uint32_t *out_near_ties,
                                 void *workspace, size_t workspace_bytes, void *stream) {
  const CallRange range("sv_accept_chain_commit");
  sv::AcceptParams p;
  bool greedy = false;
  sv_status st = chain_params(mode, logit_dt, B, gamma, V, target_logits, q, q_kind, draft_tokens,
                              temperature, top_k, top_p, seed, round, out_tokens, out_num_emitted,
                              out_num_accepted, out_near_ties, p, &greedy);
  if (st != SV_OK) return st;
  if ((st = commit_params(kv_dt, B, gamma + 1, Hkv, D, k_tree, v_tree, cache, p.cm)) != SV_OK)
    return st;
  p.commit = 1;
  return accept_launch(logit_dt, p, greedy, workspace, workspace_bytes, stream);
}

sv_status sv_accept_tree_commit(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                                const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                                const void *target_logits, const void *q, sv_q_kind q_kind,
                                int Dq, float temperature, int top_k, float top_p, uint64_t seed,
                                uint64_t round, sv_dtype kv_dt, int Hkv, int D,
                                const void *k_tree, const void *v_tree, sv_kv_cache cache,
                                int32_t *out_path_nodes, int32_t *out_tokens,
                                int32_t *out_num_emitted, int32_t *out_num_accepted,
                                uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                                void *stream) {
  const CallRange range("sv_accept_tree_commit");
  sv::AcceptParams p;
  bool greedy = false;
  sv_status st = tree_params(mode, logit_dt, B, N, V, parent, parent_stride, node_tokens, target_logits, q,
                             q_kind, Dq, temperature, top_k, top_p, seed, round, out_path_nodes,
                             out_tokens, out_num_emitted, out_num_accepted, out_near_ties, p,
                             &greedy);
  if (st != SV_OK) return st;
  if ((st = commit_params(kv_dt, B, N, Hkv, D, k_tree, v_tree, cache, p.cm)) != SV_OK) return st;
  p.commit = 1;
  return accept_launch(logit_dt, p, greedy, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------- n-gram drafts

sv_status sv_ngram_draft(int B, int Lmax, const int32_t *history, const int32_t *length,
                         int max_ngram, int min_ngram, int gamma, int32_t *out_drafts,
                         int32_t *out_num_drafts, void *stream) {
  const CallRange range("sv_ngram_draft");
  if (B < 0 || Lmax < 1) return fail(SV_ERR_INVALID_ARG, "B = %d, Lmax = %d", B, Lmax);
  if (min_ngram < 1 || max_ngram < min_ngram || max_ngram > SV_MAX_NGRAM)
    return fail(SV_ERR_INVALID_ARG, "n-gram sizes %d..%d (1 <= min <= max <= %d)", min_ngram,
                max_ngram, SV_MAX_NGRAM);
  if (gamma < 1 || gamma >= SV_MAX_TREE_NODES)
    return fail(SV_ERR_UNSUPPORTED, "gamma = %d (supported 1..%d)", gamma, SV_MAX_TREE_NODES - 1);
  if (B > 0 && (!history || !length || !out_drafts || !out_num_drafts))
    return fail(SV_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (B == 0) return SV_OK;  // an empty batch: nothing to launch, no device needed
  sv::NgramParams p{history, length, B, Lmax, max_ngram, min_ngram, gamma, out_drafts,
                    out_num_drafts, status_word()};
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  const cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure
                                                : sv::launch_ngram(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "n-gram draft launch");
  sv::count_launches(1);
  return SV_OK;
}

// --------------------------------------------------------------------- commit

sv_status sv_commit_kv(sv_dtype dt, int B, int N, int Hkv, int D, const void *k_tree,
                       const void *v_tree, const int32_t *path_nodes, int path_stride,
                       const int32_t *num_accepted, sv_kv_cache cache, void *stream) {
  const CallRange range("sv_commit_kv");
  if (path_stride < 1) return fail(SV_ERR_INVALID_ARG, "path_stride = %d", path_stride);
  if (B > 0 && (!path_nodes || !num_accepted))
    return fail(SV_ERR_INVALID_ARG, "path_nodes or num_accepted is NULL");
  sv::CommitParams p;
  sv_status st = commit_params(dt, B, N, Hkv, D, k_tree, v_tree, cache, p);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  p.path_nodes = path_nodes;
  p.path_stride = path_stride;
  p.num_accepted = num_accepted;
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_commit(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  sv::count_launches(1);
  return SV_OK;
}

}  // extern "C"

// ------------------------------------------------- LM head fused with acceptance

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

sv_status lm_head_check(int R, int Dm, int V, const void *hidden, const void *weight,
                        const void *logits) {
  if (R < 0) return fail(SV_ERR_INVALID_ARG, "rows = %d", R);
  if (Dm < 8 || Dm % 8 != 0)
    return fail(SV_ERR_UNSUPPORTED, "hidden size %d must be a positive multiple of 8", Dm);
  if (V < 8 || V % 8 != 0) return fail(SV_ERR_UNSUPPORTED, "V = %d must be a positive multiple of 8", V);
  if (R > 0 && (!hidden || !weight || !logits))
    return fail(SV_ERR_INVALID_ARG, "hidden, weight or logits is NULL");
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(logits))
    return fail(SV_ERR_INVALID_ARG, "hidden, weight and logits must be 16-byte aligned");
  return SV_OK;
}

// The projection of the B*N target rows, then the acceptance on the stored logits.  With no
// top-k / top-p the projection's epilogue gives the target rows' statistics (the statistics
// kernel then runs over the q rows only); otherwise the statistics kernel reads every row.
sv_status lm_head_accept_launch(sv::AcceptParams &p, bool greedy, int Dm, const void *hidden,
                                const void *weight, void *workspace, size_t workspace_bytes,
                                void *stream) {
  const size_t st_bytes = up256(sv::accept_ws_bytes(p.B, p.N, p.Dq));
  const size_t need = st_bytes + sv::lm_head_part_bytes(p.B * p.N, p.V);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(SV_ERR_WORKSPACE, "LM-head acceptance workspace %zu bytes, need %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(SV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  if (p.B == 0) return SV_OK;  // an empty batch: nothing to launch, no device needed
  p.status = status_word();
  if (!p.status) return fail(SV_ERR_CUDA, "no CUDA device");
  p.mode = greedy ? SV_GREEDY : SV_EXACT;
  p.c_log2 = greedy ? 0.f : (float)(1.4426950408889634 / (double)p.temperature);
  if (p.top_k >= p.V) p.top_k = 0;
  if (greedy) p.top_p = 1.f;
  p.stats = static_cast<sv::RowStat *>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool epilogue_stats = greedy || p.top_k == 0;  // (top_p < 1 needs top-k)
  void *part = static_cast<uint8_t *>(workspace) + st_bytes;
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_lm_head(hidden, weight, p.B * p.N, Dm, p.V, p.c_log2,
                                     const_cast<void *>(p.target), epilogue_stats ? part : nullptr,
                                     epilogue_stats ? p.stats : nullptr, p.status, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "LM-head projection launch");
  sv::count_launches(epilogue_stats ? 2 : 1);
  if (epilogue_stats) {
    e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_accept_given_target_stats(SV_BF16, p, num_sms(), s);
    const bool q_stats = !greedy && p.q_kind == SV_Q_LOGITS && p.Dq > 0;
    if (e == cudaSuccess) sv::count_launches(q_stats ? 2 : 1);
  } else {
    e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_accept(SV_BF16, p, num_sms(), s);
    if (e == cudaSuccess) sv::count_launches(2);
  }
  if (e != cudaSuccess) return cuda_fail(e, "acceptance launch");
  return SV_OK;
}

}  // namespace

extern "C" {

sv_status sv_lm_head(int R, int Dm, int V, const void *hidden, const void *weight, void *logits,
                     void *stream) {
  const CallRange range("sv_lm_head");
  sv_status st = lm_head_check(R, Dm, V, hidden, weight, logits);
  if (st != SV_OK) return st;
  if (R == 0) return SV_OK;  // no rows: nothing to launch, no device needed
  unsigned int *status = status_word();
  if (!status) return fail(SV_ERR_CUDA, "no CUDA device");
  cudaError_t e = take_injected_failure() ? cudaErrorLaunchFailure : sv::launch_lm_head(hidden, weight, R, Dm, V, 0.f, logits, nullptr, nullptr,
                                     status, num_sms(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "LM-head projection launch");
  sv::count_launches(1);
  return SV_OK;
}

size_t sv_accept_lmhead_workspace_size(int B, int N, int V, int Dq) {
  if (B <= 0 || N <= 0 || V <= 0 || Dq < 0) return 0;
  return up256(sv::accept_ws_bytes(B, N, Dq)) + sv::lm_head_part_bytes(B * N, V);
}

sv_status sv_accept_chain_lmhead(sv_mode mode, int B, int gamma, int V, int Dm, const void *hidden,
                                 const void *weight, void *target_logits, const void *q,
                                 sv_q_kind q_kind, const int32_t *draft_tokens, float temperature,
                                 int top_k, float top_p, uint64_t seed, uint64_t round,
                                 int32_t *out_tokens, int32_t *out_num_emitted,
                                 int32_t *out_num_accepted, uint32_t *out_near_ties,
                                 void *workspace, size_t workspace_bytes, void *stream) {
  const CallRange range("sv_accept_chain_lmhead");
  sv_status st = lm_head_check(B * (gamma + 1), Dm, V, hidden, weight, target_logits);
  if (st != SV_OK) return st;
  sv::AcceptParams p;
  bool greedy = false;
  st = chain_params(mode, SV_BF16, B, gamma, V, target_logits, q, q_kind, draft_tokens,
                    temperature, top_k, top_p, seed, round, out_tokens, out_num_emitted,
                    out_num_accepted, out_near_ties, p, &greedy);
  if (st != SV_OK) return st;
  return lm_head_accept_launch(p, greedy, Dm, hidden, weight, workspace, workspace_bytes, stream);
}

sv_status sv_accept_tree_lmhead(sv_mode mode, int B, int N, int V, int Dm, const void *hidden,
                                const void *weight, void *target_logits, const int32_t *parent,
                                int parent_stride, const int32_t *node_tokens, const void *q,
                                sv_q_kind q_kind, int Dq, float temperature, int top_k,
                                float top_p, uint64_t seed, uint64_t round,
                                int32_t *out_path_nodes, int32_t *out_tokens,
                                int32_t *out_num_emitted, int32_t *out_num_accepted,
                                uint32_t *out_near_ties, void *workspace, size_t workspace_bytes,
                                void *stream) {
  const CallRange range("sv_accept_tree_lmhead");
  sv_status st = lm_head_check(B * N, Dm, V, hidden, weight, target_logits);
  if (st != SV_OK) return st;
  sv::AcceptParams p;
  bool greedy = false;
  st = tree_params(mode, SV_BF16, B, N, V, parent, parent_stride, node_tokens, target_logits, q,
                   q_kind, Dq, temperature, top_k, top_p, seed, round, out_path_nodes, out_tokens,
                   out_num_emitted, out_num_accepted, out_near_ties, p, &greedy);
  if (st != SV_OK) return st;
  return lm_head_accept_launch(p, greedy, Dm, hidden, weight, workspace, workspace_bytes, stream);
}

}  // extern "C"

// ------------------------------------------------- acceptance without allocation

// Scratch of sv_accept_tree_noalloc: the per-row statistics (row max, argmax, top-k
// threshold, softmax sum) that the first acceptance kernel writes and the second
// reads.  A fixed array in device memory instead of a caller workspace, so that
// callers which cannot allocate device memory can still run acceptance.  Every GPU
// that loads this library holds it (SV_NOALLOC_ACCEPT_ROWS rows of 32 bytes) until
// the process exits.
static __device__ __align__(256) sv::RowStat g_sv_noalloc_rows[SV_NOALLOC_ACCEPT_ROWS];

namespace {

// Device address of the scratch array on the current device.  Looked up once per
// device, with that device current; host code must never pass the array's name.
void *noalloc_rows_address(sv_status *st) {
  static std::atomic<void *> addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = e != cudaSuccess ? cuda_fail(e, "cudaGetDevice") : fail(SV_ERR_CUDA, "device index out of range");
    return nullptr;
  }
  void *a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sv_noalloc_rows);
    if (e != cudaSuccess || p == nullptr) {
      *st = cuda_fail(e, "cudaGetSymbolAddress of the acceptance scratch array");
      return nullptr;
    }
    a = p;  // threads racing on the first lookup store the same address
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

}  // namespace

extern "C" {

sv_status sv_accept_tree_noalloc(sv_mode mode, sv_dtype logit_dt, int B, int N, int V,
                                 const int32_t *parent, int parent_stride, const int32_t *node_tokens,
                                 const void *target_logits, const void *q, sv_q_kind q_kind,
                                 int Dq, float temperature, int top_k, float top_p, uint64_t seed,
                                 uint64_t round, int32_t *out_path_nodes, int32_t *out_tokens,
                                 int32_t *out_num_emitted, int32_t *out_num_accepted,
                                 uint32_t *out_near_ties, void *stream) {
  const CallRange range("sv_accept_tree_noalloc");
  const bool greedy = mode == SV_GREEDY || temperature == 0.f;
  const long long rows = (long long)B * ((long long)N + (greedy ? 0 : (Dq > 0 ? Dq : 0)));
  if (rows > SV_NOALLOC_ACCEPT_ROWS)
    return fail(SV_ERR_UNSUPPORTED,
                "sv_accept_tree_noalloc: B*(N+Dq) = %lld logit rows exceeds its fixed scratch of "
                "%d rows; use sv_accept_tree with a workspace",
                rows, SV_NOALLOC_ACCEPT_ROWS);
  sv_status st = SV_OK;
  void *scratch = nullptr;  // (an empty batch needs none, and no device)
  if (B > 0) {
    scratch = noalloc_rows_address(&st);
    if (!scratch) return st;
  }
  return sv_accept_tree(mode, logit_dt, B, N, V, parent, parent_stride, node_tokens, target_logits, q, q_kind,
                        Dq, temperature, top_k, top_p, seed, round, out_path_nodes, out_tokens,
                        out_num_emitted, out_num_accepted, out_near_ties, scratch,
                        scratch ? sizeof(g_sv_noalloc_rows) : 0, stream);
}

}  // extern "C"
