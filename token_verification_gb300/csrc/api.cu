// api.cu - the extern "C" entry points declared in include/spec_verify.h:
// argument validation on the host, workspace carving, and dispatch to the
// kernels of sv_verify.cu / sv_tree.cu.  Nothing here allocates memory or
// synchronises the stream.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"
#include "sv_launch.h"

namespace sv {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// The region that must hold zeros when a call starts (the error flag, the
// finalize ticket, the streaming kernel's work counter and the dense-draft
// residual's counters) comes first; every call leaves it zero again.
static WorkspaceLayout layout_for(int B, int R, int V) {
  const size_t NC = ((size_t)V + kChunk - 1) / kChunk;
  WorkspaceLayout l;
  size_t o = 0;
  l.counters = o;   o += 8 * sizeof(int);
  l.arrive = o;     o = align256(o + sizeof(int) * (size_t)B);
  l.zero_bytes = o;
  l.pend = o;       o = align256(o + 2 * sizeof(int) * (size_t)B);
  l.rpar = o;       o = align256(o + sizeof(float4) * (size_t)B);
  l.rsums = o;      o = align256(o + sizeof(float) * (size_t)B * NC);
  l.rec = o;        o = align256(o + sizeof(float2) * (size_t)B * R * NC);
  l.lx = o;         o = align256(o + sizeof(float) * (size_t)B * R);
  l.thr = o;        o = align256(o + sizeof(float) * (size_t)B * R);
  l.ent = o;        o = align256(o + sizeof(float) * (size_t)B * R * NC);
  l.total = o;
  return l;
}

WorkspaceLayout workspace_layout(int B, int K, int V) { return layout_for(B, 2 * K + 1, V); }

cudaError_t device_info(DeviceInfo* out) {
  static std::atomic<int> sms[64];  // 0 until read; racing readers store the same value
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (!n) {
    err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  out->sms = n;
  return cudaSuccess;
}

// Which zero-region layout each workspace was last used with.  A call whose
// layout differs (or a workspace not seen before) first zero-fills the
// region on its stream, so calls of different shapes may share a workspace.
namespace {
struct WsKey {
  int B, R;
  bool operator==(const WsKey& o) const { return B == o.B && R == o.R; }
};
std::mutex g_ws_mu;
std::unordered_map<const void*, WsKey> g_ws_keys;
}  // namespace

static cudaError_t prepare_workspace(void* ws, const WorkspaceLayout& l, int B, int R,
                                     cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const WsKey key{B, R};
  auto it = g_ws_keys.find(ws);
  if (it != g_ws_keys.end() && it->second == key) return cudaSuccess;
  const cudaError_t err = cudaMemsetAsync(ws, 0, l.zero_bytes, stream);
  if (err == cudaSuccess) g_ws_keys[ws] = key;
  return err;
}

static void forget_workspace(const void* ws) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  g_ws_keys.erase(ws);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The limit of the kernels' waits for staged logits (spec_verify_set_wait_limit_ns).
static std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

static sv_status verify_common(int mode, const void* target, const void* draft,
                               const int32_t* draft_tokens, const float* uniforms, float T,
                               int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype, int B,
                               int K, int V, const int32_t* draft_lens, int32_t* out_cu,
                               int32_t* out_packed, int32_t* out_batch_id, float* out_accept_prob,
                               int32_t* out_status, void* ws, size_t ws_bytes,
                               cudaStream_t stream, int greedy_prob,
                               const uint32_t* mask = nullptr, int top_k = 0,
                               float top_p = 1.f, float eps = 0.f, float delta = 0.f,
                               float* out_cut = nullptr) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B > SV_MAX_B || K < 0 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return SV_ERR_SHAPE;
  if (B == 0) {
    if (out_cu && cudaMemsetAsync(out_cu, 0, sizeof(int32_t), stream) != cudaSuccess)
      return SV_ERR_CUDA;
    return SV_OK;
  }
  if (!target || !out_tokens || !out_accept_len) return SV_ERR_NULL;
  if (K > 0 && !draft_tokens) return SV_ERR_NULL;
  if (mode != kGreedy && !uniforms) return SV_ERR_NULL;
  const int R = (mode == kDense) ? 2 * K + 1 : K + 1;
  const WorkspaceLayout l = layout_for(B, R, V);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < l.total) return SV_ERR_WORKSPACE;

  const int vec_elems = dtype == SV_BF16 ? 8 : 4;
  const bool vec = (V % vec_elems == 0) && aligned16(target) && (!draft || aligned16(draft));
  const int G = chunks_per_task(dtype, vec);

  VerifyParams p;
  memset(&p, 0, sizeof p);
  p.target = target;
  p.draft = draft;
  p.draft_tokens = draft_tokens;
  p.draft_lens = draft_lens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_accept_prob = out_accept_prob;
  p.out_status = out_status;
  p.out_cu = out_cu;
  p.out_packed = out_packed;
  p.out_batch_id = out_batch_id;
  p.mask = mask;
  p.mask_words = (V + 31) / 32;
  p.mask_bulk = (mask && vec && aligned16(mask) && p.mask_words % 4 == 0) ? 1 : 0;
  p.top_k = top_k;
  p.top_p = top_p;
  p.filter = (mode != kGreedy && ((top_k > 0 && top_k < V) || top_p < 1.f)) ? 1 : 0;
  if (p.filter) {  // one CTA per row
    const long long esz = dtype == SV_BF16 ? 2 : 4;
    if ((long long)V * esz > kFilterRowBytes || (long long)B * R >= (1LL << 31)) return SV_ERR_SHAPE;
  }
  char* base = static_cast<char*>(ws);
  p.err = reinterpret_cast<int*>(base + l.counters);
  p.fin_ticket = p.err + 1;
  p.work = reinterpret_cast<unsigned*>(p.err + 2);
  p.n_pend = p.err + 3;
  p.r_exit = p.err + 4;
  p.n_bonus = p.err + 5;
  p.arrive = reinterpret_cast<int*>(base + l.arrive);
  p.pend = reinterpret_cast<int*>(base + l.pend);
  p.rpn = p.pend + B;
  p.rpar = reinterpret_cast<float4*>(base + l.rpar);
  p.rsums = reinterpret_cast<float*>(base + l.rsums);
  p.rec = reinterpret_cast<float2*>(base + l.rec);
  p.lx = reinterpret_cast<float*>(base + l.lx);
  p.thr = reinterpret_cast<float*>(base + l.thr);
  p.ent = reinterpret_cast<float*>(base + l.ent);
  p.eps = eps;
  p.delta = delta;
  p.B = B;
  p.K = K;
  p.V = V;
  p.NC = (V + kChunk - 1) / kChunk;
  p.R = R;
  p.TPR = (p.NC + G - 1) / G;
  p.item_chunks = G;
  p.total_tasks = (long long)B * R * p.TPR;
  if (p.total_tasks >= (1LL << 31)) return SV_ERR_SHAPE;
  p.div_tpr = make_fastdiv((uint32_t)p.TPR);
  p.div_r = make_fastdiv((uint32_t)R);
  p.cc = mode == kGreedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  p.greedy_prob = greedy_prob;
  p.compact_in_finalize = (out_cu || out_packed || out_batch_id) ? 1 : 0;
  p.fin_cache = fin_cache_bytes(p) <= kFinCacheLimit ? 1 : 0;
  p.out_cut = p.filter ? out_cut : nullptr;
  p.wait_ns = wait_limit_ns();
  if (prepare_workspace(ws, l, B, R, stream) != cudaSuccess) return SV_ERR_CUDA;
  return launch_verify(mode, dtype, vec, p, stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int B, int K, int V) {
  if (B < 0 || B > SV_MAX_B || K < 0 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return 0;
  return workspace_layout(B, K, V).total;
}

sv_status spec_verify_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!workspace) return SV_ERR_NULL;
  forget_workspace(workspace);
  if (cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

sv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                             const int32_t* draft_tokens, const float* uniforms, float temperature,
                             int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype, int B,
                             int K, int V, const int32_t* draft_lens, int32_t* out_cu_accept,
                             int32_t* out_packed, int32_t* out_batch_id, float* out_accept_prob,
                             int32_t* out_status, void* workspace, size_t ws_bytes,
                             sv_stream_t stream) {
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  const int mode = temperature == 0.f ? kGreedy : (draft_logits ? kDense : kOneHot);
  return verify_common(mode, target_logits, mode == kDense ? draft_logits : nullptr, draft_tokens,
                       uniforms, temperature, out_tokens, out_accept_len, dtype, B, K, V,
                       draft_lens, out_cu_accept, out_packed, out_batch_id, out_accept_prob,
                       out_status, workspace, ws_bytes, (cudaStream_t)stream, 1);
}

sv_status spec_verify_sample_masked(const void* target_logits, const void* draft_logits,
                                    const int32_t* draft_tokens, const float* uniforms,
                                    float temperature, const uint32_t* token_mask,
                                    int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype,
                                    int B, int K, int V, const int32_t* draft_lens,
                                    int32_t* out_cu_accept, int32_t* out_packed,
                                    int32_t* out_batch_id, float* out_accept_prob,
                                    int32_t* out_status, void* workspace, size_t ws_bytes,
                                    sv_stream_t stream) {
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  if (B > 0 && (!token_mask || ((uintptr_t)token_mask & 3u))) return SV_ERR_NULL;
  const int mode = temperature == 0.f ? kGreedy : (draft_logits ? kDense : kOneHot);
  return verify_common(mode, target_logits, mode == kDense ? draft_logits : nullptr, draft_tokens,
                       uniforms, temperature, out_tokens, out_accept_len, dtype, B, K, V,
                       draft_lens, out_cu_accept, out_packed, out_batch_id, out_accept_prob,
                       out_status, workspace, ws_bytes, (cudaStream_t)stream, 1, token_mask);
}

sv_status spec_verify_greedy_masked(const void* target_logits, const int32_t* draft_tokens,
                                    const uint32_t* token_mask, int32_t* out_tokens,
                                    int32_t* out_accept_len, sv_dtype dtype, int B, int K, int V,
                                    const int32_t* draft_lens, int32_t* out_cu_accept,
                                    int32_t* out_packed, int32_t* out_batch_id,
                                    int32_t* out_status, void* workspace, size_t ws_bytes,
                                    sv_stream_t stream) {
  if (B > 0 && (!token_mask || ((uintptr_t)token_mask & 3u))) return SV_ERR_NULL;
  return verify_common(kGreedy, target_logits, nullptr, draft_tokens, nullptr, 0.f, out_tokens,
                       out_accept_len, dtype, B, K, V, draft_lens, out_cu_accept, out_packed,
                       out_batch_id, nullptr, out_status, workspace, ws_bytes,
                       (cudaStream_t)stream, 0, token_mask);
}

sv_status spec_verify_sample_filtered(const void* target_logits, const void* draft_logits,
                                      const int32_t* draft_tokens, const float* uniforms,
                                      float temperature, int top_k, float top_p,
                                      const uint32_t* token_mask, int32_t* out_tokens,
                                      int32_t* out_accept_len, sv_dtype dtype, int B, int K, int V,
                                      const int32_t* draft_lens, int32_t* out_cu_accept,
                                      int32_t* out_packed, int32_t* out_batch_id,
                                      float* out_accept_prob, float* out_cut,
                                      int32_t* out_status, void* workspace, size_t ws_bytes,
                                      sv_stream_t stream) {
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  if (top_k < 0 || !(top_p > 0.f && top_p <= 1.f)) return SV_ERR_FILTER;
  if (token_mask && ((uintptr_t)token_mask & 3u)) return SV_ERR_NULL;
  const int mode = temperature == 0.f ? kGreedy : (draft_logits ? kDense : kOneHot);
  return verify_common(mode, target_logits, mode == kDense ? draft_logits : nullptr, draft_tokens,
                       uniforms, temperature, out_tokens, out_accept_len, dtype, B, K, V,
                       draft_lens, out_cu_accept, out_packed, out_batch_id, out_accept_prob,
                       out_status, workspace, ws_bytes, (cudaStream_t)stream, 1, token_mask, top_k,
                       top_p, 0.f, 0.f, out_cut);
}

sv_status spec_verify_typical(const void* target_logits, const int32_t* draft_tokens,
                              const float* uniforms, float temperature, float eps, float delta,
                              int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype, int B,
                              int K, int V, const int32_t* draft_lens, int32_t* out_cu_accept,
                              int32_t* out_packed, int32_t* out_batch_id, float* out_accept_prob,
                              int32_t* out_status, void* workspace, size_t ws_bytes,
                              sv_stream_t stream) {
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  if (!(eps >= 0.f) || !(delta >= 0.f) || isinf(eps) || isinf(delta)) return SV_ERR_FILTER;
  const int mode = temperature == 0.f ? kGreedy : kTypical;
  return verify_common(mode, target_logits, nullptr, draft_tokens, uniforms, temperature,
                       out_tokens, out_accept_len, dtype, B, K, V, draft_lens, out_cu_accept,
                       out_packed, out_batch_id, out_accept_prob, out_status, workspace, ws_bytes,
                       (cudaStream_t)stream, 1, nullptr, 0, 1.f, eps, delta);
}

size_t spec_verify_tree_workspace_size(int B, int N, int V) {
  if (B < 0 || B > SV_MAX_B || N < 0 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_V) return 0;
  return layout_for(B, N + 1, V).total;
}

}  // extern "C"

namespace sv {

// Kernel A over every row of a candidate tree (B * (N+1) rows), then the
// tree's own finalize kernel: typical acceptance or rejection sampling.
static sv_status tree_rows_call(int mode, const void* target, const int32_t* tree_parent,
                                int parent_stride, const int32_t* tree_tokens,
                                const float* uniforms, float T, float eps, float delta,
                                int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype,
                                int B, int N, int V, int max_depth, int32_t* out_path,
                                int32_t* out_status, void* workspace, size_t ws_bytes,
                                cudaStream_t stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B > SV_MAX_B || N < 0 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_V ||
      max_depth < 0 || max_depth > SV_MAX_TREE_NODES)
    return SV_ERR_SHAPE;
  if (parent_stride != 0 && parent_stride != N) return SV_ERR_TREE;
  if (B == 0) return SV_OK;
  if (!target || !out_tokens || !out_accept_len || !uniforms) return SV_ERR_NULL;
  if (N > 0 && (!tree_parent || !tree_tokens)) return SV_ERR_NULL;
  const int R = N + 1;
  const WorkspaceLayout l = layout_for(B, R, V);
  if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < l.total) return SV_ERR_WORKSPACE;
  const int vec_elems = dtype == SV_BF16 ? 8 : 4;
  const bool vec = (V % vec_elems == 0) && aligned16(target);
  const int G = chunks_per_task(dtype, vec);
  VerifyParams p;
  memset(&p, 0, sizeof p);
  p.target = target;
  char* base = static_cast<char*>(workspace);
  p.err = reinterpret_cast<int*>(base + l.counters);
  p.fin_ticket = p.err + 1;
  p.work = reinterpret_cast<unsigned*>(p.err + 2);
  p.n_pend = p.err + 3;
  p.r_exit = p.err + 4;
  p.n_bonus = p.err + 5;
  p.arrive = reinterpret_cast<int*>(base + l.arrive);
  p.pend = reinterpret_cast<int*>(base + l.pend);
  p.rpn = p.pend + B;
  p.rpar = reinterpret_cast<float4*>(base + l.rpar);
  p.rsums = reinterpret_cast<float*>(base + l.rsums);
  p.rec = reinterpret_cast<float2*>(base + l.rec);
  p.lx = reinterpret_cast<float*>(base + l.lx);
  p.thr = reinterpret_cast<float*>(base + l.thr);
  p.ent = reinterpret_cast<float*>(base + l.ent);
  p.mask_words = (V + 31) / 32;
  p.top_p = 1.f;
  p.eps = eps;
  p.delta = delta;
  p.B = B;
  p.K = N;  // the tree's rows play the part of positions 0..N
  p.V = V;
  p.NC = (V + kChunk - 1) / kChunk;
  p.R = R;
  p.TPR = (p.NC + G - 1) / G;
  p.item_chunks = G;
  p.total_tasks = (long long)B * R * p.TPR;
  if (p.total_tasks >= (1LL << 31)) return SV_ERR_SHAPE;
  p.div_tpr = make_fastdiv((uint32_t)p.TPR);
  p.div_r = make_fastdiv((uint32_t)R);
  // every row of the tree is needed and the rows are contiguous: on the
  // streaming path items run across row boundaries, all G chunks long
  const long long chunks = (long long)B * R * p.NC;
  if (vec && chunks < (1LL << 31)) {
    p.flat = 1;
    p.total_chunks = (int)chunks;
    p.div_nc = make_fastdiv((uint32_t)p.NC);
    p.total_tasks = (chunks + G - 1) / G;
  }
  p.cc = (float)(1.4426950408889634 / (double)T);
  p.wait_ns = wait_limit_ns();
  p.tree_parent = tree_parent;
  p.parent_stride = parent_stride;
  p.tree_tokens = tree_tokens;
  TreeCall t;
  memset(&t, 0, sizeof t);
  t.parent = tree_parent;
  t.parent_stride = parent_stride;
  t.tokens = tree_tokens;
  t.uniforms = uniforms;
  t.out_tokens = out_tokens;
  t.out_accept_len = out_accept_len;
  t.out_path = out_path;
  t.out_status = out_status;
  t.N = N;
  t.D1 = max_depth + 1;
  if (prepare_workspace(workspace, l, B, R, stream) != cudaSuccess) return SV_ERR_CUDA;
  const cudaError_t err = mode == kTreeSample ? launch_tree_sample(dtype, vec, p, t, stream)
                                              : launch_tree_typical(dtype, vec, p, t, stream);
  return err == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

extern "C" {

sv_status spec_verify_tree_typical(const void* target_logits, const int32_t* tree_parent,
                                   int parent_stride, const int32_t* tree_tokens,
                                   const float* uniforms, float temperature, float eps,
                                   float delta, int32_t* out_tokens, int32_t* out_accept_len,
                                   sv_dtype dtype, int B, int N, int V, int max_depth,
                                   int32_t* out_path, int32_t* out_status, void* workspace,
                                   size_t ws_bytes, sv_stream_t stream) {
  if (!(temperature > 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  if (!(eps >= 0.f) || !(delta >= 0.f) || isinf(eps) || isinf(delta)) return SV_ERR_FILTER;
  return tree_rows_call(kTypical, target_logits, tree_parent, parent_stride, tree_tokens, uniforms,
                        temperature, eps, delta, out_tokens, out_accept_len, dtype, B, N, V,
                        max_depth, out_path, out_status, workspace, ws_bytes,
                        (cudaStream_t)stream);
}

sv_status spec_verify_tree_sample(const void* target_logits, const int32_t* tree_parent,
                                  int parent_stride, const int32_t* tree_tokens,
                                  const float* uniforms, float temperature, int32_t* out_tokens,
                                  int32_t* out_accept_len, sv_dtype dtype, int B, int N, int V,
                                  int max_depth, int32_t* out_path, int32_t* out_status,
                                  void* workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_TEMPERATURE;
  if (temperature == 0.f)  // the greedy rule: the argmax walk
    return spec_verify_tree(target_logits, tree_parent, parent_stride, tree_tokens, out_tokens,
                            out_accept_len, dtype, B, N, V, max_depth, out_path, out_status,
                            stream);
  return tree_rows_call(kTreeSample, target_logits, tree_parent, parent_stride, tree_tokens,
                        uniforms, temperature, 0.f, 0.f, out_tokens, out_accept_len, dtype, B, N,
                        V, max_depth, out_path, out_status, workspace, ws_bytes,
                        (cudaStream_t)stream);
}

sv_status spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens,
                             int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype, int B,
                             int K, int V, const int32_t* draft_lens, int32_t* out_cu_accept,
                             int32_t* out_packed, int32_t* out_batch_id, int32_t* out_status,
                             void* workspace, size_t ws_bytes, sv_stream_t stream) {
  return verify_common(kGreedy, target_logits, nullptr, draft_tokens, nullptr, 0.f, out_tokens,
                       out_accept_len, dtype, B, K, V, draft_lens, out_cu_accept, out_packed,
                       out_batch_id, nullptr, out_status, workspace, ws_bytes,
                       (cudaStream_t)stream, 0);
}

sv_status spec_verify_tree(const void* target_logits, const int32_t* tree_parent,
                           int parent_stride, const int32_t* tree_tokens, int32_t* out_tokens,
                           int32_t* out_accept_len, sv_dtype dtype, int B, int N, int V,
                           int max_depth, int32_t* out_path, int32_t* out_status,
                           sv_stream_t stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B > SV_MAX_B || N < 0 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_V ||
      max_depth < 0 || max_depth > SV_MAX_TREE_NODES)
    return SV_ERR_SHAPE;
  if (parent_stride != 0 && parent_stride != N) return SV_ERR_TREE;
  if (B == 0) return SV_OK;
  if (!target_logits || !out_tokens || !out_accept_len) return SV_ERR_NULL;
  if (N > 0 && (!tree_parent || !tree_tokens)) return SV_ERR_NULL;
  TreeParams p;
  memset(&p, 0, sizeof p);
  p.target = target_logits;
  p.parent = tree_parent;
  p.parent_stride = parent_stride;
  p.tokens = tree_tokens;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_path = out_path;
  p.out_status = out_status;
  p.B = B;
  p.N = N;
  p.V = V;
  p.D1 = max_depth + 1;
  p.NC = (V + kChunk - 1) / kChunk;
  const int vec_elems = dtype == SV_BF16 ? 8 : 4;
  const bool vec = (V % vec_elems == 0) && aligned16(target_logits);
  return launch_tree(dtype, vec, p, (cudaStream_t)stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_ns.store((unsigned long long)limit_ns, std::memory_order_relaxed);
  return SV_OK;
}

uint64_t spec_verify_wait_limit_ns(void) { return (uint64_t)wait_limit_ns(); }

const char* spec_verify_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_SHAPE: return "shape outside the supported range";
    case SV_ERR_DTYPE: return "unknown dtype";
    case SV_ERR_TEMPERATURE: return "temperature negative, NaN or infinite";
    case SV_ERR_TREE: return "tree parent stride is neither 0 nor N";
    case SV_ERR_WORKSPACE: return "workspace NULL, misaligned or too small";
    case SV_ERR_CUDA: return "CUDA launch failed";
    case SV_ERR_FILTER: return "top_k negative or top_p outside (0, 1]";
  }
  return "unknown status";
}

int spec_verify_version(void) { return 101; }

}  // extern "C"
