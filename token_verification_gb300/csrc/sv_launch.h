// sv_launch.h - kernel parameter blocks and launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_common.cuh"

namespace sv {

// Summary of one logit row, built by the finalize kernel from the row's
// chunk records.  Softmax rows: m = row max (NaN if the row is unusable),
// s = sum of 2^((l_j - m) c) (without the draft token for the rows of one-hot
// drafts), wx = 2^((l_x - m) c) for the row's draft token x.  Argmax rows:
// m = max, idx = lowest index attaining it.
struct RowSum {
  float m;
  float s;
  float wx;
  int idx;
  float h;  // typical acceptance: the row's entropy in nats
};

struct VerifyParams {
  const void* target;
  const void* draft;
  const int* draft_tokens;
  const int* draft_lens;
  const float* uniforms;
  int* out_tokens;
  int* out_accept_len;
  float* out_accept_prob;
  int* out_status;
  int* out_cu;
  int* out_packed;
  int* out_batch_id;
  const uint32_t* mask;  // [B, K+1, mask_words] grammar masks, or null
  int mask_words;        // ceil(V / 32)
  int mask_bulk;         // mask rows are 16-byte aligned: copied with the logits
  int top_k;             // 0: off
  float top_p;           // 1: off
  int filter;            // top-k / top-p active: kernel A is the row-per-cluster filter kernel
  float* thr;            // [B*R] each row's cut value (lowest kept logit), filter calls
  float* ent;            // [B*R*NC] chunk entropy accumulators (typical acceptance)
  float eps, delta;      // typical acceptance: p(x) > min(eps, delta * exp(-H))
  // workspace
  int* err;          // [1] set when a bounded wait gave up
  int* fin_ticket;   // [1] requests finalised in this call
  unsigned* work;    // [1] the streaming kernel's next item (taken by atomic add)
  // dense drafts: the requests rejected at n whose residual the residual
  // kernel reads (published by the finalize kernel)
  int* n_pend;       // [1] rejected requests published
  int* r_exit;       // [1] residual CTAs finished
  int* n_bonus;      // [1] dense requests whose drafts all passed (bonus draws in kernel R)
  int* arrive;       // [B] chunk groups done per published slot
  int* pend;         // [B] the request of each slot (bonus draws from the back)
  int* rpn;          // [B] its rejected position n (or K_b for a bonus draw)
  float4* rpar;      // [B] {row max, 1/sum} of its target and draft rows at n
  float* rsums;      // [B*NC] residual chunk sums per slot
  float2* rec;       // [B*R*NC]
  float* lx;         // [B*R] the logit of each row's draft token
  int B, K, V;
  int NC;            // chunks per row
  int R;             // rows per request: K+1 target (+ K draft rows when dense)
  int TPR;           // stream items per row
  int item_chunks;   // chunks per stream item
  long long total_tasks;  // < 2^31 (checked on the host)
  FastDiv div_tpr, div_r; // divide by TPR and by R
  // Items across row boundaries: item it is chunks it*item_chunks onwards of
  // the call's rows in order (every row needed, rows at a stride of V, no
  // draft tokens or masks: the tree calls), so every item but the last is
  // item_chunks long whatever V; 0: items stop at the end of each row.
  int flat;
  int total_chunks;       // B * R * NC when flat (< 2^31)
  FastDiv div_nc;         // divide by NC
  float cc;          // log2(e) / T
  int greedy_prob;   // greedy rule reached through the sampling entry
  int compact_in_finalize;  // the finalize kernel writes the packed output
  int fin_cache;     // the finalize kernel keeps the request's records in shared memory
  float* out_cut;    // [B*R] filtered calls: each row's cut value (NaN: row not needed), or null
  unsigned long long wait_ns;  // limit of the waits for staged logits (0: give up at once)
  // tree sampling (kernel A leaves each node's children tokens out of its row's sums)
  const int* tree_parent;  // request b's parents at tree_parent + b * parent_stride
  int parent_stride;       // 0 (one tree for all requests) or N
  const int* tree_tokens;  // [B, N]
};

constexpr int kMaxTreeNodes = 256;

// Greedy tree walk.  The parent arrays live in device memory: request b's
// at parent + b * parent_stride (parent of node n at index n - 1).
struct TreeParams {
  const void* target;
  const int* parent;  // [N] or [B, N]
  int parent_stride;  // 0 or N
  const int* tokens;  // [B, N]
  int* out_tokens;
  int* out_accept_len;
  int* out_path;
  int* out_status;
  int B, N, V, D1, NC;
};

// Candidate tree of typical acceptance and of tree sampling (after kernel A
// over every tree row).
struct TreeCall {
  const int* parent;      // [N] or [B, N] (device)
  int parent_stride;      // 0 or N
  const int* tokens;      // [B, N] node n's token at n - 1
  const float* uniforms;  // typical: [B] the final draw; sampling: [B, N+1]
  int* out_tokens;        // [B, D1]
  int* out_accept_len;    // [B]
  int* out_path;          // [B, D1] or null
  int* out_status;        // [B] or null
  int N, D1;
};

enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Workspace layout for B requests, K positions, V vocabulary (dense case).
struct WorkspaceLayout {
  size_t counters, arrive, zero_bytes, pend, rpar, rsums, rec, lx, thr, ent, total;
};
WorkspaceLayout workspace_layout(int B, int K, int V);

struct DeviceInfo {
  int sms;
};
cudaError_t device_info(DeviceInfo* out);

// Chunks per stream item (row-statistics kernel).
int chunks_per_task(int dtype, bool vec);
// Shared memory the finalize kernel uses to keep a request's chunk records,
// and its whole dynamic shared memory (the records when cached, then the
// residual chunk sums of dense drafts).
size_t fin_cache_bytes(const VerifyParams& p);
size_t fin_smem_bytes(const VerifyParams& p, bool dense);
constexpr size_t kFinCacheLimit = 48 * 1024;
// Filter kernel: one CTA per row, rows of at most this many bytes.
constexpr int kFilterRowBytes = 512 * 1024;
constexpr size_t kFinSmemMax = kFinCacheLimit + sizeof(float) * ((1 << 24) / kChunk);  // V <= 2^24

// mode: 0 one-hot sampling, 1 dense sampling, 2 greedy, 3 typical acceptance
// (4, tree sampling, runs through launch_tree_sample)
cudaError_t launch_verify(int mode, int dtype, bool vec, const VerifyParams& p,
                          cudaStream_t stream);
cudaError_t launch_tree(int dtype, bool vec, const TreeParams& p, cudaStream_t stream);
// Kernel A of top-k / top-p calls (sv_filter.cu); mode 0 or 1.
// Kernel A (or A' for filtered calls) alone: the chunk records.
cudaError_t launch_records(int mode, int dtype, bool vec, const VerifyParams& p,
                           cudaStream_t stream);
cudaError_t launch_filter(int mode, int dtype, bool vec, const VerifyParams& p,
                          cudaStream_t stream);
cudaError_t launch_tree_typical(int dtype, bool vec, const VerifyParams& p, const TreeCall& t,
                                cudaStream_t stream);
cudaError_t launch_tree_sample(int dtype, bool vec, const VerifyParams& p, const TreeCall& t,
                               cudaStream_t stream);

// The limit of the kernels' waits for staged logits (set through the C ABI).
unsigned long long wait_limit_ns();

}  // namespace sv
