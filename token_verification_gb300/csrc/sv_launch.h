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
};

// A request whose dense-draft residual still has to be drawn.
struct ReqState {
  int n;        // rejected position
  int pending;  // 1 while the residual kernel owes this request its outputs
  float mp, ip; // target row n: max and 1 / sum
  float mq, iq; // draft row n: max and 1 / sum
  int pad0, pad1;
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
  // workspace
  int* res_ticket;   // [B]
  int* err;          // [1] set when a bounded wait gave up
  int* fin_ticket;   // [1] requests finalised in this call
  ReqState* state;   // [B]
  float2* rec;       // [B*R*NC]
  float* lx;         // [B*R] the logit of each row's draft token
  float* res_rec;    // [B*NC]
  int B, K, V;
  int NC;            // chunks per row
  int R;             // rows per request: K+1 target (+ K draft rows when dense)
  int TPR;           // stream items per row
  int item_chunks;   // chunks per stream item
  int TPR_res;       // residual tasks per row pair
  long long total_tasks;  // < 2^31 (checked on the host)
  FastDiv div_tpr, div_r; // divide by TPR and by R
  float cc;          // log2(e) / T
  int greedy_prob;   // greedy rule reached through the sampling entry
  int compact_in_finalize;  // the finalize kernel writes the packed output
  int fin_cache;     // the finalize kernel keeps the request's records in shared memory
};

constexpr int kMaxTreeNodes = 256;

struct TreeParams {
  const void* target;
  const int* tokens;  // [B, N]
  int* out_tokens;
  int* out_accept_len;
  int* out_path;
  int* out_status;
  int B, N, V, D1, NC;
  short first_child[kMaxTreeNodes + 1];  // 0 = none
  short next_sibling[kMaxTreeNodes + 1];
};

enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Workspace layout for B requests, K positions, V vocabulary (dense case).
struct WorkspaceLayout {
  size_t res_ticket, counters, state, zero_bytes, rec, lx, res_rec, total;
};
WorkspaceLayout workspace_layout(int B, int K, int V);

struct DeviceInfo {
  int sms;
};
cudaError_t device_info(DeviceInfo* out);

// Chunks per stream item (row-statistics kernel) and per residual task.
int chunks_per_task(int dtype, bool vec);
// Shared memory the finalize kernel uses to keep a request's chunk records.
size_t fin_cache_bytes(const VerifyParams& p);
constexpr size_t kFinCacheLimit = 48 * 1024;  // without the large-shared-memory opt-in
int residual_chunks_per_task(int dtype, bool vec);

// mode: 0 one-hot sampling, 1 dense sampling, 2 greedy
cudaError_t launch_verify(int mode, int dtype, bool vec, const VerifyParams& p, bool compact,
                          cudaStream_t stream);
cudaError_t launch_tree(int dtype, bool vec, const TreeParams& p, cudaStream_t stream);

}  // namespace sv
