// sv_ngram.cu - the n-gram (prompt-lookup) proposer.
//
// The deterministic proposer whose one-hot drafts spec_verify_sample checks
// ("投机解码" (FastDeploy docs), "使用 Ngram 解码": drafts come from matching an
// n-gram window against the prompt and the tokens generated so far; the vLLM
// Ascend guide's n-gram example: prompt_lookup_max = 4, 5 speculative
// tokens).  For n = n_max down to n_min the last n tokens of a request's
// context are looked up earlier in the context; the earliest occurrence
// followed by at least one token gives the drafts, the up to K tokens after
// it.  The longest n that occurs wins.
//
// One CTA per request makes a single pass over the context for all n at
// once.  For every end position e <= len - 2 it measures lcs(e), the length
// of the common suffix of c[0..e] and the whole context, capped at n_max: a
// start s = e - n + 1 matches the n-gram exactly when lcs(e) >= n.  The
// smallest matching start per n is kept with shared-memory atomicMin, and
// the largest n with a match decides.  Each thread first reads the last
// token of its candidate ends (coalesced, kEnds ends per thread in flight);
// only ends that match it compare further.  The pass stops early once the
// longest n-gram has matched.
#include <climits>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kNgramThreads = 256;
constexpr int kEnds = 8;  // candidate ends per thread per pass

struct NgramParams {
  const int* tokens;  // [B, L]
  const int* lens;    // [B]
  int* drafts;        // [B, K]
  int* draft_lens;    // [B]
  int* match;         // [B] or null
  int* status;        // [B] or null
  int B, L, n_min, n_max, K;
};

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(const NgramParams p) {
  __shared__ int s_tail[SV_MAX_NGRAM];      // c[len - 1 - t]
  __shared__ int s_best[SV_MAX_NGRAM + 1];  // smallest matching start per n
  __shared__ int s_pick[2];
  const int b = blockIdx.x;
  const int* c = p.tokens + (long long)b * p.L;
  const int len = __ldg(p.lens + b);
  const bool ok = len >= 0 && len <= p.L;
  if (threadIdx.x <= SV_MAX_NGRAM) s_best[threadIdx.x] = INT_MAX;
  if (ok && threadIdx.x < p.n_max && threadIdx.x < len)
    s_tail[threadIdx.x] = __ldg(c + len - 1 - threadIdx.x);
  __syncthreads();
  if (ok && len >= p.n_min + 1) {
    const int last = s_tail[0];
    // ends e in [n_min - 1, len - 2]
    for (int e0 = p.n_min - 1; e0 <= len - 2; e0 += kNgramThreads * kEnds) {
      int v[kEnds];
#pragma unroll
      for (int j = 0; j < kEnds; ++j) {
        const int e = e0 + j * kNgramThreads + threadIdx.x;
        v[j] = e <= len - 2 ? __ldg(c + e) : 0;
      }
#pragma unroll
      for (int j = 0; j < kEnds; ++j) {
        const int e = e0 + j * kNgramThreads + threadIdx.x;
        if (e > len - 2 || v[j] != last) continue;
        int l = 1;  // lcs(e), capped at n_max and at e + 1 (the start stays >= 0)
        while (l < p.n_max && l <= e && __ldg(c + e - l) == s_tail[l]) ++l;
        for (int n = p.n_min; n <= l; ++n)
          if (e - n + 1 < s_best[n]) atomicMin(&s_best[n], e - n + 1);
      }
      // Ends are visited in increasing order, so once the longest n-gram has
      // a match no later end can give it an earlier start.  (A thread that
      // made the match sees its own write, so the OR is the same for all.)
      if (__syncthreads_or(s_best[p.n_max] != INT_MAX)) break;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n_hit = 0, start = -1;
    for (int n = p.n_max; n >= p.n_min && ok; --n)
      if (s_best[n] != INT_MAX) {
        n_hit = n;
        start = s_best[n];
        break;
      }
    s_pick[0] = n_hit;
    s_pick[1] = start;
    if (p.match) p.match[b] = start;
    if (p.status) p.status[b] = ok ? 0 : SV_REQ_BAD_DRAFT_LEN;
    int k = start >= 0 ? len - (start + n_hit) : 0;
    p.draft_lens[b] = k < p.K ? k : p.K;
  }
  __syncthreads();
  const int n_hit = s_pick[0], start = s_pick[1];
  for (int t = threadIdx.x; t < p.K; t += kNgramThreads) {
    const int pos = start + n_hit + t;
    p.drafts[(long long)b * p.K + t] = (start >= 0 && pos < len) ? __ldg(c + pos) : -1;
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_ngram_propose(const int32_t* tokens, const int32_t* lens, int B, int L,
                                        int n_min, int n_max, int K, int32_t* out_drafts,
                                        int32_t* out_draft_lens, int32_t* out_match,
                                        int32_t* out_status, sv_stream_t stream) {
  if (B < 0 || B > SV_MAX_B || L < 0 || K < 0 || K > SV_MAX_K || n_min < 1 || n_max < n_min ||
      n_max > SV_MAX_NGRAM || (long long)B * L >= (1LL << 31))
    return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!lens || !out_draft_lens || (K > 0 && !out_drafts) || (L > 0 && !tokens)) return SV_ERR_NULL;
  NgramParams p;
  p.tokens = tokens;
  p.lens = lens;
  p.drafts = out_drafts;
  p.draft_lens = out_draft_lens;
  p.match = out_match;
  p.status = out_status;
  p.B = B;
  p.L = L;
  p.n_min = n_min;
  p.n_max = n_max;
  p.K = K;
  ngram_kernel<<<B, kNgramThreads, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
