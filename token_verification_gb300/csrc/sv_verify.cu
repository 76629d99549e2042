// sv_verify.cu - rejection-sampling and greedy verification kernels.
//
// Method ("【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §2.1 "算法骨架"):
// for each request, accept draft x_i with probability min(1, p_i(x_i) /
// q_i(x_i)) in position order; at the first rejection n draw from
// norm(max(0, p_n - q_n)); if all drafts are accepted draw the extra token
// from the last position's p.  Greedy rule (§11 of the same page): accept
// while x_i equals the target argmax.  Requests are independent and verified
// in parallel ("投机解码" (FastDeploy), "高效投机解码框架设计").
//
// Kernel A (verify_rows_kernel, persistent): every warp streams tasks of up
//   to G chunks of one logit row and writes one record per chunk.  Each logit
//   is read once.  The warp that completes a row (atomic ticket per row)
//   combines its records into a RowSum; the warp that completes a request's
//   last row (ticket per request) runs the acceptance tests for all positions
//   at once (one lane per position), then draws the residual / bonus token:
//   it locates the chunk from the records and rescans that single chunk.
//   No warp ever waits for another: whoever arrives last does the work.
// Kernel B (residual_kernel, dense drafts only): for each request rejected at
//   n, sums max(0, p_n - q_n) per chunk of the (target, draft) row pair, and
//   the last warp of the request draws the token the same way.
// Kernel C (compact_kernel): exclusive scan of accept_len and the packed,
//   padding-free output with per-token batch ids.
// B and C start with programmatic dependent launch and wait for their
// predecessor's results on the device.
#include "sv_common.cuh"
#include "sv_launch.h"

namespace sv {
namespace {

template <typename T>
__device__ __forceinline__ const T* row_ptr(const void* base, long long row, int V) {
  return reinterpret_cast<const T*>(base) + row * (long long)V;
}

__device__ __forceinline__ RowSum load_rowsum(const RowSum* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  RowSum r;
  r.m = __int_as_float(v.x);
  r.s = __int_as_float(v.y);
  r.wx = __int_as_float(v.z);
  r.idx = v.w;
  return r;
}

__device__ __forceinline__ void store_rowsum(RowSum* p, const RowSum& r) {
  *reinterpret_cast<int4*>(p) =
      make_int4(__float_as_int(r.m), __float_as_int(r.s), __float_as_int(r.wx), r.idx);
}

__device__ __forceinline__ ReqState load_state(const ReqState* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  ReqState s;
  s.n = a.x;
  s.pending = a.y;
  s.mp = __int_as_float(a.z);
  s.ip = __int_as_float(a.w);
  s.mq = __int_as_float(b.x);
  s.iq = __int_as_float(b.y);
  s.pad0 = s.pad1 = 0;
  return s;
}

// ---------------------------------------------------------------------------
// drawing one token
// ---------------------------------------------------------------------------

// First chunk c whose cumulative weight exceeds `target` (chunk weights from
// `weight(c)`, all in one frame).  Returns c and the fraction of chunk c's
// weight that lies below the target; if rounding leaves the target past the
// last chunk, returns the last chunk of positive weight with fraction 2
// (which selects its last positive element).  c = -1 if no weight at all.
template <class F>
__device__ int find_chunk(F weight, int NC, float target, float* frac) {
  const int lane = lane_id();
  float base = 0.f;
  for (int c0 = 0; c0 < NC; c0 += kWarp) {
    const int c = c0 + lane;
    const float w = c < NC ? weight(c) : 0.f;
    const float incl = warp_incl_scan(w);
    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && base + incl > target);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const float below = target - (base + __shfl_sync(0xffffffffu, incl - w, l));
      const float wl = __shfl_sync(0xffffffffu, w, l);
      *frac = fminf(fmaxf(below / wl, 0.f), 1.f);
      return c0 + l;
    }
    base += __shfl_sync(0xffffffffu, incl, kWarp - 1);
  }
  for (int c0 = ((NC - 1) / kWarp) * kWarp; c0 >= 0; c0 -= kWarp) {
    const int c = c0 + lane;
    const unsigned pos = __ballot_sync(0xffffffffu, c < NC && weight(c) > 0.f);
    if (pos) {
      *frac = 2.f;
      return c0 + 31 - __clz(pos);
    }
  }
  return -1;
}

// Smallest element whose cumulative weight (in index order) exceeds
// frac * (tile total), over one chunk tile of weights w held per lane
// (group k, element e at chunk offset k*32*VEC + lane*VEC + e); zero
// weights are never chosen.  Falls back to the last positive element.
template <int NV, int VEC>
__device__ int select_in_tile(const float (&w)[NV * VEC], const float (&gsum)[NV], float frac,
                              int base_j) {
  const int lane = lane_id();
  float lt = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) lt += gsum[k];
  const float thr = frac * warp_sum(lt);
  float running = 0.f;
  int tok = -1;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const float incl = warp_incl_scan(gsum[k]);
    const unsigned hit = __ballot_sync(0xffffffffu, gsum[k] > 0.f && running + incl > thr);
    if (hit && tok < 0) {
      const int l = __ffs(hit) - 1;
      int t = -1;
      if (lane == l) {
        float acc = running + incl - gsum[k];
        int last = -1;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float we = w[k * VEC + e];
          acc += we;
          if (we > 0.f) {
            last = base_j + tile_offset<VEC>(k, e, lane);
            if (t < 0 && acc > thr) t = last;
          }
        }
        if (t < 0) t = last;
      }
      tok = __shfl_sync(0xffffffffu, t, l);
    }
    running += __shfl_sync(0xffffffffu, incl, kWarp - 1);
  }
  if (tok < 0) {
    int last = -1;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if (w[k * VEC + e] > 0.f) last = base_j + tile_offset<VEC>(k, e, lane);
    tok = __reduce_max_sync(0xffffffffu, last);
  }
  return tok;
}

// Draw from w_j = 2^((l_j - m) c) over one row (w = 0 at mask_x) given the
// row's softmax chunk records: the crossing chunk from the records, then one
// rescan of that chunk in its own frame.
template <typename T, int VEC>
__device__ int draw_from_records(const T* row, const float2* rec, int NC, int V, float m, float cc,
                                 float u, int mask_x) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  const float nb = -m * cc;
  auto weight = [&](int c) {
    const float2 r = __ldcg(rec + c);
    return r.y * ex2(fmaf(r.x, cc, nb));
  };
  float tot = 0.f;
  for (int c = lane; c < NC; c += kWarp) tot += weight(c);
  tot = warp_sum(tot);
  float frac = 0.f;
  const int c = find_chunk(weight, NC, u * tot, &frac);
  if (c < 0) return -1;
  typename L::Raw raw[L::NV];
  load_chunk<T, VEC>(row, V, c, raw);
  const float nbc = -__ldcg(rec + c).x * cc;
  float w[L::NV * VEC];
  float gsum[L::NV];
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    gsum[k] = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float we = ex2(fmaf(L::get(raw[k], e), cc, nbc));
      if (c * kChunk + tile_offset<VEC>(k, e, lane) == mask_x) we = 0.f;
      w[k * VEC + e] = we;
      gsum[k] += we;
    }
  }
  return select_in_tile<L::NV, VEC>(w, gsum, frac, c * kChunk);
}

// Residual weight max(0, p_j - q_j) from the two rows' maxima and 1/sums.
__device__ __forceinline__ float residual_weight(float lt, float ld, float cc, float nbp, float ip,
                                                 float nbq, float iq) {
  const float r = ex2(fmaf(lt, cc, nbp)) * ip - ex2(fmaf(ld, cc, nbq)) * iq;
  return r > 0.f ? r : 0.f;
}

__device__ __forceinline__ void write_request(const VerifyParams& p, int b, int status, int n,
                                              int token, int x) {
  const int lane = lane_id();
  const int K = p.K;
  if (lane <= K)
    p.out_tokens[(long long)b * (K + 1) + lane] =
        status ? -1 : (lane < n ? x : (lane == n ? token : -1));
  if (lane == 0) {
    p.out_accept_len[b] = status ? 0 : n + 1;
    if (p.out_status) p.out_status[b] = status;
  }
}

// ---------------------------------------------------------------------------
// request / row finalisation (run by the last-arriving warp)
// ---------------------------------------------------------------------------

template <int MODE, typename T, int VEC>
__device__ __noinline__ void request_finalize(const VerifyParams& p, int b, int Kb) {
  const int lane = lane_id();
  const int K = p.K;
  // A bounded wait that gave up earlier in this call marks every request
  // finalised after it (its chunks may be among the unread ones).
  int status = 0;
  if (lane == 0) {
    p.req_ticket[b] = 0;
    if (__ldcg(p.err)) status = kTimeout;
  }
  status = __shfl_sync(0xffffffffu, status, 0);
  if (Kb < 0 || Kb > K) {
    status |= kBadDraftLen;
    Kb = 0;
  }
  int x = -1;
  if (lane < Kb) x = __ldg(p.draft_tokens + (long long)b * K + lane);
  if (!status && __any_sync(0xffffffffu, lane < Kb && (x < 0 || x >= p.V))) status = kBadToken;
  int n = 0, token = -1;
  float theta = -1.f;
  bool pending = false;
  if (!status) {
    const long long rb = (long long)b * p.R;
    RowSum rt{qnan(), 0.f, 0.f, -1}, rd{qnan(), 0.f, 0.f, -1};
    if (lane <= Kb) rt = load_rowsum(p.row_sum + rb + lane);
    if (MODE == kDense && lane < Kb) rd = load_rowsum(p.row_sum + rb + K + 1 + lane);
    bool bad = lane <= Kb && !is_finite(rt.m);
    if (MODE == kDense && lane < Kb) bad = bad || !is_finite(rd.m);
    bool acc = false;
    if (lane < Kb) {
      if (MODE == kGreedy) {
        acc = (x == rt.idx);
        theta = acc ? 1.f : 0.f;
      } else {
        const float u = __ldg(p.uniforms + (long long)b * (K + 1) + lane);
        if (MODE == kOneHot) {  // q = point mass at x: accept iff u < p(x)
          const float px = rt.wx / (rt.s + rt.wx);
          theta = fminf(1.f, px);
          acc = u < px;
        } else {  // accept iff u * q(x) < p(x)
          const float px = rt.wx / rt.s, qx = rd.wx / rd.s;
          theta = qx > 0.f ? fminf(1.f, px / qx) : (px > 0.f ? 1.f : 0.f);
          acc = u * qx < px;
        }
      }
    }
    const unsigned stop = __ballot_sync(0xffffffffu, lane < Kb && (bad || !acc));
    n = stop ? __ffs(stop) - 1 : Kb;
    if (__shfl_sync(0xffffffffu, bad ? 1 : 0, n)) status = kBadLogits;
    const float m_n = __shfl_sync(0xffffffffu, rt.m, n);
    const float s_n = __shfl_sync(0xffffffffu, rt.s, n);
    const int idx_n = __shfl_sync(0xffffffffu, rt.idx, n);
    const int x_n = __shfl_sync(0xffffffffu, x, n);
    const float mq_n = __shfl_sync(0xffffffffu, rd.m, n);
    const float sq_n = __shfl_sync(0xffffffffu, rd.s, n);
    if (!status) {
      if (MODE == kGreedy) {
        token = idx_n;
      } else if (MODE == kDense && n < Kb) {
        pending = true;  // the residual kernel draws from max(0, p_n - q_n)
        if (lane == 0) {
          ReqState st;
          st.n = n;
          st.pending = 1;
          st.mp = m_n;
          st.ip = 1.f / s_n;
          st.mq = mq_n;
          st.iq = 1.f / sq_n;
          st.pad0 = st.pad1 = 0;
          p.state[b] = st;
        }
      } else {
        const float uK = __ldg(p.uniforms + (long long)b * (K + 1) + K);
        const bool residual = MODE == kOneHot && n < Kb;
        if (residual && !(s_n > 0.f)) {
          token = x_n;  // no mass left beside x_n: p_n itself is the point mass at x_n
        } else {
          const T* row = row_ptr<T>(p.target, (long long)b * (K + 1) + n, p.V);
          token = draw_from_records<T, VEC>(row, p.rec + (rb + n) * p.NC, p.NC, p.V, m_n, p.cc,
                                            uK, residual ? x_n : -1);
          if (token < 0) status = kBadLogits;
        }
      }
    }
  }
  // the last request finalised in this call clears the call's counters
  if (lane == 0 && atomic_add_acq_rel(p.fin_ticket, 1) + 1 == p.B) {
    *p.err = 0;
    *p.fin_ticket = 0;
  }
  if (p.out_accept_prob && lane < K && (MODE != kGreedy || p.greedy_prob))
    p.out_accept_prob[(long long)b * K + lane] =
        (!status && lane < Kb && lane <= n) ? theta : -1.f;
  if (!pending) write_request(p, b, status, n, token, x);
}

template <int MODE, typename T, int VEC>
__device__ __noinline__ void row_finalize(const VerifyParams& p, int b, int r, long long rowid,
                                          bool need, int Kb) {
  const int lane = lane_id();
  RowSum rs{qnan(), 0.f, 0.f, -1};
  if (need) {
    const float2* rec = p.rec + rowid * p.NC;
    if (MODE == kGreedy) {
      const float2 a = combine_argmax_records(rec, p.NC);
      rs.m = a.x;
      rs.idx = __float_as_int(a.y);
    } else {
      const bool is_draft = r > p.K;
      const int i = is_draft ? r - p.K - 1 : r;
      const int x = i < Kb ? __ldg(p.draft_tokens + (long long)b * p.K + i) : -1;
      const bool has_x = x >= 0 && x < p.V;
      float lx = 0.f;
      if (has_x) {
        const T* row = is_draft ? row_ptr<T>(p.draft, (long long)b * p.K + i, p.V)
                                : row_ptr<T>(p.target, (long long)b * (p.K + 1) + i, p.V);
        lx = load_logit(row, x);
      }
      const float2 ms = combine_softmax_records(rec, p.NC, p.cc);
      rs.m = ms.x;
      rs.s = ms.y;
      if (has_x && is_finite(ms.x)) rs.wx = ex2(fmaf(lx, p.cc, -ms.x * p.cc));
    }
  }
  int old = 0;
  if (lane == 0) {
    store_rowsum(p.row_sum + rowid, rs);
    p.row_ticket[rowid] = 0;
    old = atomic_add_acq_rel(p.req_ticket + b, 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old + 1 == p.R) request_finalize<MODE, T, VEC>(p, b, Kb);
}

// ---------------------------------------------------------------------------
// kernel A: row statistics + finalisation
// ---------------------------------------------------------------------------

// A task is up to G consecutive chunks of one row.  Tasks are numbered
// request-major (request, row, chunk group), so requests complete one after
// another while the grid streams.
struct Task {
  long long rowid;
  int b, r, i, Kb, c0, nch;
  bool is_draft, need;
};

template <int G>
__device__ __forceinline__ Task decode_task(const VerifyParams& p, long long t) {
  Task k;
  k.rowid = t / p.TPR;
  const int tc = (int)(t % p.TPR);
  k.r = (int)(k.rowid % p.R);
  k.b = (int)(k.rowid / p.R);
  k.Kb = p.draft_lens ? __ldg(p.draft_lens + k.b) : p.K;
  k.is_draft = k.r > p.K;
  k.i = k.is_draft ? k.r - p.K - 1 : k.r;
  k.need = k.Kb >= 0 && k.Kb <= p.K && (k.is_draft ? k.i < k.Kb : k.i <= k.Kb);
  k.c0 = tc * G;
  k.nch = min(G, p.NC - k.c0);
  return k;
}

template <typename T>
__device__ __forceinline__ const T* task_row(const VerifyParams& p, const Task& k) {
  return k.is_draft ? row_ptr<T>(p.draft, (long long)k.b * p.K + k.i, p.V)
                    : row_ptr<T>(p.target, (long long)k.b * (p.K + 1) + k.i, p.V);
}

// The one-hot draft token of this task's row (excluded from its sums), or -1.
template <int MODE>
__device__ __forceinline__ int task_mask(const VerifyParams& p, const Task& k) {
  if (MODE != kOneHot || k.is_draft || k.i >= k.Kb) return -1;
  return __ldg(p.draft_tokens + (long long)k.b * p.K + k.i);
}

template <int MODE, typename T, int VEC>
__device__ __forceinline__ float2 chunk_record(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                               int c, float cc, int mask_x) {
  if (MODE == kGreedy) return chunk_argmax<T, VEC>(raw, c * kChunk);
  const int ml = (mask_x >= c * kChunk && mask_x < (c + 1) * kChunk) ? mask_x - c * kChunk : -1;
  return chunk_softmax<T, VEC>(raw, cc, ml);
}

// A task's arrival on its row's counter is issued at the end of the task and
// its result read only at the end of the next one, so the atomic's round trip
// overlaps work; the warp that completes the row finalises it.
template <int MODE, typename T, int VEC>
__device__ __forceinline__ void settle_task(const VerifyParams& p, const Task& k, int old_lane0) {
  const int old = __shfl_sync(0xffffffffu, old_lane0, 0);
  if (old + k.nch == p.NC) row_finalize<MODE, T, VEC>(p, k.b, k.r, k.rowid, k.need, k.Kb);
}

// Register-tile variant: the scalar path (any V, any alignment).
template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kThreads, 2) verify_rows_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  constexpr int G = L::G;
  pdl_launch_dependents();
  const int lane = lane_id();
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  bool have_prev = false;
  Task prev{};
  int prev_old = 0;
  for (long long t = gw; t < p.total_tasks; t += nw) {
    const Task k = decode_task<G>(p, t);
    if (k.need) {
      const T* row = task_row<T>(p, k);
      typename L::Raw raw[G][L::NV];
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < k.nch) load_chunk<T, VEC>(row, p.V, k.c0 + g, raw[g]);
      const int mask_x = task_mask<MODE>(p, k);
      float2* rec = p.rec + k.rowid * p.NC;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < k.nch) {
          const float2 out = chunk_record<MODE, T, VEC>(raw[g], k.c0 + g, p.cc, mask_x);
          if (lane == 0) rec[k.c0 + g] = out;
        }
    }
    int old = 0;
    if (lane == 0) old = atomic_add_acq_rel(p.row_ticket + k.rowid, k.nch);
    if (have_prev) settle_task<MODE, T, VEC>(p, prev, prev_old);
    prev = k;
    prev_old = old;
    have_prev = true;
  }
  if (have_prev) settle_task<MODE, T, VEC>(p, prev, prev_old);
}

// Shared-memory ring of the bulk-copy variant (vector paths): each warp owns
// kStages chunk buffers, each with an mbarrier.  Lane 0 keeps the next chunks
// of the warp's task sequence in flight with cp.async.bulk while the warp
// reduces the oldest one, so the bytes in flight do not depend on registers.
template <typename T>
struct Ring {
  static constexpr int kChunkBytes = kChunk * (int)sizeof(T);
  static constexpr int kStages = sizeof(T) == 2 ? 6 : 3;
  static constexpr int kWarpBytes = kStages * kChunkBytes;
  static constexpr int kBulkG = 8;  // chunks per task
  static constexpr int smem_bytes() { return (kThreads / kWarp) * (kWarpBytes + kStages * 8); }
};

template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kThreads) verify_rows_bulk_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  using RG = Ring<T>;
  constexpr int S = RG::kStages;
  constexpr int G = RG::kBulkG;
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t ring = smem_u32(smem) + warp * RG::kWarpBytes;
  const uint32_t bars = smem_u32(smem) + (kThreads / kWarp) * RG::kWarpBytes + warp * S * 8;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;

  // producer state (lane 0): the next chunk of the warp's task sequence
  long long pt = gw;
  int pg = 0;
  Task ptask{};
  bool pdone = true;
  uint32_t issued = 0;
  auto skip_empty = [&]() {
    while (!pdone && (!ptask.need || pg >= ptask.nch)) {
      pt += nw;
      pg = 0;
      if (pt >= p.total_tasks) {
        pdone = true;
        break;
      }
      ptask = decode_task<G>(p, pt);
    }
  };
  auto issue_next = [&]() {
    if (pdone) return;
    const int c = ptask.c0 + pg;
    const T* src = task_row<T>(p, ptask) + (long long)c * kChunk;
    const uint32_t bytes = (uint32_t)(min(kChunk, p.V - c * kChunk) * (int)sizeof(T));
    const int stage = (int)(issued % S);
    bulk_load(ring + stage * RG::kChunkBytes, src, bytes, bars + 8 * stage);
    ++issued;
    ++pg;
    skip_empty();
  };
  if (lane == 0 && pt < p.total_tasks) {
    pdone = false;
    ptask = decode_task<G>(p, pt);
    skip_empty();
    for (int s = 0; s < S; ++s) issue_next();
  }

  uint32_t consumed = 0;  // chunks whose copy landed and was reduced
  bool failed = false;
  bool have_prev = false;
  Task prev{};
  int prev_old = 0;
  for (long long t = gw; t < p.total_tasks; t += nw) {
    const Task k = decode_task<G>(p, t);
    if (k.need) {
      const int mask_x = task_mask<MODE>(p, k);
      float2* rec = p.rec + k.rowid * p.NC;
      for (int g = 0; g < k.nch; ++g) {
        const int c = k.c0 + g;
        const int stage = (int)(consumed % S);
        bool ok = !failed && mbar_wait(bars + 8 * stage, (consumed / S) & 1u);
        ok = __all_sync(0xffffffffu, ok);
        float2 out = make_float2(qnan(), 0.f);
        if (ok) {
          typename L::Raw raw[L::NV];
          load_chunk_smem<T, VEC>(ring + stage * RG::kChunkBytes, p.V, c, raw);
          out = chunk_record<MODE, T, VEC>(raw, c, p.cc, mask_x);
          ++consumed;
        } else if (!failed) {
          // a copy did not land in time: issue no more copies; this and the
          // warp's remaining chunks are recorded as unusable
          failed = true;
          if (lane == 0) atomicOr(p.err, 1);
        }
        __syncwarp();
        if (lane == 0) {
          rec[c] = out;
          if (!failed) {
            fence_proxy_async();
            issue_next();
          }
        }
      }
    }
    int old = 0;
    if (lane == 0) old = atomic_add_acq_rel(p.row_ticket + k.rowid, k.nch);
    if (have_prev) settle_task<MODE, T, VEC>(p, prev, prev_old);
    prev = k;
    prev_old = old;
    have_prev = true;
  }
  if (have_prev) settle_task<MODE, T, VEC>(p, prev, prev_old);
  if (failed && lane == 0) {  // let copies still in flight land before the CTA exits
    for (uint32_t j = consumed; j < issued; ++j) mbar_wait(bars + 8 * (j % S), (j / S) & 1u);
  }
}

// ---------------------------------------------------------------------------
// kernel B: dense-draft residual
// ---------------------------------------------------------------------------

template <typename T, int VEC>
__device__ __noinline__ void residual_finalize(const VerifyParams& p, int b, const ReqState& st) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  const int K = p.K;
  const float cc = p.cc;
  const float uK = __ldg(p.uniforms + (long long)b * (K + 1) + K);
  const T* tr = row_ptr<T>(p.target, (long long)b * (K + 1) + st.n, p.V);
  const T* dr = row_ptr<T>(p.draft, (long long)b * K + st.n, p.V);
  const float* rr = p.res_rec + (long long)b * p.NC;
  auto weight = [&](int c) { return __ldcg(rr + c); };
  float tot = 0.f;
  for (int c = lane; c < p.NC; c += kWarp) tot += weight(c);
  tot = warp_sum(tot);
  int token;
  if (!(tot > 0.f)) {  // no residual mass (rounding only): draw from p_n
    token = draw_from_records<T, VEC>(tr, p.rec + ((long long)b * p.R + st.n) * p.NC, p.NC, p.V,
                                      st.mp, cc, uK, -1);
  } else {
    float frac = 0.f;
    const int c = find_chunk(weight, p.NC, uK * tot, &frac);
    typename L::Raw rt[L::NV], rd[L::NV];
    load_chunk<T, VEC>(tr, p.V, c, rt);
    load_chunk<T, VEC>(dr, p.V, c, rd);
    const float nbp = -st.mp * cc, nbq = -st.mq * cc;
    float w[L::NV * VEC];
    float gsum[L::NV];
#pragma unroll
    for (int k = 0; k < L::NV; ++k) {
      gsum[k] = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float we = residual_weight(L::get(rt[k], e), L::get(rd[k], e), cc, nbp, st.ip, nbq,
                                         st.iq);
        w[k * VEC + e] = we;
        gsum[k] += we;
      }
    }
    token = select_in_tile<L::NV, VEC>(w, gsum, frac, c * kChunk);
  }
  const int x = lane < st.n ? __ldg(p.draft_tokens + (long long)b * K + lane) : -1;
  write_request(p, b, token < 0 ? kBadLogits : 0, st.n, token, x);
  if (lane == 0) {
    p.res_ticket[b] = 0;
    p.state[b].pending = 0;
  }
}

template <typename T, int VEC>
__host__ __device__ constexpr int residual_group() {
  return Lane<T, VEC>::G > 1 ? Lane<T, VEC>::G / 2 : 1;
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads, 2) residual_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  constexpr int G = residual_group<T, VEC>();
  pdl_wait();
  pdl_launch_dependents();
  const int lane = lane_id();
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long total = (long long)p.B * p.TPR_res;
  const float cc = p.cc;
  for (long long t = gw; t < total; t += nw) {
    const int b = (int)(t / p.TPR_res);
    const int tc = (int)(t % p.TPR_res);
    const ReqState st = load_state(p.state + b);
    if (!st.pending || st.n < 0 || st.n >= p.K) continue;
    const T* tr = row_ptr<T>(p.target, (long long)b * (p.K + 1) + st.n, p.V);
    const T* dr = row_ptr<T>(p.draft, (long long)b * p.K + st.n, p.V);
    const int c0 = tc * G;
    const int nch = min(G, p.NC - c0);
    typename L::Raw rt[G][L::NV], rd[G][L::NV];
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (g < nch) {
        load_chunk<T, VEC>(tr, p.V, c0 + g, rt[g]);
        load_chunk<T, VEC>(dr, p.V, c0 + g, rd[g]);
      }
    const float nbp = -st.mp * cc, nbq = -st.mq * cc;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g < nch) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < L::NV; ++k)
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            s += residual_weight(L::get(rt[g][k], e), L::get(rd[g][k], e), cc, nbp, st.ip, nbq,
                                 st.iq);
        s = warp_sum(s);
        if (lane == 0) p.res_rec[(long long)b * p.NC + c0 + g] = s;
      }
    }
    int old = 0;
    if (lane == 0) old = atomic_add_acq_rel(p.res_ticket + b, nch);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + nch == p.NC) residual_finalize<T, VEC>(p, b, st);
  }
}

// ---------------------------------------------------------------------------
// kernel C: padding-free packed output
// ---------------------------------------------------------------------------

__device__ int block_sum(int v, int* smem) {
  const int lane = lane_id(), warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) smem[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < nwarps; ++w) t += smem[w];
  return t;
}

__device__ int block_excl_scan(int v, int* smem) {
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan_int(v);
  __syncthreads();
  if (lane == kWarp - 1) smem[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += smem[w];
  return before + incl - v;
}

__global__ void compact_kernel(const VerifyParams p) {
  __shared__ int smem[32];
  pdl_wait();
  const int B = p.B, W = p.K + 1;
  const int b0 = blockIdx.x * blockDim.x;
  int before = 0, all = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int L = __ldcg(p.out_accept_len + b);
    all += L;
    if (b < b0) before += L;
  }
  before = block_sum(before, smem);
  all = block_sum(all, smem);
  const int b = b0 + threadIdx.x;
  const int L = b < B ? __ldcg(p.out_accept_len + b) : 0;
  const int cu = before + block_excl_scan(L, smem);
  if (b < B) {
    if (p.out_cu) p.out_cu[b] = cu;
    for (int k = 0; k < L; ++k) {
      if (p.out_packed) p.out_packed[cu + k] = __ldcg(p.out_tokens + (long long)b * W + k);
      if (p.out_batch_id) p.out_batch_id[cu + k] = b;
    }
  }
  if (p.out_cu && blockIdx.x == 0 && threadIdx.x == 0) p.out_cu[B] = all;
  const long long cap = (long long)B * W;
  for (long long s = all + (long long)blockIdx.x * blockDim.x + threadIdx.x; s < cap;
       s += (long long)gridDim.x * blockDim.x) {
    if (p.out_packed) p.out_packed[s] = -1;
    if (p.out_batch_id) p.out_batch_id[s] = -1;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <class K>
int blocks_per_sm(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int MODE, typename T, int VEC>
cudaError_t launch_typed(const VerifyParams& p, bool compact, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const int warps_per_cta = kThreads / kWarp;
  if constexpr (VEC * sizeof(T) == 16) {
    constexpr int smem = Ring<T>::smem_bytes();
    static int occ = 0;
    if (!occ) {
      err = cudaFuncSetAttribute(verify_rows_bulk_kernel<MODE, T, VEC>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
              &occ, verify_rows_bulk_kernel<MODE, T, VEC>, kThreads, smem) != cudaSuccess ||
          occ < 1)
        occ = 1;
    }
    const long long want = (p.total_tasks + warps_per_cta - 1) / warps_per_cta;
    const long long cap = (long long)di.sms * occ;
    const int grid = (int)(want < cap ? want : cap);
    verify_rows_bulk_kernel<MODE, T, VEC><<<grid, kThreads, smem, s>>>(p);
  } else {
    static int occ = 0;
    if (!occ) occ = blocks_per_sm(verify_rows_kernel<MODE, T, VEC>);
    const long long want = (p.total_tasks + warps_per_cta - 1) / warps_per_cta;
    const long long cap = (long long)di.sms * occ;
    const int grid = (int)(want < cap ? want : cap);
    verify_rows_kernel<MODE, T, VEC><<<grid, kThreads, 0, s>>>(p);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (MODE == kDense) {
    static int occ = 0;
    if (!occ) occ = blocks_per_sm(residual_kernel<T, VEC>);
    const long long want = ((long long)p.B * p.TPR_res + warps_per_cta - 1) / warps_per_cta;
    const long long cap = (long long)di.sms * occ;
    const int grid = (int)(want < cap ? want : cap);
    VerifyParams pc = p;
    void* args[] = {&pc};
    err = launch_pdl(reinterpret_cast<const void*>(residual_kernel<T, VEC>), dim3(grid),
                     dim3(kThreads), s, args);
    if (err != cudaSuccess) return err;
  }
  if (compact) {
    const int threads = p.B >= 1024 ? 1024 : ((p.B + kWarp - 1) / kWarp) * kWarp;
    const int grid = (p.B + threads - 1) / threads;
    VerifyParams pc = p;
    void* args[] = {&pc};
    err = launch_pdl(reinterpret_cast<const void*>(compact_kernel), dim3(grid), dim3(threads), s,
                     args);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

template <int MODE>
cudaError_t launch_mode(int dtype, bool vec, const VerifyParams& p, bool compact, cudaStream_t s) {
  if (dtype == kBF16)
    return vec ? launch_typed<MODE, uint16_t, 8>(p, compact, s)
               : launch_typed<MODE, uint16_t, 1>(p, compact, s);
  return vec ? launch_typed<MODE, float, 4>(p, compact, s) : launch_typed<MODE, float, 1>(p, compact, s);
}

}  // namespace

int chunks_per_task(int dtype, bool vec) {
  if (vec) return dtype == kBF16 ? Ring<uint16_t>::kBulkG : Ring<float>::kBulkG;
  return Lane<float, 1>::G;
}

int residual_chunks_per_task(int dtype, bool vec) {
  if (!vec) return residual_group<float, 1>();
  return dtype == kBF16 ? residual_group<uint16_t, 8>() : residual_group<float, 4>();
}

cudaError_t launch_verify(int mode, int dtype, bool vec, const VerifyParams& p, bool compact,
                          cudaStream_t stream) {
  switch (mode) {
    case kOneHot: return launch_mode<kOneHot>(dtype, vec, p, compact, stream);
    case kDense: return launch_mode<kDense>(dtype, vec, p, compact, stream);
    default: return launch_mode<kGreedy>(dtype, vec, p, compact, stream);
  }
}

}  // namespace sv
