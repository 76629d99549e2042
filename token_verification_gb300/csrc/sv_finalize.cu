// sv_finalize.cu - kernel F of the verification calls: per-request tests,
// draws and the packed output, after kernel A's chunk records.
//
// Method ("【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §2.1 "算法骨架"):
// accept draft x_i with probability min(1, p_i(x_i) / q_i(x_i)) in position
// order; at the first rejection n draw from norm(max(0, p_n - q_n)); if all
// drafts are accepted draw the extra token from the last position's p.
// Greedy rule (§11 of the same page): accept while x_i equals the target
// argmax.  Requests are independent and verified in parallel ("投机解码"
// (FastDeploy), "高效投机解码框架设计").
//
// Kernel F (finalize_kernel, one CTA per request) combines each row's chunk
//   records, with one-hot drafts draws beside each row's summary the token
//   its position would draw (the crossing chunk from the records, then one
//   rescan of that single chunk), and runs the acceptance tests of all
//   positions at once (one lane per position); typical acceptance draws after
//   the tests, at the stopping position only.  The last CTA of the call
//   writes the padding-free packed output (exclusive scan of accept_len,
//   packed tokens, per-token batch ids).  F starts with programmatic
//   dependent launch and waits on the device for kernel A's records.
// Kernel R (dense drafts only) follows F: a request rejected at n needs the
//   chunk sums of max(0, p_n - q_n), one more pass over its (target, draft)
//   row pair; F publishes those requests, R spreads their row pairs over
//   every warp of the GPU and draws their tokens.  F publishes the requests
//   whose drafts all passed too: their bonus draws from p (one warp each)
//   run in R beside the residual passes, off F's critical path.  R's last
//   CTA writes the packed output.  Typical acceptance and rejection
//   sampling on candidate trees have their own finalize kernels here.
#include "sv_rows.cuh"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// drawing one token
// ---------------------------------------------------------------------------

// First chunk c whose cumulative weight exceeds `target` (chunk weights from
// `weight(c)`, all in one frame).  Returns c and the fraction of chunk c's
// weight that lies below the target; if rounding leaves the target past the
// last chunk, returns the last chunk of positive weight with fraction 2
// (which selects its last positive element).  c = -1 if no weight at all.
// The chunk weights of the first kRecCache * 32 chunks come from `wc`
// (cached per lane: chunk lane + 32 t in wc[t]); later chunks from weight(c).
template <class F>
__device__ int find_chunk(const float (&wc)[kRecCache], F weight, int NC, float target,
                          float* frac) {
  const int lane = lane_id();
  float base = 0.f;
  auto round = [&](int c0, float w, int* out) {
    const float incl = warp_incl_scan(w);
    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && base + incl > target);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const float below = target - (base + __shfl_sync(0xffffffffu, incl - w, l));
      const float wl = __shfl_sync(0xffffffffu, w, l);
      *frac = fminf(fmaxf(below / wl, 0.f), 1.f);
      *out = c0 + l;
      return true;
    }
    base += __shfl_sync(0xffffffffu, incl, kWarp - 1);
    return false;
  };
  int found = -1;
#pragma unroll
  for (int t = 0; t < kRecCache; ++t)
    if (found < 0 && t * kWarp < NC && round(t * kWarp, wc[t], &found)) break;
  if (found >= 0) return found;
  for (int c0 = kRecCache * kWarp; c0 < NC; c0 += kWarp) {
    const int c = c0 + lane;
    if (round(c0, c < NC ? weight(c) : 0.f, &found)) return found;
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

// ---------------------------------------------------------------------------
// contiguous-run draws (vector paths): lane l takes chunks / elements
// [l*n, (l+1)*n), so one warp scan of the lane sums and one ballot locate the
// crossing lane, and that lane walks its own run
// ---------------------------------------------------------------------------

// The chunk where the cumulative weight (in chunk order) first exceeds
// u * total, over NC chunk weights weight(c).  frac = the share of that
// chunk's weight below the target; with no crossing (rounding only) the last
// chunk of positive weight with frac = 2.  Returns -1 without any weight.
template <class F>
__device__ int find_chunk_runs(F weight, int NC, float u, float* frac) {
  const int lane = lane_id();
  const int per = (NC + kWarp - 1) / kWarp;
  const int c0 = lane * per;
  float s = 0.f;
  for (int i = 0; i < per; ++i)
    if (c0 + i < NC) s += weight(c0 + i);
  const float incl = warp_incl_scan(s);
  const float target = u * __shfl_sync(0xffffffffu, incl, kWarp - 1);
  const unsigned hit = __ballot_sync(0xffffffffu, s > 0.f && incl > target);
  int c = -1;
  float f = 0.f;
  if (hit) {
    const int l = __ffs(hit) - 1;
    if (lane == l) {
      float acc = incl - s;
      for (int i = 0; i < per && c0 + i < NC; ++i) {
        const float w = weight(c0 + i);
        if (w > 0.f && acc + w > target) {
          c = c0 + i;
          f = fminf(fmaxf((target - acc) / w, 0.f), 1.f);
          break;
        }
        acc += w;
      }
      if (c < 0) {  // rounding inside the lane: its last positive chunk
        for (int i = 0; i < per && c0 + i < NC; ++i)
          if (weight(c0 + i) > 0.f) c = c0 + i;
        f = 2.f;
      }
    }
    c = __shfl_sync(0xffffffffu, c, l);
    f = __shfl_sync(0xffffffffu, f, l);
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, s > 0.f);
    if (!pos) return -1;
    const int l = 31 - __clz(pos);
    if (lane == l)
      for (int i = 0; i < per && c0 + i < NC; ++i)
        if (weight(c0 + i) > 0.f) c = c0 + i;
    c = __shfl_sync(0xffffffffu, c, l);
    f = 2.f;
  }
  *frac = f;
  return c;
}

// find_chunk_runs with each lane's run of chunk weights read once into
// registers (rows of up to 8 * 32 chunks; longer rows take find_chunk_runs):
// the same sums in the same order, one read of weights that are costly to
// read (global memory).
template <class F>
__device__ int find_chunk_runs_once(F weight, int NC, float u, float* frac) {
  constexpr int kRun = 8;
  const int per = (NC + kWarp - 1) / kWarp;
  if (per > kRun) return find_chunk_runs(weight, NC, u, frac);
  const int lane = lane_id();
  const int c0 = lane * per;
  float w[kRun];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kRun; ++i) {
    w[i] = (i < per && c0 + i < NC) ? weight(c0 + i) : 0.f;
    if (i < per && c0 + i < NC) s += w[i];
  }
  const float incl = warp_incl_scan(s);
  const float target = u * __shfl_sync(0xffffffffu, incl, kWarp - 1);
  const unsigned hit = __ballot_sync(0xffffffffu, s > 0.f && incl > target);
  int c = -1;
  float f = 0.f;
  if (hit) {
    const int l = __ffs(hit) - 1;
    if (lane == l) {
      float acc = incl - s;
#pragma unroll
      for (int i = 0; i < kRun; ++i) {
        if (c < 0 && i < per && c0 + i < NC) {
          if (w[i] > 0.f && acc + w[i] > target) {
            c = c0 + i;
            f = fminf(fmaxf((target - acc) / w[i], 0.f), 1.f);
          } else {
            acc += w[i];
          }
        }
      }
      if (c < 0) {  // rounding inside the lane: its last positive chunk
#pragma unroll
        for (int i = 0; i < kRun; ++i)
          if (i < per && c0 + i < NC && w[i] > 0.f) c = c0 + i;
        f = 2.f;
      }
    }
    c = __shfl_sync(0xffffffffu, c, l);
    f = __shfl_sync(0xffffffffu, f, l);
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, s > 0.f);
    if (!pos) return -1;
    const int l = 31 - __clz(pos);
    if (lane == l)
#pragma unroll
      for (int i = 0; i < kRun; ++i)
        if (i < per && c0 + i < NC && w[i] > 0.f) c = c0 + i;
    c = __shfl_sync(0xffffffffu, c, l);
    f = 2.f;
  }
  *frac = f;
  return c;
}

// Elements 32*lane .. 32*lane+31 of chunk c as stored (-inf past V): four
// 128-bit words of bf16 pairs, or eight of fp32; get(e) widens element e.
template <typename T>
struct Run {
  static constexpr int E = 16 / (int)sizeof(T);  // elements per 128-bit word
  uint4 q[kWarp / E];
  __device__ __forceinline__ float get(int e) const {
    const uint4 w = q[e / E];
    const int i = e % E;
    if constexpr (sizeof(T) == 2) {
      const uint32_t pr = (i >> 1) == 0 ? w.x : (i >> 1) == 1 ? w.y : (i >> 1) == 2 ? w.z : w.w;
      return __uint_as_float((i & 1) ? (pr & 0xffff0000u) : (pr << 16));
    } else {
      return __uint_as_float(i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w);
    }
  }
};

template <typename T>
__device__ __forceinline__ void load_run(const T* row, int V, int c, Run<T>& r) {
  constexpr int E = Run<T>::E;
  const int j0 = c * kChunk + lane_id() * kWarp;
  const uint4 pad = sizeof(T) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                   : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
#pragma unroll
  for (int g = 0; g < kWarp / E; ++g) {
    const int j = j0 + g * E;  // V is a multiple of E on the vector paths
    r.q[g] = j < V ? __ldg(reinterpret_cast<const uint4*>(row + j)) : pad;
  }
}

// Which of this lane's 32 elements of chunk c are allowed: the grammar mask
// word (one word covers exactly the lane's run), the top-k / top-p cut and
// the excluded token x.
template <typename T>
__device__ __forceinline__ uint32_t run_allowed(const Run<T>& v, const uint32_t* mrow,
                                                int mask_words, int c, float cut, int x) {
  const int lane = lane_id();
  uint32_t a = 0xffffffffu;
  if (mrow) a = mask_word(mrow, mask_words, c);
  if (cut > -INFINITY) {
#pragma unroll
    for (int e = 0; e < kWarp; ++e)
      if (!(v.get(e) >= cut)) a &= ~(1u << e);
  }
  const int xo = x - (c * kChunk + lane * kWarp);
  if (xo >= 0 && xo < kWarp) a &= ~(1u << xo);
  return a;
}

// Smallest element whose cumulative weight (in index order) exceeds frac
// times the chunk total, over the lanes' runs of weights weight(e) (element
// e of this lane's run, recomputed from registers rather than stored); zero
// weights are never chosen; the last positive element if rounding leaves
// none.
template <class Wt>
__device__ int pick_in_runs(Wt weight, float frac, int base_j) {
  const int lane = lane_id();
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kWarp; ++e) s += weight(e);
  const float incl = warp_incl_scan(s);
  const float thr = frac * __shfl_sync(0xffffffffu, incl, kWarp - 1);
  const unsigned hit = __ballot_sync(0xffffffffu, s > 0.f && incl > thr);
  int t = -1, l;
  if (hit) {
    l = __ffs(hit) - 1;
    if (lane == l) {
      float acc = incl - s;
      int last = -1;
#pragma unroll
      for (int e = 0; e < kWarp; ++e) {
        const float we = weight(e);
        acc += we;
        if (we > 0.f) {
          last = e;
          if (t < 0 && acc > thr) t = e;
        }
      }
      if (t < 0) t = last;
    }
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, s > 0.f);
    if (!pos) return -1;
    l = 31 - __clz(pos);
    if (lane == l)
#pragma unroll
      for (int e = 0; e < kWarp; ++e)
        if (weight(e) > 0.f) t = e;
  }
  t = __shfl_sync(0xffffffffu, t, l);
  return base_j + l * kWarp + t;
}

// Draw from w_j = 2^((l_j - m) c) over one row (w = 0 at mask_x, at the
// `nexcl` tokens of `excl` (the rejected candidates of a tree node), at the
// tokens the grammar mask row `mrow` rules out and below the top-k / top-p
// cut value) given the row's softmax chunk records, which leave out the same
// tokens: the crossing chunk from the records, then one rescan of that chunk
// in its own frame.
template <typename T, int VEC, bool kSharedRecords = false>
__device__ int draw_from_records(const T* row, const float2* rec, int NC, int V, float m, float cc,
                                 float u, int mask_x, const uint32_t* mrow, int mask_words,
                                 float cut, const int* excl = nullptr, int nexcl = 0) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  const float mc = __fmul_rn(m, cc);
  auto record = [&](int c) { return kSharedRecords ? rec[c] : __ldcg(rec + c); };
  auto weight = [&](int c) {
    const float2 r = record(c);
    return r.y * reframe(r.x, mc, cc);
  };
  if constexpr (VEC * sizeof(T) == 16) {
    float frac = 0.f;
    const int c = find_chunk_runs(weight, NC, u, &frac);
    if (c < 0) return -1;
    Run<T> v;
    load_run<T>(row, V, c, v);
    uint32_t a = run_allowed<T>(v, mrow, mask_words, c, cut, mask_x);
    for (int k = 0; k < nexcl; ++k) {
      const int xo = excl[k] - (c * kChunk + lane * kWarp);
      if (xo >= 0 && xo < kWarp) a &= ~(1u << xo);
    }
    const float nbc = -record(c).x * cc;
    return pick_in_runs(
        [&](int e) { return ((a >> e) & 1u) ? ex2(fmaf(v.get(e), cc, nbc)) : 0.f; }, frac,
        c * kChunk);
  } else {
    float wc[kRecCache];  // one batch of loads for the first 256 chunks
    float tot = 0.f;
#pragma unroll
    for (int t = 0; t < kRecCache; ++t) {
      const int c = lane + t * kWarp;
      wc[t] = c < NC ? weight(c) : 0.f;
      tot += wc[t];
    }
    for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) tot += weight(c);
    tot = warp_sum(tot);
    float frac = 0.f;
    const int c = find_chunk(wc, weight, NC, u * tot, &frac);
    if (c < 0) return -1;
    typename L::Raw raw[L::NV];
    load_chunk<T, VEC>(row, V, c, raw);
    if (mrow) allow_only_chunk<T, VEC>(raw, mask_word(mrow, mask_words, c));
    if (cut > -INFINITY) threshold_chunk<T, VEC>(raw, cut);
    const float nbc = -record(c).x * cc;
    float w[L::NV * VEC];
    float gsum[L::NV];
#pragma unroll
    for (int k = 0; k < L::NV; ++k) {
      gsum[k] = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        float we = ex2(fmaf(L::get(raw[k], e), cc, nbc));
        const int j = c * kChunk + tile_offset<VEC>(k, e, lane);
        if (j == mask_x) we = 0.f;
        for (int q = 0; q < nexcl; ++q)
          if (j == excl[q]) we = 0.f;
        w[k * VEC + e] = we;
        gsum[k] += we;
      }
    }
    return select_in_tile<L::NV, VEC>(w, gsum, frac, c * kChunk);
  }
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
// padding-free output ("投机解码" (FastDeploy), "高效投机解码框架设计")
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

// Exclusive scan of accept_len, packed tokens and per-token batch ids, by
// one CTA over all B requests (their outputs are complete and visible).
// Each thread reads all of its request's tokens before writing any, so the
// copy costs one memory round trip.
__device__ void compact_all(const VerifyParams& p, int* smem) {
  const int B = p.B, W = p.K + 1;
  int offset = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const int L = b < B ? __ldcg(p.out_accept_len + b) : 0;
    int tok[kMaxK + 1];
#pragma unroll
    for (int k = 0; k <= kMaxK; ++k)  // every token at once, with L (no wait on L)
      tok[k] = (p.out_packed && b < B && k < W) ? __ldcg(p.out_tokens + (long long)b * W + k) : -1;
    const int cu = offset + block_excl_scan(L, smem);
    if (b < B) {
      if (p.out_cu) p.out_cu[b] = cu;
#pragma unroll
      for (int k = 0; k <= kMaxK; ++k)
        if (k < L) {
          if (p.out_packed) p.out_packed[cu + k] = tok[k];
          if (p.out_batch_id) p.out_batch_id[cu + k] = b;
        }
    }
    offset += block_sum(L, smem);
  }
  if (p.out_cu && threadIdx.x == 0) p.out_cu[B] = offset;
  for (long long q = offset + threadIdx.x; q < (long long)B * W; q += blockDim.x) {
    if (p.out_packed) p.out_packed[q] = -1;
    if (p.out_batch_id) p.out_batch_id[q] = -1;
  }
}

// ---------------------------------------------------------------------------
// kernel F: per-request finalisation (one CTA per request, after kernel A)
// ---------------------------------------------------------------------------

// Summary of one row from its chunk records (one warp).
template <int MODE, typename T>
__device__ RowSum summarise_row(const VerifyParams& p, int b, int r, int Kb, int x,
                                float2* copy) {
  RowSum rs{qnan(), 0.f, 0.f, -1, 0.f};
  const long long rowid = (long long)b * p.R + r;
  const float2* rec = p.rec + rowid * p.NC;
  if (MODE == kGreedy) {
    const float2 a = combine_argmax_records(rec, p.NC);
    rs.m = a.x;
    rs.idx = __float_as_int(a.y);
    return rs;
  }
  const bool has_x = x >= 0 && x < p.V;
  const float lx = __ldcg(p.lx + rowid);  // recorded by kernel A (meaningful if has_x)
  const float2 ms = combine_softmax_records(rec, p.NC, p.cc, copy);
  rs.m = ms.x;
  rs.s = ms.y;
  if (has_x && is_finite(ms.x)) rs.wx = ex2(fmaf(lx, p.cc, -ms.x * p.cc));
  if (MODE == kTypical && is_finite(ms.x) && ms.y > 0.f) {
    const float a = combine_entropy(rec, p.ent + rowid * p.NC, p.NC, p.cc, ms.x);
    rs.h = __logf(ms.y) - 0.6931471805599453f * a / ms.y;
  }
  return rs;
}

// Threads of a finalize CTA: 8 warps.
template <int MODE>
__host__ __device__ constexpr int fin_threads() { return 256; }
constexpr int kMaxRows = 2 * kMaxK + 1;

// Where a dense-draft request draws - its rejected position n (< K_b), or
// the bonus position n = K_b when every draft passed - with the target and
// draft rows' maxima and reciprocal sums there (mq and iq unused at the
// bonus position; n < 0: nothing left to draw).
struct Residual {
  int n;
  float mp, ip, mq, iq;
};

template <int MODE, typename T, int VEC>
__device__ __forceinline__ void finalize_request(const VerifyParams& p, int b, int Kb,
                                              const RowSum* srow, const int* s_tok, int x,
                                              float u, int timed_out, Residual* resid,
                                              float uK, const float2* s_rec);
template <typename T, int VEC, bool kGlobalSums = false>
__device__ __noinline__ void residual_pick(const VerifyParams& p, int b, const Residual& st,
                                           const float* sums, const float2* srec);

// Draft token of row r of request b, or -1 (rows without one, or K_b invalid).
__device__ __forceinline__ int row_token(const VerifyParams& p, int b, int r, int Kb) {
  if (!row_needed(p, r, Kb)) return -1;
  const int i = r > p.K ? r - p.K - 1 : r;
  return i < Kb ? __ldg(p.draft_tokens + (long long)b * p.K + i) : -1;
}

// The token position r draws if the walk stops there (one warp): the
// residual max(0, p_r - q_r) of a one-hot draft (p_r without x_r; x_r itself
// when no mass is left beside it), else a draw from p_r (the bonus position,
// typical acceptance, the bonus of dense drafts).  -1 for a row without a
// finite max or a failed draw.  Each summarising warp computes it for its own
// row, so the draw overlaps the other rows and the acceptance tests.
template <int MODE, typename T, int VEC>
__device__ __forceinline__ int position_draw(const VerifyParams& p, int b, int r, int Kb,
                                             const RowSum& rs, int xr, float uK,
                                             const float2* srec) {
  if (!is_finite(rs.m)) return -1;
  const bool residual = MODE == kOneHot && r < Kb;
  if (residual && !(rs.s > 0.f)) return xr;  // p_r is the point mass at x_r
  const T* row = row_ptr<T>(p.target, (long long)b * (p.K + 1) + r, p.V);
  const uint32_t* mrow = mask_row(p, b, r);
  const float cut = row_cut(p, (long long)b * p.R + r);
  return srec ? draw_from_records<T, VEC, true>(row, srec + (long long)r * p.NC, p.NC, p.V, rs.m,
                                                p.cc, uK, residual ? xr : -1, mrow, p.mask_words,
                                                cut)
              : draw_from_records<T, VEC>(row, p.rec + ((long long)b * p.R + r) * p.NC, p.NC,
                                          p.V, rs.m, p.cc, uK, residual ? xr : -1, mrow,
                                          p.mask_words, cut);
}

// Shared memory of one request's finalisation.
struct FinShared {
  RowSum srow[kMaxRows];
  Residual resid;
  int last[32];
  int tok[kMaxRows];  // one-hot drafts: the token each position would draw
};

// Request b's finalisation by the calling CTA (every thread; any multiple
// of 32 threads).  Rows are summarised by the CTA's warps; with one-hot
// drafts each of them also draws the token its own position would emit if
// the walk stopped there (the residual or bonus draw of rejection sampling,
// §2.1 of the page cited at the top of this file); the chunk records are
// kept in shared memory (when they fit) for the draws.  Then one warp runs
// the acceptance tests of all positions at once (one lane per position) and
// takes the stopping position's token (typical acceptance: draws it then),
// or the argmax (greedy).  A dense-draft request is published for kernel R,
// which draws its token and writes its outputs.  wait() is called
// by every thread once the request's inputs are loaded and before its
// records are read.  s_rec: the request's [R*NC] records copied to shared
// memory for the draws, or null.
template <int MODE, typename T, int VEC, class Wait>
__device__ __forceinline__ void finalize_one(const VerifyParams& p, int b, FinShared& fs,
                                             float2* s_rec, Wait wait) {
  const int nwarps = (int)(blockDim.x >> 5);
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const int K = p.K;
  // The request's inputs are read before waiting for its records: kernel A
  // lets the finalize kernel launch only after its own wait, when every
  // earlier producer of the inputs has finished.
  const int Kb = p.draft_lens ? __ldg(p.draft_lens + b) : K;
  const int Kv = (Kb >= 0 && Kb <= K) ? Kb : 0;
  const int x0 = warp < p.R ? row_token(p, b, warp, Kb) : -1;
  int x = -1;
  float u = 0.f;
  const float uK = MODE != kGreedy ? __ldg(p.uniforms + (long long)b * (K + 1) + K) : 0.f;
  if (warp == 0) {
    if (lane < Kv) x = __ldg(p.draft_tokens + (long long)b * K + lane);
    if (MODE != kGreedy && lane < Kv) u = __ldg(p.uniforms + (long long)b * (K + 1) + lane);
  }
  if (threadIdx.x == 0) fs.resid.n = -1;
  wait(Kb);
  if (p.out_cut)  // filtered calls: each row's cut value, NaN for rows not needed
    for (int r = threadIdx.x; r < p.R; r += blockDim.x)
      p.out_cut[(long long)b * p.R + r] =
          row_needed(p, r, Kb) ? __ldcg(p.thr + (long long)b * p.R + r) : qnan();
  // issued before the row summaries so that its latency overlaps theirs
  const int timed_out = warp == 0 ? __ldcg(p.err) : 0;
  for (int r = warp; r < p.R; r += nwarps) {
    RowSum rs{qnan(), 0.f, 0.f, -1, 0.f};
    const int xr = r == warp ? x0 : row_token(p, b, r, Kb);
    if (row_needed(p, r, Kb))
      rs = summarise_row<MODE, T>(p, b, r, Kb, xr, s_rec ? s_rec + (long long)r * p.NC : nullptr);
    if (lane == 0) fs.srow[r] = rs;
    // target row r <= K_b: the draw of position r, for one-hot drafts
    // beside the summaries (typical acceptance draws after the tests, at the
    // stopping position only; dense drafts draw in kernel R)
    if (MODE == kOneHot && Kb >= 0 && Kb <= K && r <= Kb) {
      const int tok = position_draw<MODE, T, VEC>(p, b, r, Kb, rs, xr, uK, s_rec);
      if (lane == 0) fs.tok[r] = tok;
    }
  }
  __syncthreads();
  if (warp == 0)
    finalize_request<MODE, T, VEC>(p, b, Kb, fs.srow, fs.tok, x, u, timed_out, &fs.resid, uK,
                                   s_rec);
  __syncthreads();
  // Dense drafts, rejected at n: the request is published for the residual
  // kernel, which reads its row pair with every SM and writes its outputs.
  if (MODE == kDense && threadIdx.x == 0 && fs.resid.n >= 0) {
    // residual slots fill the slot arrays from the front, bonus draws from
    // the back (a request publishes at most one of either)
    const int slot = fs.resid.n < Kb ? atomicAdd(p.n_pend, 1) : p.B - 1 - atomicAdd(p.n_bonus, 1);
    p.pend[slot] = b;
    p.rpn[slot] = fs.resid.n;
    p.rpar[slot] = make_float4(fs.resid.mp, fs.resid.ip, fs.resid.mq, fs.resid.iq);
  }
  // Dense drafts: kernel R, which waits for this kernel to end, clears the
  // counters and writes the packed output, so the CTA is done.
  if (MODE == kDense) return;
  // The last request of the call clears the counters and writes the packed
  // output.
  if (threadIdx.x == 0) fs.last[0] = atomic_add_acq_rel(p.fin_ticket, 1) + 1 == p.B;
  __syncthreads();
  if (!fs.last[0]) return;
  if (threadIdx.x == 0) {
    *p.err = 0;
    *p.fin_ticket = 0;
    *p.work = 0u;
  }
  if (p.compact_in_finalize) compact_all(p, fs.last);
}

// Kernel F: one CTA per request, chained to kernel A by programmatic
// dependent launch.  Dynamic shared memory: [R*NC] records when cached.
template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(fin_threads<MODE>()) finalize_kernel(const VerifyParams p) {
  extern __shared__ float2 s_dyn[];
  __shared__ FinShared fs;
  finalize_one<MODE, T, VEC>(p, blockIdx.x, fs, p.fin_cache ? s_dyn : nullptr, [](int) {
    pdl_wait();
    pdl_launch_dependents();
  });
}

template <int MODE, typename T, int VEC>
__device__ __forceinline__ void finalize_request(const VerifyParams& p, int b, int Kb,
                                              const RowSum* srow, const int* s_tok, int x,
                                              float u, int timed_out, Residual* resid,
                                              float uK, const float2* s_rec) {
  const int lane = lane_id();
  const int K = p.K;
  // A bounded wait that gave up in kernel A (a device fault) invalidates the
  // whole call: its chunk records may be missing.
  int status = timed_out ? kTimeout : 0;
  if (Kb < 0 || Kb > K) {
    status |= kBadDraftLen;
    Kb = 0;
  }
  if (!status && __any_sync(0xffffffffu, lane < Kb && (x < 0 || x >= p.V))) status = kBadToken;
  int n = 0, token = -1;
  float theta = -1.f;
  bool pending = false;
  if (!status) {
    RowSum rt{qnan(), 0.f, 0.f, -1, 0.f}, rd{qnan(), 0.f, 0.f, -1, 0.f};
    if (lane <= Kb) rt = srow[lane];
    if (MODE == kDense && lane < Kb) rd = srow[K + 1 + lane];
    bool bad = lane <= Kb && !is_finite(rt.m);
    if (MODE == kDense && lane < Kb) bad = bad || !is_finite(rd.m);
    bool acc = false;
    if (lane < Kb) {
      if (MODE == kGreedy) {
        acc = (x == rt.idx);
        theta = acc ? 1.f : 0.f;
      } else if (MODE == kTypical) {  // p(x) > min(eps, delta * exp(-H)); reports p(x)
        const float px = rt.wx / rt.s;
        theta = px;
        acc = px > fminf(p.eps, p.delta * __expf(-rt.h));
      } else {
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
      } else if (MODE == kDense) {
        // kernel R draws: from max(0, p_n - q_n) (n < K_b), or from p_n (the
        // bonus position n = K_b: mq and iq are not used)
        pending = true;
        if (lane == 0) *resid = Residual{n, m_n, 1.f / s_n, mq_n, 1.f / sq_n};
      } else {
        // one-hot drafts: drawn beside the row summaries; typical acceptance:
        // drawn now, at the stopping position only
        token = MODE == kOneHot ? s_tok[n]
                                : position_draw<MODE, T, VEC>(p, b, n, Kb, srow[n], x_n, uK, s_rec);
        if (token < 0) status = kBadLogits;
      }
    }
  }
  if (p.out_accept_prob && lane < K && (MODE != kGreedy || p.greedy_prob))
    p.out_accept_prob[(long long)b * K + lane] =
        (!status && lane < Kb && lane <= n) ? theta : -1.f;
  if (!pending) write_request(p, b, status, n, token, x);
}

// ---------------------------------------------------------------------------
// dense-draft residual (inside kernel F, by all warps of the request's CTA)
// ---------------------------------------------------------------------------

template <typename T, int VEC>
__host__ __device__ constexpr int residual_group() {
  return Lane<T, VEC>::G > 1 ? Lane<T, VEC>::G / 2 : 1;
}

// One warp: the residual chunk sums max(0, p_n - q_n) of chunks [c0, hi),
// at most residual_group() of them, over request b's (target, draft) row
// pair at the rejected position st.n (kExtra: with grammar masks and top-k /
// top-p cuts applied), into sums[c].
template <typename T, int VEC, bool kExtra>
__device__ __forceinline__ void residual_group_sums(const VerifyParams& p, int b,
                                                    const Residual& st, float* sums, int c0,
                                                    int hi) {
  using L = Lane<T, VEC>;
  constexpr int G = residual_group<T, VEC>();
  const int lane = lane_id();
  const int K = p.K;
  const float cc = p.cc;
  const T* tr = row_ptr<T>(p.target, (long long)b * (K + 1) + st.n, p.V);
  const T* dr = row_ptr<T>(p.draft, (long long)b * K + st.n, p.V);
  const float nbp = -st.mp * cc, nbq = -st.mq * cc;
  const uint32_t* mrow = kExtra ? mask_row(p, b, st.n) : nullptr;
  const float cut_t = kExtra ? row_cut(p, (long long)b * p.R + st.n) : -INFINITY;
  const float cut_d = kExtra ? row_cut(p, (long long)b * p.R + K + 1 + st.n) : -INFINITY;
  typename L::Raw rt[G][L::NV], rd[G][L::NV];
  uint32_t word[G];
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (c0 + g < hi) {
      load_chunk<T, VEC>(tr, p.V, c0 + g, rt[g]);
      load_chunk<T, VEC>(dr, p.V, c0 + g, rd[g]);
      if (kExtra && mrow) word[g] = mask_word(mrow, p.mask_words, c0 + g);
    }
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (c0 + g < hi) {
      if (kExtra) {
        if (mrow) {
          allow_only_chunk<T, VEC>(rt[g], word[g]);
          allow_only_chunk<T, VEC>(rd[g], word[g]);
        }
        if (cut_t > -INFINITY) threshold_chunk<T, VEC>(rt[g], cut_t);
        if (cut_d > -INFINITY) threshold_chunk<T, VEC>(rd[g], cut_d);
      }
      float w = 0.f;
#pragma unroll
      for (int k = 0; k < L::NV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          w += residual_weight(L::get(rt[g][k], e), L::get(rd[g][k], e), cc, nbp, st.ip, nbq,
                               st.iq);
      w = warp_sum(w);
      if (lane == 0) sums[c0 + g] = w;
    }
}

// One warp: the residual draw from the chunk sums (the crossing chunk, then
// a rescan of that chunk of both rows), and the request's outputs.
// A rejected row pair whose residual has no mass (only through rounding:
// max(0, p - q) sums to 0 only when p = q) draws from p_n instead.
template <typename T, int VEC>
__device__ __noinline__ int residual_fallback(const VerifyParams& p, int b, const Residual& st,
                                              const float2* srec, float uK) {
  const int NC = p.NC;
  const T* tr = row_ptr<T>(p.target, (long long)b * (p.K + 1) + st.n, p.V);
  const uint32_t* mrow = mask_row(p, b, st.n);
  const float cut_t = row_cut(p, (long long)b * p.R + st.n);
  return srec ? draw_from_records<T, VEC, true>(tr, srec + (long long)st.n * NC, NC, p.V, st.mp,
                                                p.cc, uK, -1, mrow, p.mask_words, cut_t)
              : draw_from_records<T, VEC>(tr, p.rec + ((long long)b * p.R + st.n) * NC, NC, p.V,
                                          st.mp, p.cc, uK, -1, mrow, p.mask_words, cut_t);
}

template <typename T, int VEC, bool kGlobalSums>
__device__ __noinline__ void residual_pick(const VerifyParams& p, int b, const Residual& st,
                                           const float* sums, const float2* srec) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  const int K = p.K, NC = p.NC;
  const float cc = p.cc;
  const T* tr = row_ptr<T>(p.target, (long long)b * (K + 1) + st.n, p.V);
  const T* dr = row_ptr<T>(p.draft, (long long)b * K + st.n, p.V);
  const float nbp = -st.mp * cc, nbq = -st.mq * cc;
  // the loads that do not depend on the sums, issued together
  const float uK = __ldg(p.uniforms + (long long)b * (K + 1) + K);
  const int x_all = lane < K ? __ldg(p.draft_tokens + (long long)b * K + lane) : -1;
  const uint32_t* mrow = mask_row(p, b, st.n);
  const float cut_t = row_cut(p, (long long)b * p.R + st.n);
  const float cut_d = row_cut(p, (long long)b * p.R + K + 1 + st.n);
  auto weight = [&](int c) { return kGlobalSums ? __ldcg(sums + c) : sums[c]; };
  int token;
  if constexpr (VEC * sizeof(T) == 16) {
    float frac = 0.f;
    const int c = kGlobalSums ? find_chunk_runs_once(weight, NC, uK, &frac)
                              : find_chunk_runs(weight, NC, uK, &frac);
    if (c < 0) {  // no residual mass (rounding only): draw from p_n
      token = residual_fallback<T, VEC>(p, b, st, srec, uK);
    } else {
      Run<T> vt, vd;
      load_run<T>(tr, p.V, c, vt);
      load_run<T>(dr, p.V, c, vd);
      const uint32_t at = run_allowed<T>(vt, mrow, p.mask_words, c, cut_t, -1);
      const uint32_t ad = run_allowed<T>(vd, mrow, p.mask_words, c, cut_d, -1);
      token = pick_in_runs(
          [&](int e) {
            return residual_weight(((at >> e) & 1u) ? vt.get(e) : -INFINITY,
                                   ((ad >> e) & 1u) ? vd.get(e) : -INFINITY, cc, nbp, st.ip, nbq,
                                   st.iq);
          },
          frac, c * kChunk);
    }
    const int x = lane < st.n ? x_all : -1;
    write_request(p, b, token < 0 ? kBadLogits : 0, st.n, token, x);
  } else {
    float wc[kRecCache];
    float tot = 0.f;
#pragma unroll
    for (int t = 0; t < kRecCache; ++t) {
      const int c = lane + t * kWarp;
      wc[t] = c < NC ? weight(c) : 0.f;
      tot += wc[t];
    }
    for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) tot += weight(c);
    tot = warp_sum(tot);
    if (!(tot > 0.f)) {  // no residual mass (rounding only): draw from p_n
      token = residual_fallback<T, VEC>(p, b, st, srec, uK);
    } else {
      float frac = 0.f;
      const int c = find_chunk(wc, weight, NC, uK * tot, &frac);
      typename L::Raw rt[L::NV], rd[L::NV];
      load_chunk<T, VEC>(tr, p.V, c, rt);
      load_chunk<T, VEC>(dr, p.V, c, rd);
      if (mrow) {
        const uint32_t word = mask_word(mrow, p.mask_words, c);
        allow_only_chunk<T, VEC>(rt, word);
        allow_only_chunk<T, VEC>(rd, word);
      }
      if (cut_t > -INFINITY) threshold_chunk<T, VEC>(rt, cut_t);
      if (cut_d > -INFINITY) threshold_chunk<T, VEC>(rd, cut_d);
      float w[L::NV * VEC];
      float gsum[L::NV];
#pragma unroll
      for (int k = 0; k < L::NV; ++k) {
        gsum[k] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float we =
              residual_weight(L::get(rt[k], e), L::get(rd[k], e), cc, nbp, st.ip, nbq, st.iq);
          w[k * VEC + e] = we;
          gsum[k] += we;
        }
      }
      token = select_in_tile<L::NV, VEC>(w, gsum, frac, c * kChunk);
    }
    const int x = lane < st.n ? x_all : -1;
    write_request(p, b, token < 0 ? kBadLogits : 0, st.n, token, x);
  }
}

// ---------------------------------------------------------------------------
// kernel R: the dense-draft residual over every SM (after kernel F)
// ---------------------------------------------------------------------------

// The requests kernel F published - rejected at n with dense drafts - need
// the chunk sums of max(0, p_n - q_n), one more pass over their (target,
// draft) row pair, before their token can be drawn.  Every warp of the grid
// takes (request, chunk group) items in turn - a chunk group is
// residual_group() chunks - writes their sums to the request's slot and
// counts the group in the slot's arrival counter (acquire-release); the warp
// that completes a request's last group draws its token from the sums (the
// crossing chunk, then a rescan of that chunk of both rows) and writes its
// outputs, while the other warps go on.  The last CTA to finish writes the
// packed output of the whole call and clears the counters.  Launched with
// programmatic dependent launch behind kernel F, so its CTAs are resident
// when F ends.
constexpr int kResThreads = 256;

template <typename T, int VEC, bool kExtra>
__global__ void __launch_bounds__(kResThreads, 2) residual_kernel(const VerifyParams p) {
  __shared__ int s_flag[32];
  pdl_wait();
  pdl_launch_dependents();
  constexpr int G = residual_group<T, VEC>();
  const int lane = lane_id();
  const int NC = p.NC;
  const int groups = (NC + G - 1) / G;
  const long long ritems = (long long)__ldcg(p.n_pend) * groups;
  const long long items = ritems + __ldcg(p.n_bonus);
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += warps) {
    if (it >= ritems) {  // a request whose drafts all passed: its bonus draw from p_K_b
      const int slot = p.B - 1 - (int)(it - ritems);
      const int b = __ldcg(p.pend + slot), n = __ldcg(p.rpn + slot);
      const float m = __ldcg(p.rpar + slot).x;
      const long long r = (long long)b * p.R + n;
      const float uK = __ldg(p.uniforms + (long long)b * (p.K + 1) + p.K);
      const int x = lane < n ? __ldg(p.draft_tokens + (long long)b * p.K + lane) : -1;
      const int token = draw_from_records<T, VEC>(
          row_ptr<T>(p.target, (long long)b * (p.K + 1) + n, p.V), p.rec + r * NC, NC, p.V, m,
          p.cc, uK, -1, mask_row(p, b, n), p.mask_words, row_cut(p, r));
      write_request(p, b, token < 0 ? kBadLogits : 0, n, token, x);
      continue;
    }
    const int slot = (int)(it / groups), c0 = (int)(it - (long long)slot * groups) * G;
    const float4 q = __ldcg(p.rpar + slot);
    const Residual st{__ldcg(p.rpn + slot), q.x, q.y, q.z, q.w};
    const int b = __ldcg(p.pend + slot);
    float* sums = p.rsums + (long long)slot * NC;
    residual_group_sums<T, VEC, kExtra>(p, b, st, sums, c0, min(NC, c0 + G));
    int last = 0;
    if (lane == 0) last = atomic_add_acq_rel(p.arrive + slot, 1) + 1 == groups;
    if (__shfl_sync(0xffffffffu, last, 0)) {  // every sum of this request is in
      residual_pick<T, VEC, true>(p, b, st, sums, nullptr);
      if (lane == 0) p.arrive[slot] = 0;
    }
  }
  // the last CTA to leave: the packed output of the whole call, counters
  __syncthreads();
  if (threadIdx.x == 0) s_flag[0] = atomic_add_acq_rel(p.r_exit, 1) + 1 == (int)gridDim.x;
  __syncthreads();
  if (!s_flag[0]) return;
  if (threadIdx.x == 0) {  // every counter of the call (kernel F left them to this kernel)
    *p.err = 0;
    *p.work = 0u;
    *p.n_pend = 0;
    *p.n_bonus = 0;
    *p.r_exit = 0;
  }
  if (p.compact_in_finalize) compact_all(p, s_flag);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int MODE, typename T, int VEC>
cudaError_t launch_typed(const VerifyParams& p, cudaStream_t s) {
  cudaError_t err = launch_records(MODE, sizeof(T) == 2 ? kBF16 : kF32, VEC > 1, p, s);
  if (err != cudaSuccess) return err;
  DeviceInfo di;
  err = device_info(&di);
  if (err != cudaSuccess) return err;
  VerifyParams pc = p;
  void* args[] = {&pc};
  // F: acceptance tests and draws, one CTA per request
  const void* fin = reinterpret_cast<const void*>(finalize_kernel<MODE, T, VEC>);
  static PerDevice once;
  err = per_device(once, nullptr, [&](int&) {
    return cudaFuncSetAttribute(fin, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kFinCacheLimit);
  });
  if (err != cudaSuccess) return err;
  err = launch_pdl(fin, dim3(p.B), dim3(fin_threads<MODE>()), s, args, fin_smem_bytes(p, false));
  if (err != cudaSuccess || MODE != kDense) return err;
  // R: the residual of the requests F published, over every SM (calls with
  // grammar masks or top-k / top-p cuts take a variant that applies them)
  const bool extra = p.mask || p.filter;
  const void* rk = extra ? reinterpret_cast<const void*>(residual_kernel<T, VEC, true>)
                         : reinterpret_cast<const void*>(residual_kernel<T, VEC, false>);
  static PerDevice once_r[2];
  int occ = 1;
  err = per_device(once_r[extra ? 1 : 0], &occ, [&](int& v) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, rk, kResThreads, 0) != cudaSuccess ||
        v < 1)
      v = 1;
    return cudaSuccess;
  });
  if (err != cudaSuccess) return err;
  constexpr int G = residual_group<T, VEC>();
  const long long want = ((long long)p.B * ((p.NC + G - 1) / G + 1) + kResThreads / kWarp - 1) /
                         (kResThreads / kWarp);
  const long long cap = (long long)di.sms * occ;
  return launch_pdl(rk, dim3((unsigned)(want < cap ? want : cap)), dim3(kResThreads), s, args);
}

// ---------------------------------------------------------------------------
// typical acceptance on a candidate tree (after kernel A over all tree rows)
// ---------------------------------------------------------------------------

// One CTA per request: every row's summary (max, sum, entropy), every node's
// typical test under its parent's distribution, the accepted subtree a depth
// level at a time, the deepest accepted node (lowest id among equals) by one
// reduction, then the draw from its row.
constexpr int kTreeTypicalThreads = 512;
constexpr size_t kTreeCacheLimit = 96 * 1024;  // records kept in shared memory for the draw

// Summaries of every tree row with the loads of up to 4 rows per warp issued
// together (rows of up to 64 chunks; wider rows one at a time); the records
// go to `cache` (shared memory) when given.  Same arithmetic as
// combine_softmax_records and combine_entropy.
template <typename T, bool kEntropy>
__device__ void summarise_tree_rows(const VerifyParams& p, int b, int N, RowSum* srow,
                                    float2* cache) {
  const int lane = lane_id(), warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int NC = p.NC;
  const float cc = p.cc;
  if (NC > 2 * kWarp) {
    for (int r = warp; r <= N; r += nw) {
      const RowSum rs = summarise_row<kEntropy ? kTypical : kTreeSample, T>(
          p, b, r, N, -1, cache ? cache + (long long)r * NC : nullptr);
      if (lane == 0) srow[r] = rs;
    }
    return;
  }
  constexpr int J = 4;
  for (int r0 = warp; r0 <= N; r0 += nw * J) {
    float2 rc[J][2];
    float ea[J][2];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int r = r0 + j * nw;
      const long long base = ((long long)b * p.R + r) * NC;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = lane + q * kWarp;
        const bool in = r <= N && c < NC;
        rc[j][q] = in ? __ldcg(p.rec + base + c) : make_float2(-INFINITY, 0.f);
        ea[j][q] = (kEntropy && in) ? __ldcg(p.ent + base + c) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int r = r0 + j * nw;
      if (r > N) break;
      const float m = warp_max_nan(max_nan(rc[j][0].x, rc[j][1].x));
      RowSum rs{m == -INFINITY ? -INFINITY : qnan(), 0.f, 0.f, -1, 0.f};
      if (is_finite(m)) {
        const float mc = __fmul_rn(m, cc);
        float sum = 0.f, a = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 rq = rc[j][q];
          sum += rq.y * reframe(rq.x, mc, cc);
          if (kEntropy && rq.y > 0.f) {
            const float d = (rq.x - m) * cc;
            a += ex2(d) * fmaf(d, rq.y, ea[j][q]);
          }
        }
        sum = warp_sum(sum);
        a = warp_sum(a);
        rs.m = m;
        rs.s = sum;
        if (kEntropy && sum > 0.f) rs.h = __logf(sum) - 0.6931471805599453f * a / sum;
      }
      if (cache) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (lane + q * kWarp < NC) cache[(long long)r * NC + lane + q * kWarp] = rc[j][q];
      }
      if (lane == 0) srow[r] = rs;
    }
  }
}

// The request's candidate tree into shared memory: parents and depths
// (load_tree), tokens, and each node's token's logit in its parent's row,
// read before kernel A finishes.  Returns the request's status so far
// (kBadTree, kBadToken or 0).
template <typename T>
__device__ int load_candidates(const VerifyParams& p, const TreeCall& t, int b, short* s_par,
                               short* s_depth, short* s_anc, int* s_tok, float* s_lx) {
  const int N = t.N;
  constexpr int kPer = (kMaxTreeNodes + 127) / 128;  // nodes per thread (>= 128 threads)
  int tk[kPer];  // the tokens' loads are issued before the parents'
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = 1 + threadIdx.x + i * (int)blockDim.x;
    tk[i] = n <= N ? __ldg(t.tokens + (long long)b * N + n - 1) : 0;
  }
  const bool tree_ok =
      load_tree(t.parent + (long long)b * t.parent_stride, N, t.D1 - 1, s_par, s_depth, s_anc);
  int bad = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = 1 + threadIdx.x + i * (int)blockDim.x;
    if (n > N) continue;
    const int tok = tk[i];
    s_tok[n] = tok;
    const bool ok = tok >= 0 && tok < p.V;
    bad |= !ok;
    s_lx[n] = (tree_ok && ok)
                  ? load_logit(row_ptr<T>(p.target, (long long)b * (N + 1) + s_par[n], p.V), tok)
                  : 0.f;
  }
  bad = __syncthreads_or(bad);
  return !tree_ok ? kBadTree : (bad ? kBadToken : 0);
}

// Path and tokens of a finished walk (one warp): level k < d holds the
// token of the path's node at level k + 1, level d the drawn token; -1 past
// them (and everywhere for a request with a status).  The last request of
// the call clears the workspace counters.
__device__ void write_tree_result(const VerifyParams& p, const TreeCall& t, int b, int status,
                                  int best, int d, int token, const short* s_par,
                                  const int* s_tok) {
  const int lane = lane_id();
  for (int k = lane; k < t.D1; k += kWarp) {
    int node = -1, tok = -1;
    if (!status && k <= d) {
      int a = best;  // the path's node at level k + 1 (best itself when k = d)
      for (int up = d; up > k + 1; --up) a = s_par[a];
      if (k < d) {
        tok = s_tok[a];
        node = s_par[a];
      } else {
        tok = token;
        node = best;
      }
    }
    if (t.out_path) t.out_path[(long long)b * t.D1 + k] = node;
    t.out_tokens[(long long)b * t.D1 + k] = tok;
  }
  if (lane == 0) {
    t.out_accept_len[b] = status ? 0 : d + 1;
    if (t.out_status) t.out_status[b] = status;
    if (atomic_add_acq_rel(p.fin_ticket, 1) + 1 == p.B) {
      *p.err = 0;
      *p.fin_ticket = 0;
      *p.work = 0u;
    }
  }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kTreeTypicalThreads) tree_typical_kernel(const VerifyParams p,
                                                                         const TreeCall t) {
  extern __shared__ float2 s_cache[];
  __shared__ RowSum srow[kMaxTreeNodes + 1];
  __shared__ short s_par[kMaxTreeNodes + 1], s_depth[kMaxTreeNodes + 1], s_anc[kMaxTreeNodes + 1];
  __shared__ int s_tok[kMaxTreeNodes + 1];
  __shared__ float s_lx[kMaxTreeNodes + 1];
  __shared__ unsigned char spass[kMaxTreeNodes + 1], sacc[kMaxTreeNodes + 1];
  __shared__ int s_best, s_status;
  __shared__ unsigned s_key[kTreeTypicalThreads / kWarp];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int N = t.N;
  const bool cached = (size_t)(N + 1) * p.NC * sizeof(float2) <= kTreeCacheLimit;
  // the tree, its tokens and each node's logit in its parent's row are
  // inputs: read them before waiting for kernel A
  const int status_in = load_candidates<T>(p, t, b, s_par, s_depth, s_anc, s_tok, s_lx);
  pdl_wait();
  pdl_launch_dependents();
  summarise_tree_rows<T, true>(p, b, N, srow, cached ? s_cache : nullptr);
  __syncthreads();
  for (int n = 1 + threadIdx.x; n <= N; n += blockDim.x) {
    unsigned char ok = 0;
    if (!status_in) {
      const RowSum rp = srow[s_par[n]];
      if (is_finite(rp.m) && rp.s > 0.f) {
        const float px = ex2(fmaf(s_lx[n], p.cc, -rp.m * p.cc)) / rp.s;
        ok = px > fminf(p.eps, p.delta * __expf(-rp.h));
      }
    }
    spass[n] = ok;
  }
  // The accepted nodes, a depth level at a time (a node is accepted when it
  // passes and its parent is accepted; the tree was checked, every node's
  // depth is at most max_depth), then the deepest one, the lowest id among
  // equals, by one reduction of (depth, -id) keys.
  if (threadIdx.x == 0) sacc[0] = 1;
  __syncthreads();
  if (!status_in)
    for (int d = 1; d < t.D1; ++d) {
      for (int n = 1 + threadIdx.x; n <= N; n += blockDim.x)
        if (s_depth[n] == d) sacc[n] = sacc[s_par[n]] && spass[n];
      __syncthreads();
    }
  unsigned key = 0u;
  int bad = 0;
  if (!status_in)
    for (int n = 1 + threadIdx.x; n <= N; n += blockDim.x)
      if (sacc[n]) {
        key = max(key, ((unsigned)s_depth[n] << 16) | (0xffffu - (unsigned)n));
        bad |= !is_finite(srow[n].m);  // an accepted node's row is needed
      }
  key = __reduce_max_sync(0xffffffffu, key);
  if (lane_id() == 0) s_key[warp] = key;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    int status = status_in ? status_in : (__ldcg(p.err) ? kTimeout : 0);
    if (!status && (!is_finite(srow[0].m) || bad)) status = kBadLogits;
    unsigned k = 0u;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) k = max(k, s_key[w]);
    s_best = k ? (int)(0xffffu - (k & 0xffffu)) : 0;
    s_status = status;
  }
  __syncthreads();
  if (warp != 0) return;
  const int status0 = s_status, best = s_best;
  int token = -1;
  if (!status0) {
    const RowSum rb = srow[best];
    const T* row = row_ptr<T>(p.target, (long long)b * (N + 1) + best, p.V);
    const float u = __ldg(t.uniforms + b);
    token = cached ? draw_from_records<T, VEC, true>(row, s_cache + (long long)best * p.NC, p.NC,
                                                     p.V, rb.m, p.cc, u, -1, nullptr, 0, -INFINITY)
                   : draw_from_records<T, VEC>(row, p.rec + ((long long)b * (N + 1) + best) * p.NC,
                                               p.NC, p.V, rb.m, p.cc, u, -1, nullptr, 0,
                                               -INFINITY);
  }
  const int status = status0 ? status0 : (token < 0 ? kBadLogits : 0);
  write_tree_result(p, t, b, status, best, status ? -1 : s_depth[best], token, s_par, s_tok);
}

// ---------------------------------------------------------------------------
// lossless tree verification by rejection sampling (after kernel A over
// every tree row, whose records leave each node's children tokens out)
// ---------------------------------------------------------------------------

// One CTA per request ("推测解码与 MTP" §10.4: EAGLE verified by rejection
// sampling is lossless; candidate trees of §3.3 / §4.2).  Every candidate is
// a one-hot draft of the distribution at its parent.  From the root, the
// children of the current node are tested in increasing id: with the
// row's weights w_j = 2^((l_j - m) c), child k (token x_k, not repeated
// among the earlier children) is accepted iff u_k * W_k < w(x_k), where
// W_k = S_excl + the weights of the distinct children tokens from k on - the
// residual left after the earlier children were rejected, a sum of positive
// terms (no cancellation); S_excl, the row's mass without its children's
// tokens, comes straight from kernel A's records.  A repeated token has no
// mass left and is rejected.  The first accepted child is emitted and the
// walk moves to it; when none is (or at a leaf) one token is drawn from the
// node's records, which are exactly the residual without the rejected
// children, with uniforms[b, 0].
constexpr int kTreeSampleThreads = 512;

template <typename T, int VEC>
__global__ void __launch_bounds__(kTreeSampleThreads) tree_sample_kernel(const VerifyParams p,
                                                                        const TreeCall t) {
  extern __shared__ float2 s_cache[];
  __shared__ RowSum srow[kMaxTreeNodes + 1];
  __shared__ short s_par[kMaxTreeNodes + 1], s_depth[kMaxTreeNodes + 1], s_anc[kMaxTreeNodes + 1];
  __shared__ int s_tok[kMaxTreeNodes + 1];
  __shared__ float s_lx[kMaxTreeNodes + 1], s_u[kMaxTreeNodes + 1];
  __shared__ int s_kid[kMaxTreeNodes];
  __shared__ float s_w[kMaxTreeNodes];
  __shared__ int s_excl[kMaxTreeNodes];
  const int b = blockIdx.x;
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const int N = t.N;
  const bool cached = (size_t)(N + 1) * p.NC * sizeof(float2) <= kTreeCacheLimit;
  const int status_in = load_candidates<T>(p, t, b, s_par, s_depth, s_anc, s_tok, s_lx);
  for (int n = threadIdx.x; n <= N; n += blockDim.x)
    s_u[n] = __ldg(t.uniforms + (long long)b * (N + 1) + n);
  pdl_wait();
  pdl_launch_dependents();
  summarise_tree_rows<T, false>(p, b, N, srow, cached ? s_cache : nullptr);
  __syncthreads();
  if (warp != 0) return;
  int status = status_in ? status_in : (__ldcg(p.err) ? kTimeout : 0);
  int node = 0, nk_final = 0;
  const float cc = p.cc;
  while (!status) {
    const RowSum rs = srow[node];
    if (!is_finite(rs.m)) {
      status = kBadLogits;
      break;
    }
    // the node's children in increasing id
    int nk = 0;
    for (int c0 = 1; c0 <= N; c0 += kWarp) {
      const int c = c0 + lane;
      const bool kid = c <= N && s_par[c] == node;
      const unsigned m = __ballot_sync(0xffffffffu, kid);
      if (kid) s_kid[nk + __popc(m & ((1u << lane) - 1u))] = c;
      nk += __popc(m);
    }
    __syncwarp();
    // their tokens' weights, 0 for a token an earlier child already carries
    for (int k = lane; k < nk; k += kWarp) {
      const int c = s_kid[k], x = s_tok[c];
      bool dup = false;
      for (int j = 0; j < k && !dup; ++j) dup = s_tok[s_kid[j]] == x;
      s_w[k] = dup ? 0.f : ex2(fmaf(s_lx[c], cc, -rs.m * cc));
    }
    __syncwarp();
    // W_k = S_excl + sum_{j >= k} w_j (suffix sums, blocks from the last);
    // the first child whose test passes is the accepted one
    int acc = -1;
    float carry = rs.s;
    for (int k0 = ((nk - 1) / kWarp) * kWarp; k0 >= 0 && nk > 0; k0 -= kWarp) {
      const int k = k0 + (kWarp - 1 - lane);  // lane 0 holds the block's last child
      const float w = k < nk ? s_w[k] : 0.f;
      const float suffix = warp_incl_scan(w);  // over this block's children from k on
      const float Wk = carry + suffix;
      const bool pass = k < nk && w > 0.f && s_u[s_kid[k]] * Wk < w;
      const unsigned hit = __ballot_sync(0xffffffffu, pass);
      if (hit) acc = k0 + (kWarp - 1 - (31 - __clz(hit)));  // the lowest child id of the block
      carry += __shfl_sync(0xffffffffu, suffix, kWarp - 1);
    }
    if (acc < 0) {  // every child rejected, or a leaf: draw here
      nk_final = nk;
      break;
    }
    node = s_kid[acc];
  }
  int token = -1;
  if (!status) {
    // the final node's children (all rejected) are left out of the draw,
    // as they are of its records
    for (int k = lane; k < nk_final; k += kWarp) s_excl[k] = s_tok[s_kid[k]];
    __syncwarp();
    const int* excl = s_excl;
    const RowSum rf = srow[node];
    const T* row = row_ptr<T>(p.target, (long long)b * (N + 1) + node, p.V);
    token = cached ? draw_from_records<T, VEC, true>(row, s_cache + (long long)node * p.NC, p.NC,
                                                     p.V, rf.m, cc, s_u[0], -1, nullptr, 0,
                                                     -INFINITY, excl, nk_final)
                   : draw_from_records<T, VEC>(row, p.rec + ((long long)b * (N + 1) + node) * p.NC,
                                               p.NC, p.V, rf.m, cc, s_u[0], -1, nullptr, 0,
                                               -INFINITY, excl, nk_final);
    if (token < 0) status = kBadLogits;
  }
  write_tree_result(p, t, b, status, node, status ? -1 : s_depth[node], token, s_par, s_tok);
}

template <typename T, int VEC>
cudaError_t launch_tree_typical_typed(const VerifyParams& p, const TreeCall& t, cudaStream_t s) {
  cudaError_t err = launch_records(kTypical, sizeof(T) == 2 ? kBF16 : kF32, VEC > 1, p, s);
  if (err != cudaSuccess) return err;
  VerifyParams pc = p;
  TreeCall tc = t;
  void* args[] = {&pc, &tc};
  const void* fn = reinterpret_cast<const void*>(tree_typical_kernel<T, VEC>);
  static PerDevice once;
  err = per_device(once, nullptr, [&](int&) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kTreeCacheLimit);
  });
  if (err != cudaSuccess) return err;
  const size_t cache = (size_t)(t.N + 1) * p.NC * sizeof(float2);
  return launch_pdl(fn, dim3(p.B), dim3(kTreeTypicalThreads), s, args,
                    cache <= kTreeCacheLimit ? cache : 0);
}

template <typename T, int VEC>
cudaError_t launch_tree_sample_typed(const VerifyParams& p, const TreeCall& t, cudaStream_t s) {
  cudaError_t err = launch_records(kTreeSample, sizeof(T) == 2 ? kBF16 : kF32, VEC > 1, p, s);
  if (err != cudaSuccess) return err;
  VerifyParams pc = p;
  TreeCall tc = t;
  void* args[] = {&pc, &tc};
  const void* fn = reinterpret_cast<const void*>(tree_sample_kernel<T, VEC>);
  static PerDevice once;
  err = per_device(once, nullptr, [&](int&) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kTreeCacheLimit);
  });
  if (err != cudaSuccess) return err;
  const size_t cache = (size_t)(t.N + 1) * p.NC * sizeof(float2);
  return launch_pdl(fn, dim3(p.B), dim3(kTreeSampleThreads), s, args,
                    cache <= kTreeCacheLimit ? cache : 0);
}
template <int MODE>
cudaError_t launch_mode(int dtype, bool vec, const VerifyParams& p, cudaStream_t s) {
  if (dtype == kBF16)
    return vec ? launch_typed<MODE, uint16_t, 8>(p, s) : launch_typed<MODE, uint16_t, 1>(p, s);
  return vec ? launch_typed<MODE, float, 4>(p, s) : launch_typed<MODE, float, 1>(p, s);
}

}  // namespace

size_t fin_cache_bytes(const VerifyParams& p) { return sizeof(float2) * (size_t)p.R * p.NC; }

size_t fin_smem_bytes(const VerifyParams& p, bool) { return p.fin_cache ? fin_cache_bytes(p) : 0; }

cudaError_t launch_tree_typical(int dtype, bool vec, const VerifyParams& p, const TreeCall& t,
                                cudaStream_t stream) {
  if (dtype == kBF16)
    return vec ? launch_tree_typical_typed<uint16_t, 8>(p, t, stream)
               : launch_tree_typical_typed<uint16_t, 1>(p, t, stream);
  return vec ? launch_tree_typical_typed<float, 4>(p, t, stream)
             : launch_tree_typical_typed<float, 1>(p, t, stream);
}

cudaError_t launch_tree_sample(int dtype, bool vec, const VerifyParams& p, const TreeCall& t,
                               cudaStream_t stream) {
  if (dtype == kBF16)
    return vec ? launch_tree_sample_typed<uint16_t, 8>(p, t, stream)
               : launch_tree_sample_typed<uint16_t, 1>(p, t, stream);
  return vec ? launch_tree_sample_typed<float, 4>(p, t, stream)
             : launch_tree_sample_typed<float, 1>(p, t, stream);
}

cudaError_t launch_verify(int mode, int dtype, bool vec, const VerifyParams& p,
                          cudaStream_t stream) {
  switch (mode) {
    case kOneHot: return launch_mode<kOneHot>(dtype, vec, p, stream);
    case kDense: return launch_mode<kDense>(dtype, vec, p, stream);
    case kTypical: return launch_mode<kTypical>(dtype, vec, p, stream);
    default: return launch_mode<kGreedy>(dtype, vec, p, stream);
  }
}

}  // namespace sv
