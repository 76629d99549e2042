// sv_filter.cu - kernel A for top-k / top-p filtered verification calls.
#include "sv_rows.cuh"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// kernel A for top-k / top-p calls: one row per thread-block cluster
// ---------------------------------------------------------------------------
//
// Filtering needs, per row, the k-th largest logit and the value at which
// the mass of the leading value classes reaches top_p - an order statistic
// and a quantile of the mass, which a single streaming pass cannot give.  A
// cluster of CTAs takes one row, each CTA a slice of whole chunks (at most
// 64 KB).  The slice is read from HBM once, for the row max; the later
// passes read it again and find it in L2, so shared memory holds only
// histograms and short lists, several rows are in flight per SM, and the
// passes' latency is hidden behind other rows' loads.
//
// With the max m known, the weights w = 2^((l - m) c) follow.  Candidates
// are the elements within 2^-20 of the max's weight; every element above a
// candidate is one.  One pass sums the row's mass, the mass outside the
// candidates and a histogram of the candidates over distance levels (eighths
// of a bit of weight below the max: a level is a range of values).  When the
// cut must lie among the candidates - at least k of them for top-k; for
// top-p more than top_p of the mass in them - the level holding the cut
// follows from the histogram, the elements of that one level are gathered
// into a list per CTA, and every CTA finds the cut's value class from the
// lists of the whole cluster.  Otherwise (a flat row, a large k, a list too
// long) a radix descent on order-preserving keys finds it, 8 bits per pass.
// Masses are summed as 2^-38 fixed-point integers in per-warp histograms and
// merged in rank order, so every CTA of the cluster takes the same
// decisions.  Finally each warp reduces its chunks to the same records the
// streaming kernel writes, over the kept elements only, and the row's cut
// value goes to the workspace for the finalize kernel's rescans.

constexpr int kCutThreads = 256;
constexpr int kCutWarps = kCutThreads / kWarp;
constexpr int kMaxChunksPerWarp = 4;  // slices of at most 32 chunks
constexpr int kListCap = 64;          // elements of the cut's level per CTA
constexpr float kCandBits = 20.f;
constexpr int kLimbBits = 19;

// Unsigned keys in the order of the values (-0.0 is taken as +0.0).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// floor(w * 2^38) for a weight (or a sum of up to 8 weights) w in [0, 8],
// from the bits of w with integer operations only (w = mant * 2^(e - 150),
// so w * 2^38 = mant * 2^(e - 112)).
__device__ __forceinline__ unsigned long long fixed_mass(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)(b >> 23);
  if (e == 0) return 0ull;  // zero (weights below 2^-126 are flushed)
  const unsigned long long mant = (b & 0x7fffffu) | 0x800000u;
  return e >= 112 ? mant << (e - 112) : (e > 112 - 24 ? mant >> (112 - e) : 0ull);
}

// floor(total * p_q / 2^32): a fraction p_q / 2^32 of a fixed-point mass.
__device__ __forceinline__ unsigned long long frac_of(unsigned long long total, uint32_t p_q) {
  return (total >> 32) * p_q + (((total & 0xffffffffull) * p_q) >> 32);
}

// Distance levels: a candidate's weight exponent a = (l - m) c in [-20, 0]
// falls into level floor(-8 a), kept as digit 255 - level so that larger
// values have larger digits, as key digits do.
__device__ __forceinline__ int level_digit(float a) { return 255 - __float2int_rz(-8.f * a); }

// Shared memory of a filter CTA.  Per-warp histograms: a warp sees at most
// 4096 elements, so a 19-bit limb sum stays below 2^31.
struct CutShared {
  uint32_t part[kCutWarps][256][2];  // per warp: low / high limbs of each bin (counts: [0])
  unsigned long long hist[2][256];   // this CTA's bins, read by the cluster (double-buffered)
  unsigned long long tot[256];       // the cluster's bins
  float red_m[kCutWarps], red_s[kCutWarps], red_t[kCutWarps];
  int red_n[kCutWarps];
  float cta_max, cta_s, cta_tail;  // read by the cluster
  int cta_n;
  int list_n;  // elements of the cut's level in this slice (read by the cluster)
  uint32_t list_key[kListCap];
  unsigned long long list_w[kListCap];
  uint32_t all_key[kFilterMaxCta * kListCap];  // the cluster's lists, in rank order
  unsigned long long all_w[kFilterMaxCta * kListCap];
  uint32_t best, lowest;
};

// Adds one element's weight w (MASS: as a fixed-point mass) or a count of
// `n` to bin `bin` of a per-warp histogram.
template <bool MASS>
__device__ __forceinline__ void add_to_bin(uint32_t (*mine)[2], int bin, float w, uint32_t n = 1) {
  if (MASS) {
    const unsigned long long q = fixed_mass(w);
    atomicAdd(&mine[bin][0], (uint32_t)(q & ((1u << kLimbBits) - 1u)));
    atomicAdd(&mine[bin][1], (uint32_t)(q >> kLimbBits));
  } else {
    atomicAdd(&mine[bin][0], n);
  }
}

// The digit whose bin reaches the target, scanning bins from 255 down:
// the first where base plus the bins down to it is >= target; without one
// (rounding only) the lowest non-empty bin.  `front` receives the sum of the
// bins above it.  Run by whole warps (each gets the result), integers only.
__device__ __forceinline__ int pick_digit(const unsigned long long* tot, unsigned long long base,
                                          unsigned long long target, unsigned long long& front) {
  const int lane = lane_id();
  unsigned long long part[8], s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    part[j] = tot[255 - (lane * 8 + j)];
    s += part[j];
  }
  unsigned long long incl = s;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const unsigned long long excl = incl - s;
  const unsigned hit = __ballot_sync(0xffffffffu, base + incl >= target);
  int j_hit = -1, j_low = -1;
  unsigned long long f_hit = 0, f_low = 0, acc = excl;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j_hit < 0 && base + acc + part[j] >= target) {
      j_hit = j;  // found on the first lane of `hit` (its bins reach the target)
      f_hit = acc;
    }
    if (part[j]) {
      j_low = j;
      f_low = acc;
    }
    acc += part[j];
  }
  int l, j;
  unsigned long long f;
  if (hit) {
    l = __ffs(hit) - 1;
    j = j_hit;
    f = f_hit;
  } else {
    const unsigned any = __ballot_sync(0xffffffffu, j_low >= 0);
    l = any ? 31 - __clz(any) : 0;
    j = j_low < 0 ? 7 : j_low;
    f = j_low < 0 ? acc - part[7] : f_low;
  }
  j = __shfl_sync(0xffffffffu, j, l);
  front = __shfl_sync(0xffffffffu, f, l);
  return 255 - (l * 8 + j);
}

// This CTA's histogram (the warps' limbs recombined) into hist[buf]; the
// warps' bins are cleared for the next pass as they are read.
__device__ __forceinline__ void publish_hist(CutShared* sh, int buf) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < kCutWarps; ++w) {
      t += ((unsigned long long)sh->part[w][i][1] << kLimbBits) + sh->part[w][i][0];
      sh->part[w][i][0] = 0u;
      sh->part[w][i][1] = 0u;
    }
    sh->hist[buf][i] = t;
  }
}

// After the cluster barrier: the cluster's histogram, summed in rank order
// (the remote loads issued together).
__device__ __forceinline__ void gather_hist(CutShared* sh, int buf, int ncta) {
  cg::cluster_group cluster = cg::this_cluster();
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    unsigned long long v[kFilterMaxCta];
#pragma unroll
    for (int r = 0; r < kFilterMaxCta; ++r)
      v[r] = r < ncta ? cluster.map_shared_rank(sh, r)->hist[buf][i] : 0ull;
    unsigned long long t = 0;
#pragma unroll
    for (int r = 0; r < kFilterMaxCta; ++r) t += v[r];
    sh->tot[i] = t;
  }
}

// The sum of the cluster's histogram, by every lane of the calling warp.
__device__ __forceinline__ unsigned long long warp_hist_total(const unsigned long long* tot) {
  unsigned long long t = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) t += tot[lane_id() * 8 + j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// The row, its grammar mask and the CTA's slice of chunks: warp w takes
// chunks c_lo + w + 8 t.
template <typename T>
struct Slice {
  const T* row;
  const uint32_t* mrow;
  int c_lo, nch;
};

// Chunk cl of the slice as this lane's register tile (disallowed tokens
// -inf; groups past V the -inf pad).  Warp-wide.
template <typename T, int VEC>
__device__ __forceinline__ void slice_chunk(const VerifyParams& p, const Slice<T>& s, int cl,
                                            typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV]) {
  const int c = s.c_lo + cl;
  load_chunk<T, VEC>(s.row, p.V, c, raw);
  if (s.mrow) allow_only_chunk<T, VEC>(raw, mask_word(s.mrow, p.mask_words, c));
}

// Calls f(j, v) for each candidate of chunk cl marked in `bits` (bit
// k * VEC + e: element e of the lane's group k), with its token index j and
// logit v read again (an L1 / L2 hit; candidates are never masked out).
template <typename T, int VEC, class F>
__device__ __forceinline__ void for_each_candidate(const VerifyParams& p, const Slice<T>& s, int cl,
                                                   uint32_t bits, F f) {
  const int base = (s.c_lo + cl) * kChunk;
  while (bits) {  // four loads in flight at a time
    int j[4];
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      j[q] = -1;
      if (bits) {
        const int t = __ffs(bits) - 1;
        bits &= bits - 1u;
        j[q] = base + tile_offset<VEC>(t / VEC, t % VEC, lane_id());
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = j[q] >= 0 ? load_logit(s.row, j[q]) : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (j[q] >= 0) f(j[q], v[q]);
  }
}

template <typename T, int VEC>
__device__ __forceinline__ float tile_max(const typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV]) {
  using L = Lane<T, VEC>;
  if constexpr (sizeof(T) == 2 && VEC == 8) {
    return lane_max_bf16(raw);
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) m = max_nan(m, L::get(raw[k], e));
    return m;
  }
}

// One radix pass over the slice (see radix_descent): elements >= keep
// (kKeep), in distance level lvl (kLevel), with the key prefix so far
// (kPrefix).  Runs of consecutive elements of a lane that fall into the same
// bin are merged before one atomic (a run's mass summed in fp32, at most
// VEC weights, then fixed).
template <typename T, int VEC, bool MASS, bool kPrefix, bool kKeep, bool kLevel>
__device__ __forceinline__ void accumulate(const VerifyParams& p, const Slice<T>& s, float keep,
                                           int lvl, uint32_t prefix, uint32_t pmask, int shift,
                                           float nb, uint32_t (*mine)[2]) {
  using L = Lane<T, VEC>;
  const int warp = threadIdx.x >> 5;
  const float cc = p.cc;
  for (int t = 0; t < kMaxChunksPerWarp; ++t) {
    const int cl = warp + kCutWarps * t;
    if (cl >= s.nch) break;
    typename L::Raw raw[L::NV];
    slice_chunk<T, VEC>(p, s, cl, raw);
#pragma unroll
    for (int k = 0; k < L::NV; ++k) {
      int run_bin = -1;
      float run_mass = 0.f;
      uint32_t run_count = 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float v = L::get(raw[k], e);
        if (kKeep && !(v >= keep)) continue;
        const float a = fmaf(v, cc, nb);
        if (kLevel && !(a >= -kCandBits && level_digit(a) == lvl)) continue;
        const uint32_t key = order_key(v);
        if (kPrefix && (key & pmask) != prefix) continue;
        const int bin = (key >> shift) & 255;
        if (bin != run_bin) {
          if (run_bin >= 0) add_to_bin<MASS>(mine, run_bin, run_mass, run_count);
          run_bin = bin;
          run_mass = 0.f;
          run_count = 0;
        }
        if (MASS) run_mass += ex2(a);
        else ++run_count;
      }
      if (run_bin >= 0) add_to_bin<MASS>(mine, run_bin, run_mass, run_count);
    }
  }
}

// Radix descent over the keys of the slice, all CTAs of the cluster
// together.  COUNT: the key of the element of rank `target` from the top.
// MASS: the key of the value class where `front` plus the running mass from
// the top reaches the target; with `from_total` the target is p_q / 2^32 of
// the mass of the elements >= keep, which the first pass sums.  Elements
// below `keep` (and, with lvl >= 0, outside distance level lvl) are ignored.
// Every warp takes each digit itself from the cluster's histogram.
template <typename T, int VEC, bool MASS>
__device__ uint32_t radix_descent(const VerifyParams& p, const Slice<T>& s, float keep, float nb,
                                  int lvl, unsigned long long target, unsigned long long front,
                                  bool from_total, uint32_t p_q, CutShared* sh, int& pass,
                                  int ncta) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int D = sizeof(T) == 2 ? 2 : 4;
  uint32_t prefix = 0, pmask = 0;
  uint32_t(*mine)[2] = sh->part[threadIdx.x >> 5];
  for (int d = 0; d < D; ++d, ++pass) {
    const int shift = 24 - 8 * d;
    const int buf = pass & 1;
    if (lvl >= 0) {
      if (d == 0)
        accumulate<T, VEC, MASS, false, false, true>(p, s, keep, lvl, 0u, 0u, shift, nb, mine);
      else
        accumulate<T, VEC, MASS, true, false, true>(p, s, keep, lvl, prefix, pmask, shift, nb,
                                                    mine);
    } else if (d == 0) {
      if (keep == -INFINITY)
        accumulate<T, VEC, MASS, false, false, false>(p, s, keep, lvl, 0u, 0u, shift, nb, mine);
      else
        accumulate<T, VEC, MASS, false, true, false>(p, s, keep, lvl, 0u, 0u, shift, nb, mine);
    } else {
      accumulate<T, VEC, MASS, true, true, false>(p, s, keep, lvl, prefix, pmask, shift, nb,
                                                  mine);
    }
    __syncthreads();
    publish_hist(sh, buf);
    cluster.sync();  // every CTA's histogram of this pass is complete
    gather_hist(sh, buf, ncta);
    __syncthreads();
    if (MASS && d == 0 && from_total) target = frac_of(warp_hist_total(sh->tot), p_q);
    unsigned long long fr;
    const int digit = pick_digit(sh->tot, front, target, fr);
    front += fr;
    if (!MASS) {  // counts: the target becomes the rank inside the chosen bin
      target -= fr;
      front = 0;
    }
    prefix |= (uint32_t)digit << shift;
    pmask |= 0xffu << shift;
  }
  if (D == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xffffu;  // bf16: the low half of its keys
  return prefix;
}

template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kCutThreads, 4) filter_rows_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  CutShared* sh = reinterpret_cast<CutShared*>(smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int ncta = p.filter_ncta;
  const int rank = (int)cluster.block_rank();
  const int rowid = blockIdx.x / ncta;
  pdl_launch_dependents();
  pdl_wait();
  const int b = (int)fast_div((uint32_t)rowid, p.div_r);
  const int r = rowid - b * p.R;
  const int Kb = p.draft_lens ? __ldg(p.draft_lens + b) : p.K;
  if (!row_needed(p, r, Kb)) return;  // the whole cluster leaves: no barrier is pending
  const int i_pos = r > p.K ? r - p.K - 1 : r;
  const int x = i_pos < Kb ? __ldg(p.draft_tokens + (long long)b * p.K + i_pos) : -1;
  Slice<T> sl;
  sl.row = item_row<T>(p, rowid);
  sl.mrow = item_mask(p, rowid);
  sl.c_lo = min(p.NC, rank * p.filter_cpc);
  sl.nch = min(p.NC, sl.c_lo + p.filter_cpc) - sl.c_lo;
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const bool use_k = p.top_k > 0 && p.top_k < p.V, use_p = p.top_p < 1.f;
  const uint32_t p_q = use_p ? (uint32_t)(p.top_p * 4294967296.f) : 0u;  // top_p * 2^32 (< 1)
  for (int i = threadIdx.x; i < kCutWarps * 256 * 2; i += blockDim.x)
    (&sh->part[0][0][0])[i] = 0u;

  // 1. the row max over the cluster (NaN wins): the slice's one HBM read,
  //    two chunks per warp in flight where a tile is 16 registers (bf16
  //    vectors), one otherwise
  constexpr int kPair = sizeof(typename L::Raw) * L::NV <= 64 ? 2 : 1;
  float lm = -INFINITY;
  for (int t = 0; t < kMaxChunksPerWarp; t += kPair) {
    const int cl0 = warp + kCutWarps * t, cl1 = cl0 + kCutWarps;
    if (cl0 >= sl.nch) break;
    typename L::Raw r0[L::NV], r1[L::NV];
    slice_chunk<T, VEC>(p, sl, cl0, r0);
    if (kPair == 2 && cl1 < sl.nch) slice_chunk<T, VEC>(p, sl, cl1, r1);
    lm = max_nan(lm, tile_max<T, VEC>(r0));
    if (kPair == 2 && cl1 < sl.nch) lm = max_nan(lm, tile_max<T, VEC>(r1));
  }
  lm = warp_max_nan(lm);
  if (lane == 0) sh->red_m[warp] = lm;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = -INFINITY;
    for (int w = 0; w < kCutWarps; ++w) t = max_nan(t, sh->red_m[w]);
    sh->cta_max = t;
  }
  cluster.sync();
  float m = -INFINITY;
  for (int q = 0; q < ncta; ++q) m = max_nan(m, cluster.map_shared_rank(sh, q)->cta_max);
  const float nb = -m * p.cc;

  // 2. the cut value (only for rows with a finite max; others keep their
  //    markers and are reported by the finalize kernel)
  float thr = -INFINITY;
  bool done = false;  // records written (the candidate path)
  if (is_finite(m)) {
    // 2a. the row's mass, its mass outside the candidates, the number of
    //     candidates and their distance-level histogram (counts for top-k,
    //     weights for top-p), summed in a fixed order: every CTA of the
    //     cluster gets the same values and takes the same path
    uint32_t(*mine)[2] = sh->part[warp];
    float s0 = 0.f, s1 = 0.f, tail = 0.f;
    uint32_t cbits[kMaxChunksPerWarp];
#pragma unroll
    for (int t = 0; t < kMaxChunksPerWarp; ++t) cbits[t] = 0u;
#pragma unroll
    for (int t = 0; t < kMaxChunksPerWarp; ++t) {
      const int cl = warp + kCutWarps * t;
      if (cl >= sl.nch) break;
      typename L::Raw raw[L::NV];
      slice_chunk<T, VEC>(p, sl, cl, raw);
      uint32_t bits = 0u;
#pragma unroll
      for (int k = 0; k < L::NV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float a = fmaf(L::get(raw[k], e), p.cc, nb);
          const float w = ex2(a);
          if (e & 1) s1 += w; else s0 += w;
          if (a >= -kCandBits) bits |= 1u << (k * VEC + e);
          else tail += w;
        }
      cbits[t] = bits;
      // the level histogram from the marks (kept out of the loop above,
      // where a rare branch would cost every lane)
      for_each_candidate<T, VEC>(p, sl, cl, bits, [&](int, float v) {
        const float a = fmaf(v, p.cc, nb);
        if (use_k) add_to_bin<false>(mine, level_digit(a), 0.f);
        else add_to_bin<true>(mine, level_digit(a), ex2(a));
      });
    }
    int nc = 0;
#pragma unroll
    for (int t = 0; t < kMaxChunksPerWarp; ++t) nc += __popc(cbits[t]);
    const float s = warp_sum(s0 + s1);
    tail = warp_sum(tail);
    nc = (int)__reduce_add_sync(0xffffffffu, (unsigned)nc);
    if (lane == 0) {
      sh->red_s[warp] = s;
      sh->red_t[warp] = tail;
      sh->red_n[warp] = nc;
    }
    __syncthreads();
    publish_hist(sh, 0);
    if (threadIdx.x == 0) {
      float a = 0.f, tt = 0.f;
      int c = 0;
      for (int w = 0; w < kCutWarps; ++w) {
        a += sh->red_s[w];
        tt += sh->red_t[w];
        c += sh->red_n[w];
      }
      sh->cta_s = a;
      sh->cta_tail = tt;
      sh->cta_n = c;
      sh->list_n = 0;
      sh->best = 0u;
      sh->lowest = 0xffffffffu;
    }
    cluster.sync();
    float S = 0.f, tail_all = 0.f;
    long long n_cand = 0;
    for (int q = 0; q < ncta; ++q) {
      const CutShared* o = cluster.map_shared_rank(sh, q);
      S += o->cta_s;
      tail_all += o->cta_tail;
      n_cand += o->cta_n;
    }
    gather_hist(sh, 0, ncta);
    int pass = 1;
    __syncthreads();
    // 2b. the cut among the candidates when it must lie there: top-k needs
    //     k candidates (the k-th largest is then one); top-p alone needs the
    //     candidates to hold more than top_p of the mass (margin 1e-4 of it
    //     against rounding), so that the crossing class is one of them
    const bool fast = use_k ? n_cand >= p.top_k : tail_all <= (1.f - p.top_p - 1e-4f) * S;
    if (fast) {
      const unsigned long long target =
          use_k ? (unsigned long long)p.top_k
                : frac_of((unsigned long long)(S * 274877906944.f /* 2^38: the fixed-point unit */),
                          p_q);
      unsigned long long above;
      const int lvl = pick_digit(sh->tot, 0ull, target, above);
      // the elements of the cut's level, one list per CTA
#pragma unroll
      for (int t = 0; t < kMaxChunksPerWarp; ++t) {
        const int cl = warp + kCutWarps * t;
        if (cl >= sl.nch) break;
        for_each_candidate<T, VEC>(p, sl, cl, cbits[t], [&](int, float v) {
          const float a = fmaf(v, p.cc, nb);
          if (level_digit(a) == lvl) {
            const int i = atomicAdd(&sh->list_n, 1);
            if (i < kListCap) {
              sh->list_key[i] = order_key(v);
              sh->list_w[i] = use_k ? 1ull : fixed_mass(ex2(a));
            }
          }
        });
      }
      cluster.sync();
      // the cluster's lists, in rank order
      int n_all = 0;
      bool over = false;
      for (int q = 0; q < ncta; ++q) {
        const CutShared* o = cluster.map_shared_rank(sh, q);
        const int nq = o->list_n;
        over = over || nq > kListCap;
        for (int i = threadIdx.x; i < min(nq, kListCap); i += blockDim.x) {
          sh->all_key[n_all + i] = o->list_key[i];
          sh->all_w[n_all + i] = o->list_w[i];
        }
        n_all += min(nq, kListCap);
      }
      __syncthreads();
      uint32_t key;
      if (!over) {
        // the cut's class: the largest key whose class brings the running
        // total from the top to the target (the lowest key if rounding
        // leaves none)
        for (int i = threadIdx.x; i < n_all; i += blockDim.x) {
          const uint32_t ki = sh->all_key[i];
          unsigned long long ge = 0;
          for (int j = 0; j < n_all; ++j)
            if (sh->all_key[j] >= ki) ge += sh->all_w[j];
          if (above + ge >= target) atomicMax(&sh->best, ki);
          atomicMin(&sh->lowest, ki);
        }
        __syncthreads();
        key = sh->best ? sh->best : sh->lowest;
      } else {  // a long level: radix descent inside it
        key = use_k ? radix_descent<T, VEC, false>(p, sl, -INFINITY, nb, lvl, target - above, 0ull,
                                                   false, 0u, sh, pass, ncta)
                    : radix_descent<T, VEC, true>(p, sl, -INFINITY, nb, lvl, target, above, false,
                                                  0u, sh, pass, ncta);
      }
      thr = key_value(key);
      if (use_k && use_p)  // top-p over the elements >= the k-th largest
        thr = key_value(radix_descent<T, VEC, true>(p, sl, thr, nb, -1, 0ull, 0ull, true, p_q, sh,
                                                    pass, ncta));
      // 3. chunk records over the kept elements, which are all candidates:
      //    {max, sum of 2^((l - max) c) leaving out the draft token (one-hot)}
      //    as the streaming kernel writes them
#pragma unroll
      for (int t = 0; t < kMaxChunksPerWarp; ++t) {
        const int cl = warp + kCutWarps * t;
        if (cl >= sl.nch) break;
        float lm2 = -INFINITY;
        for_each_candidate<T, VEC>(p, sl, cl, cbits[t], [&](int, float v) {
          if (v >= thr) lm2 = fmaxf(lm2, v);
        });
        const float cm = warp_max_nan(lm2);
        float cs = 0.f;
        if (cm > -INFINITY) {
          const float nbc = -cm * p.cc;
          for_each_candidate<T, VEC>(p, sl, cl, cbits[t], [&](int j, float v) {
            if (v >= thr && !(MODE == kOneHot && j == x)) cs += ex2(fmaf(v, p.cc, nbc));
          });
        }
        cs = warp_sum(cs);
        if (lane == 0) p.rec[(long long)rowid * p.NC + sl.c_lo + cl] = make_float2(cm, cs);
      }
      if (threadIdx.x == 0 && x >= sl.c_lo * kChunk && x < min(p.V, (sl.c_lo + sl.nch) * kChunk)) {
        const bool allowed = !sl.mrow || ((__ldg(sl.mrow + (x >> 5)) >> (x & 31)) & 1u);
        const float v = load_logit(sl.row, x);
        p.lx[rowid] = (allowed && v >= thr) ? v : -INFINITY;
      }
      done = true;
    } else {
      if (use_k)
        thr = key_value(radix_descent<T, VEC, false>(p, sl, -INFINITY, nb, -1,
                                                     (unsigned long long)p.top_k, 0ull, false, 0u,
                                                     sh, pass, ncta));
      if (use_p)
        thr = key_value(radix_descent<T, VEC, true>(p, sl, thr, nb, -1, 0ull, 0ull, true, p_q, sh,
                                                    pass, ncta));
    }
  }
  // 3. chunk records over the kept elements, as the streaming kernel writes
  //    them (every element read again)
  for (int t = 0; !done && t < kMaxChunksPerWarp; ++t) {
    const int cl = warp + kCutWarps * t;
    if (cl >= sl.nch) break;
    const int c = sl.c_lo + cl;
    typename L::Raw raw[L::NV];
    slice_chunk<T, VEC>(p, sl, cl, raw);
    if (thr > -INFINITY) threshold_chunk<T, VEC>(raw, thr);
    record_draft_logit<T, VEC>(p, raw, c, rowid, x);
    const float2 out = chunk_record<MODE, T, VEC>(raw, c, p.cc, MODE == kOneHot ? x : -1);
    if (lane == 0) p.rec[(long long)rowid * p.NC + c] = out;
  }
  if (rank == 0 && threadIdx.x == 0) p.thr[rowid] = thr;
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_filter(int mode, int dtype, bool vec, const VerifyParams& p, cudaStream_t s) {
  VerifyParams pc = p;
  void* args[] = {&pc};
  const void* fk = nullptr;
  if (mode == kOneHot) {
    if (dtype == kBF16)
      fk = vec ? (const void*)filter_rows_kernel<kOneHot, uint16_t, 8>
               : (const void*)filter_rows_kernel<kOneHot, uint16_t, 1>;
    else
      fk = vec ? (const void*)filter_rows_kernel<kOneHot, float, 4>
               : (const void*)filter_rows_kernel<kOneHot, float, 1>;
  } else if (mode == kDense) {
    if (dtype == kBF16)
      fk = vec ? (const void*)filter_rows_kernel<kDense, uint16_t, 8>
               : (const void*)filter_rows_kernel<kDense, uint16_t, 1>;
    else
      fk = vec ? (const void*)filter_rows_kernel<kDense, float, 4>
               : (const void*)filter_rows_kernel<kDense, float, 1>;
  } else {
    return cudaErrorInvalidValue;  // greedy and typical calls are never filtered
  }
  static PerDevice once[2][2][2];
  const cudaError_t err =
      per_device(once[mode == kDense][dtype == kBF16][vec ? 1 : 0], nullptr, [&](int&) {
        return cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sizeof(CutShared));
      });
  if (err != cudaSuccess) return err;
  return launch_pdl(fk, dim3((unsigned)(p.B * p.R * p.filter_ncta)), dim3(kCutThreads), s, args,
                    sizeof(CutShared), p.filter_ncta);
}

}  // namespace sv
