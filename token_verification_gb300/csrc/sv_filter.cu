// sv_filter.cu - kernel A for top-k / top-p filtered verification calls.
#include "sv_rows.cuh"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// kernel A for top-k / top-p calls: one row per CTA
// ---------------------------------------------------------------------------
//
// Filtering needs, per row, the k-th largest logit and the value at which
// the mass of the leading value classes reaches top_p - an order statistic
// and a quantile of the mass, which a single streaming pass cannot give.  One
// CTA takes one row (filtered rows are at most 512 KB): it reads the row from
// HBM once, for the row max m, and its later passes find the row in L2, so
// shared memory holds only histograms, candidate marks and a short list, and
// two rows are in flight per SM.
//
// With m known, the weights w = 2^((l - m) c) follow.  Candidates are the
// elements within 2^-18 of the max's weight (kCandBits); every element above
// a candidate is one.  One pass sums the row's mass, the mass outside the candidates,
// marks the candidates and histograms them over distance levels (eighths of
// a bit of weight below the max: a level is a range of values).  When the cut
// must lie among the candidates - at least k of them for top-k; for top-p
// more than top_p of the mass in them - the level holding the cut follows
// from the histogram, the elements of that one level are gathered into a
// list, and the cut's value class is found in it.  Otherwise (a flat row, a
// large k, a long level) a radix descent on order-preserving keys finds it,
// 8 bits per pass.  Masses are summed as 2^-38 fixed-point integers, so the
// decisions do not depend on the order of the atomic adds.  Finally each
// warp reduces its chunks to the same records the streaming kernel writes,
// over the kept elements only (from the candidate marks when every kept
// element is a candidate), and the row's cut value goes to the workspace for
// the finalize kernel's rescans.

constexpr int kCutThreads = 512;
constexpr int kCutWarps = kCutThreads / kWarp;
constexpr int kMaxChunks = kFilterRowBytes / (kChunk * 2);  // bf16 rows of up to 512 KB
constexpr int kListCap = 512;     // elements of the cut's level
constexpr float kCandBits = 18.f;  // candidates: weight >= 2^-18 of the max's
constexpr int kStageBytes = 4096;  // per warp: its candidates' logits
constexpr int kLimbBits = 13;      // three limbs: a warp pair's bin sums stay below 2^28

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

// The least value v of type T (bf16 as its float value) with fmaf(v, c,
// -m c) >= -kCandBits: every element at or above it is a candidate, none
// below.  The float bound m - kCandBits / c is moved by single steps of T's
// spacing until it is the least one (fmaf is monotone in v).
template <typename T>
__device__ float cand_bound(float m, float cc) {
  const float nb = -m * cc;
  auto ok = [&](float v) { return fmaf(v, cc, nb) >= -kCandBits; };
  auto up = [](float v) {  // the next value of T above v
    if (sizeof(T) == 2) {
      const uint32_t b = __float_as_uint(v) >> 16;
      const uint32_t n = (b & 0x8000u) ? (b == 0x8000u ? 0x0001u : b - 1u) : b + 1u;
      return __uint_as_float(n << 16);
    }
    return nextafterf(v, INFINITY);
  };
  auto down = [](float v) {
    if (sizeof(T) == 2) {
      const uint32_t b = __float_as_uint(v) >> 16;
      const uint32_t n = (b & 0x8000u) ? b + 1u : (b == 0u ? 0x8001u : b - 1u);
      return __uint_as_float(n << 16);
    }
    return nextafterf(v, -INFINITY);
  };
  float v = m - kCandBits / cc;
  if (sizeof(T) == 2) v = __uint_as_float(__float_as_uint(v) & 0xffff0000u);  // toward zero
  if (!(v >= -FLT_MAX))  // every finite element is a candidate: the least finite value
    return sizeof(T) == 2 ? __uint_as_float(0xff7f0000u) : -FLT_MAX;
  for (int i = 0; i < 64 && !ok(v); ++i) v = up(v);
  for (int i = 0; i < 64 && ok(down(v)); ++i) v = down(v);
  return v;
}

// Both halves of a bf16 pair set to v (a bf16 value held as a float).
__device__ __forceinline__ uint32_t bf16_pair_of(float v) {
  const uint32_t h = __float_as_uint(v) >> 16;
  return h | (h << 16);
}

// Sets bit POS of `bits` if the low bf16 of w is >= the threshold's, bit
// POS + 1 if the high one is: one packed comparison (its first predicate
// is the low halves') and two predicated ORs; -inf and NaN never pass.
template <int POS>
__device__ __forceinline__ void mark_ge_bf16x2(uint32_t& bits, uint32_t w, uint32_t t2) {
  asm("{\n\t.reg .pred p, q;\n\t"
      "setp.ge.bf16x2 p|q, %1, %2;\n\t"
      "@p or.b32 %0, %0, %3;\n\t@q or.b32 %0, %0, %4;\n\t}"
      : "+r"(bits)
      : "r"(w), "r"(t2), "n"(1u << POS), "n"(2u << POS));
}

template <int K>
__device__ __forceinline__ void mark_group_bf16(uint32_t& bits, const uint4& g, uint32_t t2) {
  mark_ge_bf16x2<8 * K + 0>(bits, g.x, t2);
  mark_ge_bf16x2<8 * K + 2>(bits, g.y, t2);
  mark_ge_bf16x2<8 * K + 4>(bits, g.z, t2);
  mark_ge_bf16x2<8 * K + 6>(bits, g.w, t2);
}

// Distance levels: a candidate's weight exponent a = (l - m) c in [-18, 0]
// falls into level floor(-8 a), kept as digit 255 - level so that larger
// values have larger digits, as key digits do.
__device__ __forceinline__ int level_digit(float a) { return 255 - __float2int_rz(-8.f * a); }

// Shared memory of a filter CTA.  Histograms per warp pair, of three 13-bit
// limbs (a warp pair sees at most 2^15 elements, so a limb sum stays below
// 2^28; three 32-bit atomics cost less than one 64-bit one).  Each warp stages the logits of its candidates in (chunk, lane,
// element) order; chunk c's run starts at seg[c] in the stage of warp c % 16.
struct CutShared {
  uint32_t part[kCutWarps / 2][256][3];  // per warp pair: limbs of each bin (counts: [0])
  unsigned long long tot[256];           // the CTA's bins
  unsigned char stage[kCutWarps][kStageBytes];
  int seg[kMaxChunks], seg_n[kMaxChunks];
  int stage_n[kCutWarps];
  float red_t[kCutWarps];
  int red_n[kCutWarps];
  float2 rec1[kMaxChunks];  // per chunk {max, sum of 2^((l - max) c)} over the whole chunk
  float row_max, row_s, row_tail, cand_lo;
  int row_n, over, x_entry;
  int list_n;  // elements of the cut's level
  uint32_t list_key[kListCap];
  unsigned long long list_w[kListCap];
  uint32_t best, lowest;
};

__device__ __forceinline__ float stage_value(const uint16_t* st, int i) {
  return __uint_as_float((uint32_t)st[i] << 16);
}
__device__ __forceinline__ float stage_value(const float* st, int i) { return st[i]; }
__device__ __forceinline__ uint16_t stage_bits(float v, const uint16_t*) {
  return (uint16_t)(__float_as_uint(v) >> 16);
}
__device__ __forceinline__ float stage_bits(float v, const float*) { return v; }

// Adds one element's weight w (MASS: as a fixed-point mass) or a count of
// `n` to bin `bin` of a warp pair's histogram.
template <bool MASS>
__device__ __forceinline__ void add_to_bin(uint32_t (*mine)[3], int bin, float w, uint32_t n = 1) {
  if (MASS) {
    const unsigned long long q = fixed_mass(w);
    constexpr uint32_t kMask = (1u << kLimbBits) - 1u;
    atomicAdd(&mine[bin][0], (uint32_t)q & kMask);
    atomicAdd(&mine[bin][1], (uint32_t)(q >> kLimbBits) & kMask);
    atomicAdd(&mine[bin][2], (uint32_t)(q >> (2 * kLimbBits)));
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

// The warps' histograms (limbs recombined) into tot, cleared for the next
// pass as they are read.  Between two __syncthreads.
__device__ __forceinline__ void combine_hist(CutShared* sh) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < kCutWarps / 2; ++w) {
      t += (unsigned long long)sh->part[w][i][0] +
           ((unsigned long long)sh->part[w][i][1] << kLimbBits) +
           ((unsigned long long)sh->part[w][i][2] << (2 * kLimbBits));
      sh->part[w][i][0] = sh->part[w][i][1] = sh->part[w][i][2] = 0u;
    }
    sh->tot[i] = t;
  }
}

// The sum of the histogram, by every lane of the calling warp.
__device__ __forceinline__ unsigned long long warp_hist_total(const unsigned long long* tot) {
  unsigned long long t = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) t += tot[lane_id() * 8 + j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// The row and its grammar mask; warp w takes chunks w + 16 t.
template <typename T>
struct Slice {
  const T* row;
  const uint32_t* mrow;
  int nch;
};

// Chunk c of the row as this lane's register tile (disallowed tokens -inf;
// groups past V the -inf pad).  Warp-wide.
template <typename T, int VEC>
__device__ __forceinline__ void row_chunk(const VerifyParams& p, const Slice<T>& s, int c,
                                          typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV]) {
  load_chunk<T, VEC>(s.row, p.V, c, raw);
  if (s.mrow) allow_only_chunk<T, VEC>(raw, mask_word(s.mrow, p.mask_words, c));
}

// Element t (bit t of the candidate marks: group t / 8, element t % 8) of a
// lane's bf16 tile, as its 16 bits.
__device__ __forceinline__ uint16_t tile_bf16(const uint4 (&raw)[4], int t) {
  const uint4 r01 = (t & 8) ? raw[1] : raw[0];
  const uint4 r23 = (t & 8) ? raw[3] : raw[2];
  const uint4 rk = (t & 16) ? r23 : r01;
  const uint32_t w01 = (t & 2) ? rk.y : rk.x;
  const uint32_t w23 = (t & 2) ? rk.w : rk.z;
  const uint32_t wq = (t & 4) ? w23 : w01;
  return (uint16_t)((t & 1) ? (wq >> 16) : (wq & 0xffffu));
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

// One radix pass over the row (see radix_descent): elements >= keep
// (kKeep) with the key prefix so far (kPrefix).  Runs of consecutive
// elements of a lane that fall into the same bin are merged before one
// atomic (a run's mass summed in fp32, at most VEC weights, then fixed).
template <typename T, int VEC, bool MASS, bool kPrefix, bool kKeep>
__device__ __forceinline__ void accumulate(const VerifyParams& p, const Slice<T>& s, float keep,
                                           uint32_t prefix, uint32_t pmask, int shift, float nb,
                                           uint32_t (*mine)[3]) {
  using L = Lane<T, VEC>;
  const float cc = p.cc;
  for (int c = threadIdx.x >> 5; c < s.nch; c += kCutWarps) {
    typename L::Raw raw[L::NV];
    row_chunk<T, VEC>(p, s, c, raw);
#pragma unroll
    for (int k = 0; k < L::NV; ++k) {
      int run_bin = -1;
      float run_mass = 0.f;
      uint32_t run_count = 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float v = L::get(raw[k], e);
        if (kKeep && !(v >= keep)) continue;
        const uint32_t key = order_key(v);
        if (kPrefix && (key & pmask) != prefix) continue;
        const int bin = (key >> shift) & 255;
        if (bin != run_bin) {
          if (run_bin >= 0) add_to_bin<MASS>(mine, run_bin, run_mass, run_count);
          run_bin = bin;
          run_mass = 0.f;
          run_count = 0;
        }
        if (MASS) run_mass += ex2(fmaf(v, cc, nb));
        else ++run_count;
      }
      if (run_bin >= 0) add_to_bin<MASS>(mine, run_bin, run_mass, run_count);
    }
  }
}

// Radix descent over the keys of the whole row (rows whose cut may lie
// outside the candidates).  COUNT: the key of the element of rank `target`
// from the top.  MASS: the key of the value class where the running mass
// from the top reaches p_q / 2^32 of the mass of the elements >= keep, which
// the first pass sums.  Elements below `keep` are ignored.  Every warp takes
// each digit itself from the histogram.
template <typename T, int VEC, bool MASS>
__device__ uint32_t radix_descent(const VerifyParams& p, const Slice<T>& s, float keep, float nb,
                                  unsigned long long target, uint32_t p_q, CutShared* sh) {
  constexpr int D = sizeof(T) == 2 ? 2 : 4;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long front = 0;
  uint32_t(*mine)[3] = sh->part[threadIdx.x >> 6];
  for (int d = 0; d < D; ++d) {
    const int shift = 24 - 8 * d;
    if (d == 0) {
      if (keep == -INFINITY)
        accumulate<T, VEC, MASS, false, false>(p, s, keep, 0u, 0u, shift, nb, mine);
      else
        accumulate<T, VEC, MASS, false, true>(p, s, keep, 0u, 0u, shift, nb, mine);
    } else {
      accumulate<T, VEC, MASS, true, true>(p, s, keep, prefix, pmask, shift, nb, mine);
    }
    __syncthreads();
    combine_hist(sh);
    __syncthreads();
    if (MASS && d == 0) target = frac_of(warp_hist_total(sh->tot), p_q);
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

// The cut among the staged candidates: the distance-level histogram of the
// candidates >= keep (counts, or fixed-point weights for MASS), the level
// where the running total from the top reaches the target (with
// `from_total`: p_q / 2^32 of their total mass), the list of that level's
// elements, and in it the largest key whose class brings the total to the
// target (the lowest key if rounding leaves none).  False when the level
// holds more than kListCap elements.  Called by every thread.
template <typename T, bool MASS>
__device__ bool stage_cut(CutShared* sh, float keep, float cc, float nb, unsigned long long target,
                          bool from_total, uint32_t p_q, uint32_t& key) {
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t(*mine)[3] = sh->part[warp >> 1];
  const T* st = reinterpret_cast<const T*>(sh->stage[warp]);
  const int n_w = sh->stage_n[warp];
  if (threadIdx.x == 0) {
    sh->list_n = 0;
    sh->best = 0u;
    sh->lowest = 0xffffffffu;
  }
  for (int i = lane; i < n_w; i += kWarp) {
    const float v = stage_value(st, i);
    if (!(v >= keep)) continue;
    const float a = fmaf(v, cc, nb);
    add_to_bin<MASS>(mine, level_digit(a), MASS ? ex2(a) : 0.f);
  }
  __syncthreads();
  combine_hist(sh);
  __syncthreads();
  if (MASS && from_total) target = frac_of(warp_hist_total(sh->tot), p_q);
  unsigned long long above;
  const int lvl = pick_digit(sh->tot, 0ull, target, above);
  for (int i = lane; i < n_w; i += kWarp) {
    const float v = stage_value(st, i);
    if (!(v >= keep)) continue;
    const float a = fmaf(v, cc, nb);
    if (level_digit(a) == lvl) {
      const int j = atomicAdd(&sh->list_n, 1);
      if (j < kListCap) {
        sh->list_key[j] = order_key(v);
        sh->list_w[j] = MASS ? fixed_mass(ex2(a)) : 1ull;
      }
    }
  }
  __syncthreads();
  const int n_all = sh->list_n;
  if (n_all > kListCap) return false;
  for (int i = threadIdx.x; i < n_all; i += blockDim.x) {
    const uint32_t ki = sh->list_key[i];
    unsigned long long ge = 0;
    for (int j = 0; j < n_all; ++j)
      if (sh->list_key[j] >= ki) ge += sh->list_w[j];
    if (above + ge >= target) atomicMax(&sh->best, ki);
    atomicMin(&sh->lowest, ki);
  }
  __syncthreads();
  key = sh->best ? sh->best : sh->lowest;
  __syncthreads();  // before a second call resets the list
  return true;
}

template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kCutThreads, 2) filter_rows_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  CutShared* sh = reinterpret_cast<CutShared*>(smem);
  const int rowid = blockIdx.x;
  // Launched early (programmatic dependent launch): wait for the predecessor,
  // then let the finalize kernel launch - it reads the call's inputs before
  // its own wait, which is safe once everything before this kernel is done.
  pdl_wait();
  pdl_launch_dependents();
  const int b = (int)fast_div((uint32_t)rowid, p.div_r);
  const int r = rowid - b * p.R;
  const int Kb = p.draft_lens ? __ldg(p.draft_lens + b) : p.K;
  if (!row_needed(p, r, Kb)) return;
  const int i_pos = r > p.K ? r - p.K - 1 : r;
  const int x = i_pos < Kb ? __ldg(p.draft_tokens + (long long)b * p.K + i_pos) : -1;
  Slice<T> sl;
  sl.row = item_row<T>(p, rowid);
  sl.mrow = item_mask(p, rowid);
  sl.nch = p.NC;
  // the draft token's logit (and whether the mask allows it), loaded now and
  // used at the end
  float x_logit = -INFINITY;
  if (threadIdx.x == 0 && x >= 0 && x < p.V) {
    const bool allowed = !sl.mrow || ((__ldg(sl.mrow + (x >> 5)) >> (x & 31)) & 1u);
    if (allowed) x_logit = load_logit(sl.row, x);
  }
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const bool use_k = p.top_k > 0 && p.top_k < p.V, use_p = p.top_p < 1.f;
  const uint32_t p_q = use_p ? (uint32_t)(p.top_p * 4294967296.f) : 0u;  // top_p * 2^32 (< 1)
  for (int i = threadIdx.x; i < (kCutWarps / 2) * 256 * 3; i += blockDim.x)
    (&sh->part[0][0][0])[i] = 0u;

  // 1. per chunk its max and the sum of 2^((l - max_c) c), as the streaming
  //    kernel's records - the row's one HBM read.  On the vector paths each
  //    warp first asks L2 for all of its chunks (bulk prefetches), so the
  //    whole row is in flight at once; two chunks per warp are loaded at a
  //    time where a tile is 16 registers (bf16 vectors), one otherwise.  The
  //    row max (NaN wins) and the row's mass in its frame follow from them.
  constexpr int kPair = L::NV * ((sizeof(typename L::Raw) + 3) / 4) <= 16 ? 2 : 1;  // registers
  if (VEC * sizeof(T) == 16 && lane == 0)
    for (int c = warp; c < sl.nch; c += kCutWarps)
      prefetch_l2(sl.row + c * kChunk, (uint32_t)(min(kChunk, p.V - c * kChunk) * sizeof(T)));
  auto no_exclusion = [](typename L::Raw(&)[L::NV]) {};
  for (int c0 = warp; c0 < sl.nch; c0 += kPair * kCutWarps) {
    const int c1 = c0 + kCutWarps;
    typename L::Raw r0[L::NV], r1[L::NV];
    row_chunk<T, VEC>(p, sl, c0, r0);
    if (kPair == 2 && c1 < sl.nch) row_chunk<T, VEC>(p, sl, c1, r1);
    const float2 q0 = chunk_softmax_ex<T, VEC>(r0, p.cc, no_exclusion);
    if (lane == 0) sh->rec1[c0] = q0;
    if (kPair == 2 && c1 < sl.nch) {
      const float2 q1 = chunk_softmax_ex<T, VEC>(r1, p.cc, no_exclusion);
      if (lane == 0) sh->rec1[c1] = q1;
    }
  }
  __syncthreads();
  if (warp == 0) {
    float mm = -INFINITY;
    for (int c = lane; c < sl.nch; c += kWarp) mm = max_nan(mm, sh->rec1[c].x);
    mm = warp_max_nan(mm);
    float a = 0.f;
    if (is_finite(mm))
      for (int c = lane; c < sl.nch; c += kWarp) {
        const float2 r = sh->rec1[c];
        if (r.x > -INFINITY) a = fmaf(r.y, ex2((r.x - mm) * p.cc), a);
      }
    a = warp_sum(a);
    if (lane == 0) {
      sh->row_max = mm;
      sh->row_s = a;
      sh->over = 0;
      sh->x_entry = -1;
      // the candidates' bound: the least value v with fmaf(v, c, -m c) >=
      // -18, as a value of the row's type (compared raw in pass 2)
      if (is_finite(mm)) sh->cand_lo = cand_bound<T>(mm, p.cc);
    }
  }
  __syncthreads();
  const float m = sh->row_max;
  const float nb = -m * p.cc;

  // 2. the cut value (only for rows with a finite max; others keep their
  //    markers and are reported by the finalize kernel)
  float thr = -INFINITY;
  bool done = false;  // records written (the candidate path)
  if (is_finite(m)) {
    // 2a. the candidates - the elements within 2^-18 of the max's weight -
    //     marked by a comparison with their bound, the row re-read from L2;
    //     each warp stages its candidates' logits (a warp whose stage fills
    //     up sends the row down the full-row path), then the candidates'
    //     mass; the mass outside them is the row's mass less theirs
    constexpr int kCap = kStageBytes / (int)sizeof(T);
    constexpr bool kPacked = sizeof(T) == 2 && VEC == 8;
    T* st = reinterpret_cast<T*>(sh->stage[warp]);
    const float lo = sh->cand_lo;
    const uint32_t lo2 = kPacked ? bf16_pair_of(lo) : 0u;
    int base = 0;
    bool over = false;
    // (bf16 vectors: the next chunk's load is issued before this one is
    // marked, into the other of two tiles)
    constexpr bool kPipe = kPair == 2;
    auto mark_and_stage = [&](typename L::Raw(&raw)[L::NV], int c) {
      uint32_t bits = 0u;
      if constexpr (kPacked) {  // the tile's 4 groups of 8 (bit 8 k + e: group k, element e)
        mark_group_bf16<0>(bits, raw[0], lo2);
        mark_group_bf16<1>(bits, raw[1], lo2);
        mark_group_bf16<2>(bits, raw[2], lo2);
        mark_group_bf16<3>(bits, raw[3], lo2);
      } else {
#pragma unroll
        for (int k = 0; k < L::NV; ++k)
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (L::get(raw[k], e) >= lo) bits |= 1u << (k * VEC + e);
      }
      const int cnt = __popc(bits);
      const int incl = warp_incl_scan_int(cnt);
      const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
      if (!over && base + total <= kCap) {
        int q = base + incl - cnt;  // the lane's candidates in element order
        if constexpr (kPacked) {
          for (uint32_t bb = bits; bb; bb &= bb - 1u) st[q++] = tile_bf16(raw, __ffs(bb) - 1);
        } else {
#pragma unroll
          for (int k = 0; k < L::NV; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              if ((bits >> (k * VEC + e)) & 1u) st[q++] = stage_bits(L::get(raw[k], e), st);
        }
        const int xo = x - c * kChunk;  // the draft token's entry, if it is a candidate here
        if (MODE == kOneHot && xo >= 0 && xo < kChunk && lane == (xo / VEC) % kWarp) {
          const int pos = (xo / (kWarp * VEC)) * VEC + xo % VEC;
          if ((bits >> pos) & 1u) sh->x_entry = base + incl - cnt + __popc(bits & ((1u << pos) - 1u));
        }
        if (lane == 0) {
          sh->seg[c] = base;
          sh->seg_n[c] = total;
        }
        base += total;
      } else {
        over = true;
      }
    };
    typename L::Raw ra[L::NV], rb[L::NV];
    if (kPipe) {
      if (warp < sl.nch) row_chunk<T, VEC>(p, sl, warp, ra);
      for (int c = warp; c < sl.nch; c += 2 * kCutWarps) {
        const int c1 = c + kCutWarps;
        if (c1 < sl.nch) row_chunk<T, VEC>(p, sl, c1, rb);
        mark_and_stage(ra, c);
        if (c1 < sl.nch) {
          if (c1 + kCutWarps < sl.nch) row_chunk<T, VEC>(p, sl, c1 + kCutWarps, ra);
          mark_and_stage(rb, c1);
        }
      }
    } else {
      for (int c = warp; c < sl.nch; c += kCutWarps) {
        row_chunk<T, VEC>(p, sl, c, ra);
        mark_and_stage(ra, c);
      }
    }
    float sc = 0.f;  // the staged candidates' mass
    if (!over)
      for (int i = lane; i < base; i += kWarp) sc += ex2(fmaf(stage_value(st, i), p.cc, nb));
    sc = warp_sum(sc);
    if (lane == 0) {
      sh->red_t[warp] = sc;
      sh->red_n[warp] = base;
      sh->stage_n[warp] = base;
      if (over) sh->over = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float tt = 0.f;
      int n = 0;
      for (int w = 0; w < kCutWarps; ++w) {
        tt += sh->red_t[w];
        n += sh->red_n[w];
      }
      sh->row_tail = sh->row_s - tt;
      sh->row_n = n;
    }
    __syncthreads();
    const float S = sh->row_s;
    // 2b. the cut among the candidates when it must lie there: top-k needs
    //     k candidates (the k-th largest is then one); top-p alone needs the
    //     candidates to hold more than top_p of the mass (margin 1e-4 of it
    //     against rounding), so that the crossing class is one of them
    bool fast = !sh->over &&
                (use_k ? sh->row_n >= p.top_k : sh->row_tail <= (1.f - p.top_p - 1e-4f) * S);
    if (fast) {
      uint32_t key;
      if (use_k) {
        fast = stage_cut<T, false>(sh, -INFINITY, p.cc, nb, (unsigned long long)p.top_k, false, 0u,
                                   key);
        if (fast && use_p)  // top-p over the elements >= the k-th largest
          fast = stage_cut<T, true>(sh, key_value(key), p.cc, nb, 0ull, true, p_q, key);
      } else {
        fast = stage_cut<T, true>(
            sh, -INFINITY, p.cc, nb,
            frac_of((unsigned long long)(S * 274877906944.f /* 2^38: the fixed-point unit */), p_q),
            false, 0u, key);
      }
      if (fast) {
        thr = key_value(key);
        // 3. chunk records over the kept elements, which are all staged:
        //    {max, sum of 2^((l - max) c) leaving out the draft token
        //    (one-hot)} as the streaming kernel writes them
        // Warp w takes its own chunks (w + 16 t), whose runs are in its
        // stage: the run's first 32 values are held one per lane (the rest,
        // in long runs, are read again), the max comes from one warp-wide
        // reduction of order keys, the sum from a fixed-order warp sum.
        const int x_entry = sh->x_entry;
        const int xc = (MODE == kOneHot && x >= 0 && x < p.V) ? x / kChunk : -1;
        const T* cst = reinterpret_cast<const T*>(sh->stage[warp]);
        for (int c = warp; c < sl.nch; c += kCutWarps) {
          const int b0 = sh->seg[c], n0 = sh->seg_n[c];
          const float v0 = lane < n0 ? stage_value(cst, b0 + lane) : -INFINITY;
          uint32_t kmax = v0 >= thr ? order_key(v0) : 0u;
          for (int i = lane + kWarp; i < n0; i += kWarp) {
            const float v = stage_value(cst, b0 + i);
            if (v >= thr) kmax = max(kmax, order_key(v));
          }
          kmax = __reduce_max_sync(0xffffffffu, kmax);
          const float cm = kmax ? key_value(kmax) : -INFINITY;
          float cs = 0.f;
          if (kmax) {
            const float nbc = -cm * p.cc;
            const int skip = (c == xc ? x_entry : -1) - b0;  // its place in the run
            if (v0 >= thr && lane != skip) cs = ex2(fmaf(v0, p.cc, nbc));
            for (int i = lane + kWarp; i < n0; i += kWarp) {
              const float v = stage_value(cst, b0 + i);
              if (v >= thr && i != skip) cs += ex2(fmaf(v, p.cc, nbc));
            }
            cs = warp_sum(cs);
          }
          if (lane == 0) p.rec[(long long)rowid * p.NC + c] = make_float2(cm, cs);
        }
        if (threadIdx.x == 0 && x >= 0 && x < p.V) p.lx[rowid] = x_logit >= thr ? x_logit : -INFINITY;
        done = true;
      }
    }
    if (!fast) {  // the full-row path: radix descent over every element
      if (use_k)
        thr = key_value(radix_descent<T, VEC, false>(p, sl, -INFINITY, nb,
                                                     (unsigned long long)p.top_k, 0u, sh));
      if (use_p) thr = key_value(radix_descent<T, VEC, true>(p, sl, thr, nb, 0ull, p_q, sh));
    }
  }
  // 3. chunk records over the kept elements, as the streaming kernel writes
  //    them (every element read again)
  for (int c = warp; !done && c < sl.nch; c += kCutWarps) {
    typename L::Raw raw[L::NV];
    row_chunk<T, VEC>(p, sl, c, raw);
    if (thr > -INFINITY) threshold_chunk<T, VEC>(raw, thr);
    record_draft_logit<T, VEC>(p, raw, c, rowid, x);
    const float2 out = chunk_record<MODE, T, VEC>(raw, c, p.cc, MODE == kOneHot ? x : -1);
    if (lane == 0) p.rec[(long long)rowid * p.NC + c] = out;
  }
  if (threadIdx.x == 0) p.thr[rowid] = thr;
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
  return launch_pdl(fk, dim3((unsigned)(p.B * p.R)), dim3(kCutThreads), s, args,
                    sizeof(CutShared));
}

}  // namespace sv
