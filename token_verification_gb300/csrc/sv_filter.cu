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
// and a quantile of the mass, which a single streaming pass cannot give.  So
// a cluster of CTAs holds the whole row in shared memory (one bulk copy per
// CTA slab of up to 64 KB) and makes every further pass there; HBM is still
// read once.  The cut values are found by radix descent on order-preserving
// keys, 8 bits per pass (2 passes for bf16, 4 for fp32): a 256-bin histogram
// per CTA of the elements still matching the key prefix, summed over the
// cluster through distributed shared memory, then one warp picks the bin
// where the running count (top-k) or mass (top-p) from the top reaches the
// target.  Masses are summed as 2^-38 fixed-point integers, so the totals do
// not depend on the order of the atomic adds and every CTA of the cluster
// takes the same decisions.  Finally each warp reduces its chunks to the same
// records kernel A writes, over the kept elements only, and the row's cut
// value goes to the workspace for the finalize kernel's rescans.

constexpr int kFilterThreads = 512;
constexpr int kFilterWarps = kFilterThreads / kWarp;

// Unsigned keys in the order of the values (-0.0 is taken as +0.0).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The 16 bytes of slab group g as fp32 values (8 bf16 or 4 fp32).
template <typename T>
__device__ __forceinline__ void slab_group(const T* slab, int g, float (&v)[16 / sizeof(T)]) {
  const uint4 q = reinterpret_cast<const uint4*>(slab)[g];
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(w[j]);
  }
}

// Shared memory of a filter CTA after its slab (16-byte aligned offsets).
struct FilterShared {
  uint32_t part[kFilterWarps / 2][256][2];  // per warp pair: low / high limbs of each bin
  unsigned long long hist[2][256];  // this CTA's bins, read by the cluster (double-buffered)
  unsigned long long tot[256];      // cluster totals of the current pass
  float red[kFilterWarps];          // block reduction scratch
  float row_max;                    // this CTA's max (read by the cluster)
  int sel_digit;
  unsigned long long sel_front;
};

__host__ __device__ constexpr size_t filter_shared_bytes(int cpc, int esz) {
  return (size_t)cpc * kChunk * esz + sizeof(FilterShared);
}

// Masses are counted in units of 2^-38 of the row's largest probability and
// added as two 19-bit limbs with native 32-bit shared atomics into
// histograms private to a pair of warps (a warp pair sees at most 4096
// elements of a 64 KB slab, so a limb sum stays below 2^31); the limbs are
// recombined exactly into 64-bit totals.
constexpr int kLimbBits = 19;

// floor(w * 2^38) for a weight (or a sum of up to 16 weights) w in [0, 16],
// from the bits of w with integer operations only (w = mant * 2^(e - 150),
// so w * 2^38 = mant * 2^(e - 112)).
__device__ __forceinline__ unsigned long long fixed_mass(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)(b >> 23);
  if (e == 0) return 0ull;  // zero (weights below 2^-126 are flushed)
  const unsigned long long mant = (b & 0x7fffffu) | 0x800000u;
  return e >= 112 ? mant << (e - 112) : (e > 112 - 24 ? mant >> (112 - e) : 0ull);
}

// One warp: the digit whose bin holds the target, scanning bins from 255
// down.  front is the sum of the bins above it; without a bin that reaches
// the target (rounding only) the lowest non-empty bin is taken.
__device__ void pick_digit(const unsigned long long* tot, double base, double target,
                           FilterShared* sh) {
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
  const unsigned hit = __ballot_sync(0xffffffffu, base + (double)incl >= target);
  if (hit) {
    if (lane == __ffs(hit) - 1) {
      unsigned long long acc = excl;
      for (int j = 0; j < 8; ++j) {
        if (base + (double)(acc + part[j]) >= target) {
          sh->sel_digit = 255 - (lane * 8 + j);
          sh->sel_front = acc;
          break;
        }
        acc += part[j];
      }
    }
  } else {
    int low = -1;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (part[j]) low = j;
    const unsigned any = __ballot_sync(0xffffffffu, low >= 0);
    const int l = any ? 31 - __clz(any) : 0;
    if (lane == l) {
      const int j = low < 0 ? 7 : low;
      unsigned long long acc = excl;
      for (int t = 0; t < j; ++t) acc += part[t];
      sh->sel_digit = 255 - (lane * 8 + j);
      sh->sel_front = acc;
    }
  }
}

// Radix descent over the slab's keys, all CTAs of the cluster together.
// COUNT: the key of the k-th largest element (target = k).  MASS: the key of
// the value class where the running mass from the top reaches the target
// (top_p times the total mass of the elements >= keep); `total` receives the
// total in the first pass.  Elements below `keep` are ignored.
// One histogram pass over the slab (see radix_descent).
template <typename T, bool MASS, bool kPrefix, bool kKeep>
__device__ __forceinline__ void accumulate(const T* slab, int n, float keep, uint32_t prefix,
                                           uint32_t pmask, int shift, float cc, float nb,
                                           uint32_t (*mine)[2]) {
  constexpr int E = 16 / (int)sizeof(T);
  int run_bin = -1;
  float run_mass = 0.f;
  uint32_t run_count = 0;
  auto flush = [&]() {
    if (run_bin < 0) return;
    if (MASS) {
      const unsigned long long q = fixed_mass(run_mass);
      atomicAdd(&mine[run_bin][0], (uint32_t)(q & ((1u << kLimbBits) - 1u)));
      atomicAdd(&mine[run_bin][1], (uint32_t)(q >> kLimbBits));
    } else {
      atomicAdd(&mine[run_bin][0], run_count);
    }
  };
  const int groups = (n + E - 1) / E;
  for (int g = threadIdx.x; g < groups; g += blockDim.x) {
    float v[E];
    slab_group<T>(slab, g, v);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (kKeep && !(v[e] >= keep)) continue;
      const uint32_t key = order_key(v[e]);
      if (kPrefix && (key & pmask) != prefix) continue;
      const int bin = (key >> shift) & 255;
      if (bin != run_bin) {
        flush();
        run_bin = bin;
        run_mass = 0.f;
        run_count = 0;
      }
      if (MASS) run_mass += ex2(fmaf(v[e], cc, nb));
      else ++run_count;
    }
    flush();
    run_bin = -1;
  }
}

template <typename T, bool MASS>
__device__ uint32_t radix_descent(const T* slab, int n, float keep, float m, float cc,
                                  double target_or_p, FilterShared* sh, int& pass, int ncta) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int D = sizeof(T) == 2 ? 2 : 4;
  uint32_t prefix = 0, pmask = 0;
  double front = 0.0, target = MASS ? 0.0 : target_or_p;
  const float nb = -m * cc;
  for (int d = 0; d < D; ++d, ++pass) {
    const int shift = 24 - 8 * d;
    const int buf = pass & 1;
    uint32_t* part = &sh->part[0][0][0];
    for (int i = threadIdx.x; i < (kFilterWarps / 2) * 256 * 2; i += blockDim.x) part[i] = 0u;
    __syncthreads();
    uint32_t(*mine)[2] = sh->part[(threadIdx.x >> 5) >> 1];
    // Each thread reads 16-byte groups of consecutive elements and merges
    // runs of elements that fall into the same bin before one atomic per
    // run (a run's mass is summed in fp32, at most 8 weights, then fixed).
    // The slab is padded with -inf to whole groups; the first pass needs no
    // prefix test, and without a top-k cut nothing is below `keep`.
    if (d == 0) {
      if (keep == -INFINITY)
        accumulate<T, MASS, false, false>(slab, n, keep, 0u, 0u, shift, cc, nb, mine);
      else
        accumulate<T, MASS, false, true>(slab, n, keep, 0u, 0u, shift, cc, nb, mine);
    } else {
      accumulate<T, MASS, true, true>(slab, n, keep, prefix, pmask, shift, cc, nb, mine);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      unsigned long long t = 0;
      for (int w = 0; w < kFilterWarps / 2; ++w)
        t += ((unsigned long long)sh->part[w][i][1] << kLimbBits) + sh->part[w][i][0];
      sh->hist[buf][i] = t;
    }
    cluster.sync();  // every CTA's histogram of this pass is complete
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      unsigned long long t = 0;
      for (int r = 0; r < ncta; ++r) t += cluster.map_shared_rank(sh, r)->hist[buf][i];
      sh->tot[i] = t;
    }
    __syncthreads();
    if (MASS && d == 0) {  // the first pass sees every element >= keep
      if (threadIdx.x < kWarp) {
        unsigned long long t = 0;
        for (int i = threadIdx.x; i < 256; i += kWarp) t += sh->tot[i];
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) sh->sel_front = t;
      }
      __syncthreads();
      target = target_or_p * (double)sh->sel_front;
      __syncthreads();
    }
    if (threadIdx.x < kWarp) pick_digit(sh->tot, front, target, sh);
    __syncthreads();
    const int digit = sh->sel_digit;
    front += (double)sh->sel_front;
    if (!MASS) {  // counts: the target becomes the rank inside the chosen bin
      target -= (double)sh->sel_front;
      front = 0.0;
    }
    prefix |= (uint32_t)digit << shift;
    pmask |= 0xffu << shift;
    __syncthreads();
  }
  if (D == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xffffu;  // bf16: the low half of its keys
  return prefix;
}

template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kFilterThreads) filter_rows_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  extern __shared__ __align__(128) unsigned char smem[];
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
  const T* row = item_row<T>(p, rowid);
  const uint32_t* mrow = item_mask(p, rowid);
  const int cpc = p.filter_cpc;
  const int c_lo = min(p.NC, rank * cpc), c_hi = min(p.NC, c_lo + cpc);
  const int e_lo = c_lo * kChunk;
  const int n = max(0, min(p.V, c_hi * kChunk) - e_lo);
  T* slab = reinterpret_cast<T*>(smem);
  FilterShared* sh = reinterpret_cast<FilterShared*>(smem + (size_t)cpc * kChunk * sizeof(T));
  const int lane = lane_id(), warp = threadIdx.x >> 5;

  // 1. the slab: one bulk copy on the vector path, plain loads otherwise
  if constexpr (VEC * sizeof(T) == 16) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t bar_a = smem_u32(&bar);
    if (threadIdx.x == 0) {
      mbar_init(bar_a, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      if (n > 0)
        bulk_load(smem_u32(slab), row + e_lo, (uint32_t)(n * sizeof(T)), bar_a);
      else
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_a) : "memory");
    }
    // one thread waits for the copy (bounded); the barrier below passes the
    // completed bytes on to the rest of the CTA
    if (threadIdx.x == 0 && !mbar_wait(bar_a, 0)) atomicOr(p.err, 1);
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) slab[i] = row[e_lo + i];
  }
  __syncthreads();
  // the slab's last 16-byte group is completed with -inf (no mass, and
  // below every real logit, so no pass is changed by it)
  {
    constexpr int E = 16 / (int)sizeof(T);
    const int padded = (n + E - 1) / E * E;
    for (int i = n + threadIdx.x; i < padded; i += blockDim.x) {
      if constexpr (sizeof(T) == 2) slab[i] = (T)0xff80u;
      else slab[i] = -INFINITY;
    }
    __syncthreads();
  }
  // 2. grammar mask: disallowed logits become -inf
  if (mrow) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int j = e_lo + i;
      if (!((__ldg(mrow + (j >> 5)) >> (j & 31)) & 1u)) {
        if constexpr (sizeof(T) == 2) slab[i] = (T)0xff80u;
        else slab[i] = -INFINITY;
      }
    }
    __syncthreads();
  }
  // 3. the row's max over the cluster (NaN wins)
  float lm = -INFINITY;
  {
    constexpr int E = 16 / (int)sizeof(T);
    for (int g = threadIdx.x; g * E < n; g += blockDim.x) {
      float v[E];
      slab_group<T>(slab, g, v);
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (g * E + e < n) lm = max_nan(lm, v[e]);
    }
  }
  lm = warp_max_nan(lm);
  if (lane == 0) sh->red[warp] = lm;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = -INFINITY;
    for (int w = 0; w < kFilterWarps; ++w) t = max_nan(t, sh->red[w]);
    sh->row_max = t;
  }
  cluster.sync();
  float m = -INFINITY;
  for (int q = 0; q < ncta; ++q) m = max_nan(m, cluster.map_shared_rank(sh, q)->row_max);
  // 4. the cut value (only for rows with a finite max; others keep their
  //    markers and are reported by the finalize kernel)
  float thr = -INFINITY;
  int pass = 0;
  if (is_finite(m)) {
    if (p.top_k > 0 && p.top_k < p.V)
      thr = key_value(radix_descent<T, false>(slab, n, -INFINITY, m, p.cc, (double)p.top_k, sh,
                                              pass, ncta));
    if (p.top_p < 1.f)
      thr = key_value(radix_descent<T, true>(slab, n, thr, m, p.cc, (double)p.top_p, sh, pass,
                                             ncta));
  }
  // 5. chunk records over the kept elements, as kernel A writes them
  for (int cl = warp; cl < c_hi - c_lo; cl += kFilterWarps) {
    const int c = c_lo + cl;
    typename L::Raw raw[L::NV];
    const T* base = slab + cl * kChunk;
#pragma unroll
    for (int k = 0; k < L::NV; ++k) {
      const int off = tile_offset<VEC>(k, 0, lane);
      raw[k] = (c * kChunk + off < p.V) ? *reinterpret_cast<const typename L::Raw*>(base + off)
                                        : L::pad();
    }
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
                                    (int)(kFilterSlabBytes + sizeof(FilterShared)));
      });
  if (err != cudaSuccess) return err;
  return launch_pdl(fk, dim3((unsigned)(p.B * p.R * p.filter_ncta)), dim3(kFilterThreads), s,
                    args, filter_shared_bytes(p.filter_cpc, dtype == kBF16 ? 2 : 4),
                    p.filter_ncta);
}

}  // namespace sv
