// sv_common.cuh - device building blocks shared by the verification kernels.
//
// Data layout.  A logit row (one request, one position) of V elements is cut
// into chunks of kChunk = 1024 elements.  One warp reduces one chunk: lane l
// holds 32 elements, in NV groups of VEC consecutive elements; group k of lane
// l starts at element k*32*VEC + l*VEC of the chunk, so each group load of the
// warp covers 32*VEC consecutive elements (coalesced 128-bit loads for the
// vector paths).  A chunk reduces to one record (float2): for softmax rows
// {chunk max m_c, sum of 2^((l_j - m_c) * c)} with c = log2(e) / T, for argmax
// rows {chunk max, lowest index attaining it}.
//
// The vector paths need V to be a multiple of VEC and a 16-byte aligned base
// pointer (then every row start is 16-byte aligned); otherwise the scalar path
// (VEC = 1) is used.  Elements past V are padded with -inf, which never wins
// a max and contributes 2^-inf = 0 to a sum.
#pragma once

#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

namespace sv {

constexpr int kWarp = 32;
constexpr int kChunk = 1024;           // elements per chunk record
constexpr int kThreads = 256;          // threads per CTA of the streaming kernels
constexpr int kMaxK = 31;              // K + 1 <= 32: one lane per position
constexpr float kLog2e = 1.4426950408889634f;

// per-request status bits (the public SV_REQ_* values)
constexpr int kBadToken = 1;
constexpr int kBadLogits = 2;
constexpr int kBadDraftLen = 4;
constexpr int kTimeout = 8;
constexpr int kBadTree = 16;

enum Mode : int { kOneHot = 0, kDense = 1, kGreedy = 2, kTypical = 3, kTreeSample = 4 };

// ---------------------------------------------------------------------------
// scalar primitives
// ---------------------------------------------------------------------------

__device__ __forceinline__ int lane_id() { return threadIdx.x & (kWarp - 1); }

// 2^x on the SFU; ex2.approx.ftz: relative error about 2^-22, 2^-inf = +0,
// results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The factor that moves a sum of 2^(l c - fl(m c)) - a chunk record's
// weights, each in the frame of its own rounded offset fl(m c) - into the
// frame fl(M c) of a larger maximum M: 2^(fl(m c) - fl(M c)), the difference
// of the two rounded offsets (exact when they are within a factor of two).
// 2^(fmaf(m, c, -fl(M c))) would carry the rounding error of m c into the
// exponent: up to half an ulp of M c, about 7e-7 of relative error in a sum
// of logits near 20 / c, which the residual max(0, p - q) of a small mass
// amplifies in its draws.  mc = fl(M c) = __fmul_rn(M, c).
__device__ __forceinline__ float reframe(float m, float mc, float c) {
  return ex2(__fmul_rn(m, c) - mc);
}

// max that propagates NaN (a NaN anywhere in a row must surface).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float warp_max_nan(float x) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ bool is_finite(float x) { return fabsf(x) <= FLT_MAX; }

// Unsigned division by a run-time invariant d >= 1 through a multiply and
// shifts (Granlund & Montgomery, "Division by invariant integers using
// multiplication", 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// q = (t + ((n - t) >> 1)) >> (l - 1) where t = mulhi(m, n), for every 32-bit n.
struct FastDiv {
  uint32_t d, m, s1, s2;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < d) ++l;
  FastDiv f;
  f.d = d;
  f.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  f.s1 = l > 0 ? 1 : 0;
  f.s2 = l > 0 ? l - 1 : 0;
  return f;
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffff); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_incl_scan(float x) {
  const int lane = lane_id();
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ int warp_incl_scan_int(int x) {
  const int lane = lane_id();
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// PDL (programmatic dependent launch): let the next kernel on the stream be
// scheduled early / wait for the previous kernel's results.  Both are no-ops
// when the launch did not request programmatic serialisation.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One add with release + acquire semantics at GPU scope: publishes this
// thread's earlier writes (chunk records) and, for the last arriver, makes
// the other arrivers' writes visible.  Replaces a fence + plain atomic.
__device__ __forceinline__ int atomic_add_acq_rel(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v)
               : "memory");
  return old;
}

// ---------------------------------------------------------------------------
// packed arithmetic (two bf16 in a 32-bit word, two fp32 in a 64-bit pair)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ---------------------------------------------------------------------------
// shared-memory staging: bulk copies completed on an mbarrier
// ---------------------------------------------------------------------------

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // no wait lasts longer than 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Copy `bytes` (a multiple of 16, both ends 16-byte aligned) from global
// into shared memory; completion is signalled on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// An L2 cache policy that makes the lines it brings in the first to be
// evicted: a single streaming pass over the logits then leaves in L2 what
// the later kernels of the call need (their code, the chunk records, the
// counters) instead of data it will never read again.
__device__ __forceinline__ unsigned long long l2_evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// A bulk copy like bulk_copy below, with an L2 cache policy.
__device__ __forceinline__ void bulk_copy_hint(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// One arrival that also announces `bytes` of copies, and a copy that only
// completes bytes (for several copies signalling one barrier phase).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar`, for at most `limit_ns` of wall time
// (kWaitLimitNs by default); false if it did not complete.  limit_ns = 0
// gives up at once without polling (the caller's own copies are still
// drained with the default limit before it leaves).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// per-lane tiles
// ---------------------------------------------------------------------------

// bf16 logits are handled as their raw 16-bit patterns (uint16_t).
template <typename T, int VEC>
struct Lane;

template <>
struct Lane<uint16_t, 8> {  // bf16, 8 per 128-bit load
  using Raw = uint4;
  static constexpr int VEC = 8, NV = 4, G = 4;  // G: chunks loaded per batch
  static __device__ __forceinline__ Raw load(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
  static __device__ __forceinline__ Raw pad() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  static __device__ __forceinline__ float get(const Raw& r, int e) {
    const uint32_t w = (e >> 1) == 0 ? r.x : (e >> 1) == 1 ? r.y : (e >> 1) == 2 ? r.z : r.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  // overwrite element e with -inf
  static __device__ __forceinline__ void kill(Raw& r, int e) {
    const uint32_t keep = (e & 1) ? 0x0000ffffu : 0xffff0000u;
    const uint32_t ninf = (e & 1) ? 0xff800000u : 0x0000ff80u;
    const int q = e >> 1;
    if (q == 0) r.x = (r.x & keep) | ninf;
    if (q == 1) r.y = (r.y & keep) | ninf;
    if (q == 2) r.z = (r.z & keep) | ninf;
    if (q == 3) r.w = (r.w & keep) | ninf;
  }
  // overwrite with -inf every element e whose bit e of `bits` is clear
  static __device__ __forceinline__ void allow_only(Raw& r, uint32_t bits) {
    // byte i of flags(n) is 0xff when bit i of the nibble n is set (the four
    // shifted copies of n in the product do not overlap, so nothing carries)
    auto flags = [](uint32_t n) { return ((n * 0x00204081u) & 0x01010101u) * 0xffu; };
    auto keep = [](uint32_t w, uint32_t k) { return (w & k) | (0xff80ff80u & ~k); };
    const uint32_t lo = flags(bits & 15u), hi = flags((bits >> 4) & 15u);
    r.x = keep(r.x, __byte_perm(lo, 0, 0x1100));
    r.y = keep(r.y, __byte_perm(lo, 0, 0x3322));
    r.z = keep(r.z, __byte_perm(hi, 0, 0x1100));
    r.w = keep(r.w, __byte_perm(hi, 0, 0x3322));
  }
};

template <>
struct Lane<float, 4> {  // fp32, 4 per 128-bit load
  using Raw = uint4;
  static constexpr int VEC = 4, NV = 8, G = 2;
  static __device__ __forceinline__ Raw load(const float* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
  static __device__ __forceinline__ Raw pad() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
  }
  static __device__ __forceinline__ float get(const Raw& r, int e) {
    return __uint_as_float(e == 0 ? r.x : e == 1 ? r.y : e == 2 ? r.z : r.w);
  }
  static __device__ __forceinline__ void kill(Raw& r, int e) {
    if (e == 0) r.x = 0xff800000u;
    if (e == 1) r.y = 0xff800000u;
    if (e == 2) r.z = 0xff800000u;
    if (e == 3) r.w = 0xff800000u;
  }
  static __device__ __forceinline__ void allow_only(Raw& r, uint32_t bits) {
    r.x = (bits & 1u) ? r.x : 0xff800000u;
    r.y = (bits & 2u) ? r.y : 0xff800000u;
    r.z = (bits & 4u) ? r.z : 0xff800000u;
    r.w = (bits & 8u) ? r.w : 0xff800000u;
  }
};

template <>
struct Lane<uint16_t, 1> {  // bf16, scalar path
  using Raw = unsigned short;
  static constexpr int VEC = 1, NV = 32, G = 1;
  static __device__ __forceinline__ Raw load(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
  }
  static __device__ __forceinline__ Raw pad() { return (unsigned short)0xff80u; }
  static __device__ __forceinline__ float get(const Raw& r, int) {
    return __uint_as_float((uint32_t)r << 16);
  }
  static __device__ __forceinline__ void kill(Raw& r, int) { r = pad(); }
  static __device__ __forceinline__ void allow_only(Raw& r, uint32_t bits) {
    if (!(bits & 1u)) r = pad();
  }
};

template <>
struct Lane<float, 1> {  // fp32, scalar path
  using Raw = float;
  static constexpr int VEC = 1, NV = 32, G = 1;
  static __device__ __forceinline__ Raw load(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ Raw pad() { return -INFINITY; }
  static __device__ __forceinline__ float get(const Raw& r, int) { return r; }
  static __device__ __forceinline__ void kill(Raw& r, int) { r = pad(); }
  static __device__ __forceinline__ void allow_only(Raw& r, uint32_t bits) {
    if (!(bits & 1u)) r = pad();
  }
};

// one logit, widened to fp32
__device__ __forceinline__ float load_logit(const uint16_t* row, int j) {
  return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + j) << 16);
}
__device__ __forceinline__ float load_logit(const float* row, int j) { return __ldg(row + j); }

// offset of group k, element e of this lane inside a chunk
template <int VEC>
__device__ __forceinline__ int tile_offset(int k, int e, int lane) {
  return k * kWarp * VEC + lane * VEC + e;
}

// ---------------------------------------------------------------------------
// grammar masks: ceil(V/32) 32-bit words per row; token j is allowed when
// bit j % 32 of word j / 32 is set.  One chunk's 1024 tokens are 32 words:
// lane l holds word (chunk * 32 + l).
// ---------------------------------------------------------------------------

// The chunk's mask word of this lane from global memory (0 past the row).
__device__ __forceinline__ uint32_t mask_word(const uint32_t* mrow, int words, int c) {
  const int i = c * kWarp + lane_id();
  return i < words ? __ldg(mrow + i) : 0u;
}

// Disallowed elements of this lane's chunk tile become -inf (a warp-wide
// call: each group's bits come from the lane holding their word).
template <typename T, int VEC>
__device__ __forceinline__ void allow_only_chunk(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                                 uint32_t word) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    const int first = tile_offset<VEC>(k, 0, lane);  // VEC consecutive tokens, one word
    const uint32_t w = __shfl_sync(0xffffffffu, word, first >> 5);
    L::allow_only(raw[k], (w >> (first & 31)) & ((1u << VEC) - 1u));
  }
}

template <typename T, int VEC>
__device__ __forceinline__ void load_chunk(const T* row, int V, int c,
                                           typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV]) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    const int j = c * kChunk + tile_offset<VEC>(k, 0, lane);
    raw[k] = (j < V) ? L::load(row + j) : L::pad();
  }
}

// The same tile from a chunk staged in shared memory at `stage` (vector
// paths only); groups at or past V get the -inf pad.
template <typename T, int VEC>
__device__ __forceinline__ void load_chunk_smem(uint32_t stage, int V, int c,
                                                typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV]) {
  using L = Lane<T, VEC>;
  static_assert(VEC * sizeof(T) == 16, "shared-memory tiles are 128-bit groups");
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    const int off = tile_offset<VEC>(k, 0, lane);
    raw[k] = (c * kChunk + off < V) ? lds128(stage + off * (int)sizeof(T)) : L::pad();
  }
}

// Overwrite the element at chunk offset mask_local (held by one lane) with -inf.
template <typename T, int VEC>
__device__ __forceinline__ void mask_element(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                             int mask_local) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    const int base = tile_offset<VEC>(k, 0, lane);
    if (mask_local >= base && mask_local < base + VEC) L::kill(raw[k], mask_local - base);
  }
}

// bf16 vector tile (4 x 128-bit groups = 16 words = 32 logits per lane):
// NaN-propagating max on packed bf16 pairs.
__device__ __forceinline__ float lane_max_bf16(const uint4 (&raw)[4]) {
  // a depth-4 tree over the 16 words (a serial chain would be 15 deep)
  uint32_t m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    m[k] = bf16x2_max_nan(bf16x2_max_nan(raw[k].x, raw[k].y), bf16x2_max_nan(raw[k].z, raw[k].w));
  const uint32_t t = bf16x2_max_nan(bf16x2_max_nan(m[0], m[1]), bf16x2_max_nan(m[2], m[3]));
  return max_nan(bf16_lo(t), bf16_hi(t));
}

// Softmax record of one chunk: {m_c, sum_j 2^(l_j*cc - m_c*cc)}, leaving
// out the element at chunk offset mask_local (>= 0) - the one-hot residual
// excludes the draft token; the max still includes it.  m_c = -inf for an
// all -inf chunk; NaN marks a chunk that holds NaN or +inf.  The bf16 vector
// tile uses packed instructions (bf16x2 max, fma.rn.f32x2, add.rn.f32x2);
// every weight is rounded exactly as the scalar fmaf + ex2 of the rescan.
// With `ent` given, *ent receives sum_j w_j t_j over the chunk, t_j = (l_j -
// max) c the base-2 exponent of w_j (the chunk's share of the row entropy;
// -inf elements, whose weight is 0, add nothing).
// `exclude(raw)` runs after the max: it overwrites the elements left out of
// the sum with -inf (chunk_softmax: at most one, at chunk offset mask_local).
template <typename T, int VEC, class Exclude>
__device__ __forceinline__ float2 chunk_softmax_ex(
    typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV], float cc, Exclude exclude,
    float* ent = nullptr) {
  using L = Lane<T, VEC>;
  constexpr bool kPacked = sizeof(T) == 2 && VEC == 8;
  float lm = -INFINITY;
  if constexpr (kPacked) {
    lm = lane_max_bf16(raw);
  } else {
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) lm = max_nan(lm, L::get(raw[k], e));
  }
  const float cm = warp_max_nan(lm);
  if (!is_finite(cm)) {
    if (ent) *ent = 0.f;
    return make_float2(cm == -INFINITY ? -INFINITY : qnan(), 0.f);
  }
  exclude(raw);
  const float nb = -cm * cc;
  float s, et = 0.f;
  if constexpr (kPacked) {
    const f32x2 c2 = pack2(cc, cc), nb2 = pack2(nb, nb);
    f32x2 acc[4];  // four independent accumulation chains
    f32x2 eacc[2];  // the entropy accumulator: w t as one packed fma per pair
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = pack2(0.f, 0.f);
    eacc[0] = eacc[1] = pack2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const f32x2 a2 = fma2(pack2(bf16_lo(w[q]), bf16_hi(w[q])), c2, nb2);
        float a0, a1;
        unpack2(a2, a0, a1);
        const f32x2 e2 = pack2(ex2(a0), ex2(a1));
        acc[q] = add2(acc[q], e2);
        if (ent) eacc[q & 1] = fma2(e2, a2, eacc[q & 1]);
      }
    }
    float s0, s1, s2, s3;
    unpack2(add2(acc[0], acc[1]), s0, s1);
    unpack2(add2(acc[2], acc[3]), s2, s3);
    s = (s0 + s1) + (s2 + s3);
    if (ent) {
      float t0, t1;
      unpack2(add2(eacc[0], eacc[1]), t0, t1);
      et = t0 + t1;
      // a -inf logit (weight 0, exponent -inf) made the product NaN: this
      // lane's accumulator again with the exponent clamped (rare)
      if (et != et) {
        et = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float a0 = fmaf(bf16_lo(w[q]), cc, nb), a1 = fmaf(bf16_hi(w[q]), cc, nb);
            et = fmaf(ex2(a1), fmaxf(a1, -256.f), fmaf(ex2(a0), fmaxf(a0, -256.f), et));
          }
        }
      }
    }
  } else {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float a = fmaf(L::get(raw[k], e), cc, nb);
        const float w = ex2(a);
        if ((k * VEC + e) & 1) s1 += w; else s0 += w;
        if (ent) et = fmaf(w, fmaxf(a, -256.f), et);
      }
    s = s0 + s1;
  }
  if (ent) *ent = warp_sum(et);
  return make_float2(cm, warp_sum(s));
}

template <typename T, int VEC>
__device__ __forceinline__ float2 chunk_softmax(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                                float cc, int mask_local, float* ent = nullptr) {
  return chunk_softmax_ex<T, VEC>(
      raw, cc,
      [mask_local](typename Lane<T, VEC>::Raw(&r)[Lane<T, VEC>::NV]) {
        if (mask_local >= 0) mask_element<T, VEC>(r, mask_local);
      },
      ent);
}

// Argmax record of one chunk: {max, lowest global index attaining it} (index
// INT_MAX if the max is NaN).  Exact: compares the stored values.
template <typename T, int VEC>
__device__ __forceinline__ float2 chunk_argmax(const typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                               int chunk_base) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  float lm = -INFINITY;
  if constexpr (sizeof(T) == 2 && VEC == 8) {
    lm = lane_max_bf16(raw);
  } else {
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) lm = max_nan(lm, L::get(raw[k], e));
  }
  const float cm = warp_max_nan(lm);
  unsigned idx = 0x7fffffffu;
  if (lm == cm) {  // this lane holds a maximum (rare branch)
#pragma unroll
    for (int k = L::NV - 1; k >= 0; --k)
#pragma unroll
      for (int e = VEC - 1; e >= 0; --e)
        if (L::get(raw[k], e) == cm) idx = (unsigned)(chunk_base + tile_offset<VEC>(k, e, lane));
  }
  idx = __reduce_min_sync(0xffffffffu, idx);
  return make_float2(cm, __int_as_float((int)idx));
}

// Warp-wide combination of argmax records held one per lane, where a lane's
// record already has the lowest index among its own equal maxima.
__device__ __forceinline__ float2 warp_combine_argmax(float2 r) {
  const float m = warp_max_nan(r.x);
  const unsigned idx = __reduce_min_sync(0xffffffffu, r.x == m ? (unsigned)__float_as_int(r.y)
                                                               : 0x7fffffffu);
  return make_float2(m, __int_as_float((int)idx));
}

// Combine a row's chunk records (ascending chunk order per lane).
__device__ __forceinline__ float2 combine_argmax_records(const float2* rec, int NC) {
  const int lane = lane_id();
  float2 best = make_float2(-INFINITY, __int_as_float(0x7fffffff));
  bool first = true;
  for (int c = lane; c < NC; c += kWarp) {
    const float2 r = __ldcg(rec + c);
    if (first || r.x > best.x || (r.x != r.x && best.x == best.x)) best = r;
    first = false;
  }
  return warp_combine_argmax(best);
}

// Combine a row's softmax chunk records into {m, S} with S in the frame of
// fl(m c) (the weights 2^(l c - fl(m c))).
constexpr int kRecCache = 8;  // records cached per lane (rows of up to 256 chunks)

// `copy` (shared memory, or nullptr) receives the records as they are read.
__device__ __forceinline__ float2 combine_softmax_records(const float2* rec, int NC, float cc,
                                                          float2* copy = nullptr) {
  const int lane = lane_id();
  float2 cache[kRecCache];
  float lm = -INFINITY;
#pragma unroll
  for (int t = 0; t < kRecCache; ++t) {
    const int c = lane + t * kWarp;
    cache[t] = c < NC ? __ldcg(rec + c) : make_float2(-INFINITY, 0.f);
    if (copy && c < NC) copy[c] = cache[t];
    lm = max_nan(lm, cache[t].x);
  }
  for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) {
    const float2 r = __ldcg(rec + c);
    if (copy) copy[c] = r;
    lm = max_nan(lm, r.x);
  }
  const float m = warp_max_nan(lm);
  if (!is_finite(m)) return make_float2(m == -INFINITY ? -INFINITY : qnan(), 0.f);
  const float mc = __fmul_rn(m, cc);  // the row's frame (the draws' weights use it too)
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < kRecCache; ++t) s += cache[t].y * reframe(cache[t].x, mc, cc);
  for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) {
    const float2 r = __ldcg(rec + c);
    s += r.y * reframe(r.x, mc, cc);
  }
  return make_float2(m, warp_sum(s));
}

// Entropy accumulator of a row from its chunk records and the chunks'
// accumulators (see chunk_softmax): sum_j w_j t_j in the frame of the row
// max m, with w_j = 2^t_j, t_j = (l_j - m) c.  A chunk of maximum m_c
// contributes 2^((m_c - m) c) (A_c + (m_c - m) c S_c).  The row entropy in
// nats is then ln S - ln 2 * A / S.
__device__ __forceinline__ float combine_entropy(const float2* rec, const float* ent, int NC,
                                                 float cc, float m) {
  float a = 0.f;
  for (int c = lane_id(); c < NC; c += kWarp) {
    const float2 r = __ldcg(rec + c);
    if (!(r.y > 0.f)) continue;
    const float d = (r.x - m) * cc;
    a += ex2(d) * fmaf(d, r.y, __ldcg(ent + c));
  }
  return warp_sum(a);
}

// ---------------------------------------------------------------------------
// candidate trees in device memory
// ---------------------------------------------------------------------------

constexpr int kTreeMaxNodes = 256;  // candidate nodes per tree (the root excluded)

// Request's parent array (parent of node n = 1..N at parent[n - 1]) into
// s_par[0..N] (s_par[0] = 0), with s_anc = s_par and s_depth[n] = (n > 0) as
// the start of tree_depths_ok.  True when every parent is an earlier node, so
// the links cannot cycle (an out-of-range parent is stored as 0).  Called by
// every thread of the CTA.
__device__ __forceinline__ bool load_parents(const int* parent, int N, short* s_par,
                                             short* s_depth, short* s_anc) {
  int bad = 0;
  for (int n = threadIdx.x; n <= N; n += blockDim.x) {
    int pa = 0;
    if (n > 0) {
      pa = __ldg(parent + n - 1);
      if (pa < 0 || pa >= n) {
        bad = 1;
        pa = 0;
      }
    }
    s_par[n] = (short)pa;
    s_anc[n] = (short)pa;
    s_depth[n] = (short)(n > 0);
  }
  return !__syncthreads_or(bad);
}

// Every node's depth into s_depth by pointer jumping over the links that
// load_parents stored (s_anc is scratch): rounds of depth[n] += depth[anc[n]],
// anc[n] = anc[anc[n]] until the jumps span the tree.  True when no node is
// deeper than max_depth.  Trees of fewer than 64 nodes are done by warp 0 in
// registers (nodes lane and lane + 32, exchanged by shuffles); larger ones
// in shared memory by the CTA (>= 128 threads).  Called by every thread of
// the CTA; the same data gives every CTA the same answer.
__device__ __forceinline__ bool tree_depths_ok(int N, int max_depth, short* s_depth, short* s_anc) {
  int bad = 0;
  if (N < 2 * kWarp) {
    if (threadIdx.x < kWarp) {
      const int lane = threadIdx.x, n1 = lane + kWarp;
      int d0 = lane <= N ? s_depth[lane] : 0, a0 = lane <= N ? s_anc[lane] : 0;
      int d1 = n1 <= N ? s_depth[n1] : 0, a1 = n1 <= N ? s_anc[n1] : 0;
      for (int span = 1; span <= N; span <<= 1) {
        const int x0 = __shfl_sync(0xffffffffu, d0, a0 & 31), y0 = __shfl_sync(0xffffffffu, d1, a0 & 31);
        const int p0 = __shfl_sync(0xffffffffu, a0, a0 & 31), q0 = __shfl_sync(0xffffffffu, a1, a0 & 31);
        const int x1 = __shfl_sync(0xffffffffu, d0, a1 & 31), y1 = __shfl_sync(0xffffffffu, d1, a1 & 31);
        const int p1 = __shfl_sync(0xffffffffu, a0, a1 & 31), q1 = __shfl_sync(0xffffffffu, a1, a1 & 31);
        d0 += a0 < kWarp ? x0 : y0;
        a0 = a0 < kWarp ? p0 : q0;
        d1 += a1 < kWarp ? x1 : y1;
        a1 = a1 < kWarp ? p1 : q1;
      }
      if (lane <= N) s_depth[lane] = (short)d0;
      if (n1 <= N) s_depth[n1] = (short)d1;
      bad = (lane <= N && d0 > max_depth) || (n1 <= N && d1 > max_depth);
    }
    return !__syncthreads_or(bad);
  }
  constexpr int kPer = (kTreeMaxNodes + 1 + 127) / 128;  // nodes per thread (>= 128 threads)
  for (int span = 1; span <= N; span <<= 1) {
    short nd[kPer], na[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int n = threadIdx.x + i * (int)blockDim.x;
      if (n <= N) {
        const int a = s_anc[n];
        nd[i] = (short)(s_depth[n] + s_depth[a]);
        na[i] = s_anc[a];
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int n = threadIdx.x + i * (int)blockDim.x;
      if (n <= N) {
        s_depth[n] = nd[i];
        s_anc[n] = na[i];
      }
    }
    __syncthreads();
  }
  for (int n = threadIdx.x; n <= N; n += blockDim.x) bad |= s_depth[n] > max_depth;
  return !__syncthreads_or(bad);
}

// load_parents, then tree_depths_ok: true when the request's parent array is
// a tree of depth <= max_depth.
__device__ __forceinline__ bool load_tree(const int* parent, int N, int max_depth, short* s_par,
                                          short* s_depth, short* s_anc) {
  if (!load_parents(parent, N, s_par, s_depth, s_anc)) return false;
  return tree_depths_ok(N, max_depth, s_depth, s_anc);
}

// Asks L2 for `bytes` bytes at ptr (16-byte aligned, a multiple of 16): a
// bulk prefetch, no data returned.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

}  // namespace sv
