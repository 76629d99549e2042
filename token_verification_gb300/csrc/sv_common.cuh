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

enum Mode : int { kOneHot = 0, kDense = 1, kGreedy = 2 };

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
};

template <>
struct Lane<float, 1> {  // fp32, scalar path
  using Raw = float;
  static constexpr int VEC = 1, NV = 32, G = 1;
  static __device__ __forceinline__ Raw load(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ Raw pad() { return -INFINITY; }
  static __device__ __forceinline__ float get(const Raw& r, int) { return r; }
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

// Softmax record of one chunk: {m_c, sum_j 2^(l_j*cc - m_c*cc)}, skipping the
// element at chunk offset mask_local (>= 0) - the one-hot residual excludes
// the draft token.  m_c = -inf for an all -inf chunk; NaN marks a chunk that
// holds NaN or +inf.
template <typename T, int VEC>
__device__ __forceinline__ float2 chunk_softmax(const typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                                float cc, int mask_local) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  float lm = -INFINITY;
#pragma unroll
  for (int k = 0; k < L::NV; ++k)
#pragma unroll
    for (int e = 0; e < VEC; ++e) lm = max_nan(lm, L::get(raw[k], e));
  const float cm = warp_max_nan(lm);
  if (!is_finite(cm)) return make_float2(cm == -INFINITY ? -INFINITY : qnan(), 0.f);
  const float nb = -cm * cc;
  float s0 = 0.f, s1 = 0.f;
  if (mask_local < 0) {
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float w = ex2(fmaf(L::get(raw[k], e), cc, nb));
        if ((k * VEC + e) & 1) s1 += w; else s0 += w;
      }
  } else {
#pragma unroll
    for (int k = 0; k < L::NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        float w = ex2(fmaf(L::get(raw[k], e), cc, nb));
        if (tile_offset<VEC>(k, e, lane) == mask_local) w = 0.f;
        if ((k * VEC + e) & 1) s1 += w; else s0 += w;
      }
  }
  return make_float2(cm, warp_sum(s0 + s1));
}

// Argmax record of one chunk: {max, lowest global index attaining it} (index
// INT_MAX if the max is NaN).  Exact: compares the stored values.
template <typename T, int VEC>
__device__ __forceinline__ float2 chunk_argmax(const typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                               int chunk_base) {
  using L = Lane<T, VEC>;
  const int lane = lane_id();
  float lm = -INFINITY;
#pragma unroll
  for (int k = 0; k < L::NV; ++k)
#pragma unroll
    for (int e = 0; e < VEC; ++e) lm = max_nan(lm, L::get(raw[k], e));
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

// Combine a row's softmax chunk records into {m, S} with S in the frame of m.
constexpr int kRecCache = 8;  // records cached per lane (rows of up to 256 chunks)

__device__ __forceinline__ float2 combine_softmax_records(const float2* rec, int NC, float cc) {
  const int lane = lane_id();
  float2 cache[kRecCache];
  float lm = -INFINITY;
#pragma unroll
  for (int t = 0; t < kRecCache; ++t) {
    const int c = lane + t * kWarp;
    cache[t] = c < NC ? __ldcg(rec + c) : make_float2(-INFINITY, 0.f);
    lm = max_nan(lm, cache[t].x);
  }
  for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) lm = max_nan(lm, __ldcg(rec + c).x);
  const float m = warp_max_nan(lm);
  if (!is_finite(m)) return make_float2(m == -INFINITY ? -INFINITY : qnan(), 0.f);
  const float nb = -m * cc;
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < kRecCache; ++t) s += cache[t].y * ex2(fmaf(cache[t].x, cc, nb));
  for (int c = lane + kRecCache * kWarp; c < NC; c += kWarp) {
    const float2 r = __ldcg(rec + c);
    s += r.y * ex2(fmaf(r.x, cc, nb));
  }
  return make_float2(m, warp_sum(s));
}

}  // namespace sv
