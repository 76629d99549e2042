// sv_rows.cuh - device helpers shared by the verification kernels (streaming
// records, filtered records, finalize) and the launch helper; internal.
#pragma once

#include <cooperative_groups.h>

#include <mutex>

#include "sv_common.cuh"
#include "sv_launch.h"

namespace sv {
namespace {

namespace cg = cooperative_groups;

template <typename T>
__device__ __forceinline__ const T* row_ptr(const void* base, long long row, int V) {
  return reinterpret_cast<const T*>(base) + row * (long long)V;
}

// Elements below a row's top-k / top-p cut value become -inf.
template <typename T, int VEC>
__device__ __forceinline__ void threshold_chunk(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                                float thr) {
  using L = Lane<T, VEC>;
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    uint32_t bits = 0;
#pragma unroll
    for (int e = 0; e < VEC; ++e) bits |= (L::get(raw[k], e) >= thr ? 1u : 0u) << e;
    L::allow_only(raw[k], bits);
  }
}

// The row's top-k / top-p cut value (-inf: nothing cut).
__device__ __forceinline__ float row_cut(const VerifyParams& p, long long rowid) {
  return p.filter ? __ldcg(p.thr + rowid) : -INFINITY;
}

// Grammar mask row of position i of request b (target row i and dense
// draft row i share it), or null without masks.
__device__ __forceinline__ const uint32_t* mask_row(const VerifyParams& p, int b, int i) {
  return p.mask ? p.mask + ((long long)b * (p.K + 1) + i) * p.mask_words : nullptr;
}

// Whether row r of request b is needed: target rows 0..K_b, draft rows
// 0..K_b-1 (K_b = draft_lens[b] or K; nothing when K_b is invalid).
__device__ __forceinline__ bool row_needed(const VerifyParams& p, int r, int Kb) {
  if (Kb < 0 || Kb > p.K) return false;
  return r > p.K ? (r - p.K - 1) < Kb : r <= Kb;
}

template <int MODE, typename T, int VEC>
__device__ __forceinline__ float2 chunk_record(typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV],
                                               int c, float cc, int mask_x,
                                               float* ent = nullptr) {
  if (MODE == kGreedy) return chunk_argmax<T, VEC>(raw, c * kChunk);
  if (MODE == kTypical) {  // no exclusion; the chunk's entropy accumulator too
    float a = 0.f;
    const float2 r = chunk_softmax<T, VEC>(raw, cc, -1, &a);
    if (lane_id() == 0) *ent = a;
    return r;
  }
  const int ml = (mask_x >= c * kChunk && mask_x < (c + 1) * kChunk) ? mask_x - c * kChunk : -1;
  return chunk_softmax<T, VEC>(raw, cc, ml);
}

// Tree sampling: the record of chunk c of node r's row leaves out of its sum
// the tokens of r's children - the candidates tested against that row, every
// one of which is removed from the residual before the final draw - and
// keeps them in its max.  Node n's parent and token (n = 1..N) are at index
// n - 1 of the request's arrays.
template <typename T, int VEC>
__device__ __forceinline__ float2 tree_chunk_record(
    const VerifyParams& p, typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV], int rowid, int c) {
  using Raw = typename Lane<T, VEC>::Raw;
  const int b = (int)fast_div((uint32_t)rowid, p.div_r);
  const int r = rowid - b * p.R;
  const int N = p.K;
  const int* par = p.tree_parent + (long long)b * p.parent_stride;
  const int* tok = p.tree_tokens + (long long)b * N;
  const int lo = c * kChunk;
  // Trees of up to 64 nodes: the children's offsets in this chunk are looked
  // up before the max, two nodes per lane, their four loads in flight at once.
  int off0 = -1, off1 = -1;
  if (N <= 2 * kWarp) {
    const int n0 = lane_id(), n1 = n0 + kWarp;
    const int pa0 = n0 < N ? __ldg(par + n0) : -1, pa1 = n1 < N ? __ldg(par + n1) : -1;
    const int t0 = n0 < N ? __ldg(tok + n0) - lo : -1, t1 = n1 < N ? __ldg(tok + n1) - lo : -1;
    if (pa0 == r && t0 >= 0 && t0 < kChunk) off0 = t0;
    if (pa1 == r && t1 >= 0 && t1 < kChunk) off1 = t1;
  }
  return chunk_softmax_ex<T, VEC>(raw, p.cc, [&](Raw(&rr)[Lane<T, VEC>::NV]) {
    if (N <= 2 * kWarp) {
      for (unsigned hit = __ballot_sync(0xffffffffu, off0 >= 0); hit; hit &= hit - 1u)
        mask_element<T, VEC>(rr, __shfl_sync(0xffffffffu, off0, __ffs(hit) - 1));
      for (unsigned hit = __ballot_sync(0xffffffffu, off1 >= 0); hit; hit &= hit - 1u)
        mask_element<T, VEC>(rr, __shfl_sync(0xffffffffu, off1, __ffs(hit) - 1));
      return;
    }
    for (int n0 = 0; n0 < N; n0 += kWarp) {
      const int n = n0 + lane_id();
      int off = -1;
      if (n < N && __ldg(par + n) == r) {
        const int t = __ldg(tok + n) - lo;
        if (t >= 0 && t < kChunk) off = t;
      }
      for (unsigned hit = __ballot_sync(0xffffffffu, off >= 0); hit; hit &= hit - 1u)
        mask_element<T, VEC>(rr, __shfl_sync(0xffffffffu, off, __ffs(hit) - 1));
    }
  });
}

// If the row's draft token x lies in chunk c, the lane holding it records
// the logit l_x for the finalize kernel (p(x) = 2^((l_x - m) c) / S).
template <typename T, int VEC>
__device__ __forceinline__ void record_draft_logit(
    const VerifyParams& p, const typename Lane<T, VEC>::Raw (&raw)[Lane<T, VEC>::NV], int c,
    int rowid, int x) {
  using L = Lane<T, VEC>;
  const int off = x - c * kChunk;
  if (off < 0 || off >= kChunk) return;
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < L::NV; ++k) {
    const int base = tile_offset<VEC>(k, 0, lane);
    if (off >= base && off < base + VEC) p.lx[rowid] = L::get(raw[k], off - base);
  }
}

template <typename T>
__device__ __forceinline__ const T* item_row(const VerifyParams& p, int rowid) {
  const int b = (int)fast_div((uint32_t)rowid, p.div_r);
  const int r = rowid - b * p.R;
  return r > p.K ? row_ptr<T>(p.draft, (long long)b * p.K + (r - p.K - 1), p.V)
                 : row_ptr<T>(p.target, (long long)b * (p.K + 1) + r, p.V);
}

// The grammar mask row of a logit row (target row i or draft row i of
// request b: the mask of position i), or null without masks.
__device__ __forceinline__ const uint32_t* item_mask(const VerifyParams& p, int rowid) {
  if (!p.mask) return nullptr;
  const int b = (int)fast_div((uint32_t)rowid, p.div_r);
  const int r = rowid - b * p.R;
  return mask_row(p, b, r > p.K ? r - p.K - 1 : r);
}

// One-time set-up of a kernel on each device (function attributes and
// occupancy are per device): the first call with a device current runs
// `setup(value)`; later calls return the cached value.  Thread-safe.
struct PerDevice {
  std::mutex mu;
  unsigned long long done = 0;  // bit d: device d set up
  int value[64] = {};
};
template <class F>
cudaError_t per_device(PerDevice& once, int* value, F setup) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(once.mu);
  if (!((once.done >> dev) & 1ull)) {
    int v = 0;
    err = setup(v);
    if (err != cudaSuccess) return err;
    once.value[dev] = v;
    once.done |= 1ull << dev;
  }
  if (value) *value = once.value[dev];
  return cudaSuccess;
}

// Launch with programmatic dependent launch allowed (and a cluster of
// `cluster` CTAs along x when cluster > 1).
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, cudaStream_t s, void** args,
                       size_t smem = 0, int cluster = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace
}  // namespace sv
