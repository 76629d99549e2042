// sv_tree.cu - greedy tree verification (Medusa / EAGLE candidate trees).
//
// Method ("【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §3.3 "Tree
// Attention"): the candidates of one step form a tree under the root; node n's
// target row was computed seeing only n's ancestors; the accepted path is the
// longest root path on which every node's token equals the target argmax at
// its parent.  Starting at the root, the walk takes the argmax of the current
// node's row, moves to the child carrying that token, and stops at a node
// without such a child; the argmax there is the extra token.
//
// One thread-block cluster per request.  Each step, the cluster's warps split
// the current row into 1024-element chunks (exact argmax, lowest index on
// ties), each CTA reduces its warps, the CTAs exchange their results through
// distributed shared memory after a cluster barrier, and every CTA derives the
// same next node from the same data, so all of them run the same number of
// steps.  Only the rows on the accepted path are read; with PREFETCH, the
// children's rows are pulled into L2 while the current row is reduced, so the
// next step's loads hit L2.
#include <cooperative_groups.h>

#include "sv_common.cuh"
#include "sv_launch.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kTreeThreads = 128;
constexpr int kTreeWarps = kTreeThreads / kWarp;

__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <typename T, int VEC, bool PREFETCH>
__global__ void __launch_bounds__(kTreeThreads) tree_kernel(const __grid_constant__ TreeParams p) {
  using L = Lane<T, VEC>;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / CL;
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int gw = rank * kTreeWarps + warp;
  const int W = CL * kTreeWarps;

  __shared__ int s_tok[kMaxTreeNodes + 1];
  __shared__ short s_par[kMaxTreeNodes + 1], s_depth[kMaxTreeNodes + 1], s_anc[kMaxTreeNodes + 1];
  __shared__ int s_kid[kMaxTreeNodes];
  __shared__ int s_nkid;
  __shared__ float2 s_warp[kTreeWarps];
  __shared__ float2 s_cta[2];
  __shared__ int s_path[kMaxTreeNodes + 1];
  __shared__ int s_out[kMaxTreeNodes + 1];

  // every CTA of the cluster loads the same tree and reaches the same verdict
  const bool tree_ok = load_tree(p.parent + (long long)b * p.parent_stride, p.N, p.D1 - 1, s_par,
                                 s_depth, s_anc);
  int bad = 0;
  for (int n = 1 + threadIdx.x; n <= p.N; n += blockDim.x) {
    const int t = __ldg(p.tokens + (long long)b * p.N + n - 1);
    s_tok[n] = t;
    bad |= (t < 0 || t >= p.V);
  }
  bad = __syncthreads_or(bad);
  int status = !tree_ok ? kBadTree : (bad ? kBadToken : 0);
  int node = 0, depth = 0, parity = 0;
  while (!status) {
    __syncthreads();  // the previous step's reads of s_kid are done
    // the current node's children, in increasing id (warp 0)
    if (warp == 0) {
      int nk = 0;
      for (int c0 = 1; c0 <= p.N; c0 += kWarp) {
        const int c = c0 + lane;
        const bool kid = c <= p.N && s_par[c] == node;
        const unsigned m = __ballot_sync(0xffffffffu, kid);
        if (kid) s_kid[nk + __popc(m & ((1u << lane) - 1u))] = c;
        nk += __popc(m);
      }
      if (lane == 0) s_nkid = nk;
    }
    __syncthreads();
    const int nkid = s_nkid;
    const T* row = reinterpret_cast<const T*>(p.target) + ((long long)b * (p.N + 1) + node) * p.V;
    float2 best = make_float2(-INFINITY, __int_as_float(0x7fffffff));
    bool first = true;
    for (int c = gw; c < p.NC; c += W) {
      typename L::Raw raw[L::NV];
      load_chunk<T, VEC>(row, p.V, c, raw);
      if (PREFETCH && lane == 0) {
        const unsigned bytes = (unsigned)(min(kChunk, p.V - c * kChunk) * sizeof(T));
        for (int k = 0; k < nkid; ++k)
          prefetch_l2(reinterpret_cast<const T*>(p.target) +
                          ((long long)b * (p.N + 1) + s_kid[k]) * p.V + (long long)c * kChunk,
                      bytes);
      }
      const float2 r = chunk_argmax<T, VEC>(raw, c * kChunk);
      if (first || r.x > best.x || (r.x != r.x && best.x == best.x)) best = r;
      first = false;
    }
    if (lane == 0) s_warp[warp] = best;
    __syncthreads();
    if (warp == 0) {
      float2 v = lane < kTreeWarps ? s_warp[lane] : make_float2(-INFINITY, __int_as_float(0x7fffffff));
      v = warp_combine_argmax(v);
      if (lane == 0) s_cta[parity] = v;
    }
    cluster.sync();
    float2 v = make_float2(-INFINITY, __int_as_float(0x7fffffff));
    if (lane < CL) v = *cluster.map_shared_rank(&s_cta[parity], lane);
    v = warp_combine_argmax(v);
    if (!is_finite(v.x)) {
      status = kBadLogits;
      break;
    }
    const int a = __float_as_int(v.y);
    if (threadIdx.x == 0) {
      s_path[depth] = node;
      s_out[depth] = a;
    }
    ++depth;
    int next = 0;  // the lowest child carrying the argmax
    for (int k = 0; k < nkid; ++k)
      if (s_tok[s_kid[k]] == a) {
        next = s_kid[k];
        break;
      }
    if (!next) break;
    node = next;
    parity ^= 1;
  }
  cluster.sync();  // keep every CTA's shared memory alive until all reads are done
  if (rank == 0) {
    __syncthreads();
    const long long o = (long long)b * p.D1;
    for (int k = threadIdx.x; k < p.D1; k += blockDim.x) {
      const bool on = !status && k < depth;
      p.out_tokens[o + k] = on ? s_out[k] : -1;
      if (p.out_path) p.out_path[o + k] = on ? s_path[k] : -1;
    }
    if (threadIdx.x == 0) {
      p.out_accept_len[b] = status ? 0 : depth;
      if (p.out_status) p.out_status[b] = status;
    }
  }
}

template <typename T, int VEC, bool PREFETCH>
cudaError_t launch_tree_typed(const TreeParams& p, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  // cluster size: enough CTAs to cover the SMs, at most one warp per chunk
  int cl = 1;
  while (cl < 8 && (long long)p.B * cl < di.sms && (cl * 2) * kTreeWarps <= p.NC) cl *= 2;
  if ((long long)p.B * cl < 2LL * di.sms && cl < 8 && (cl * 2) * kTreeWarps <= p.NC) cl *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * cl));
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_kernel<T, VEC, PREFETCH>, p);
}

}  // namespace

cudaError_t launch_tree(int dtype, bool vec, const TreeParams& p, cudaStream_t stream) {
  if (dtype == kBF16)
    return vec ? launch_tree_typed<uint16_t, 8, true>(p, stream)
               : launch_tree_typed<uint16_t, 1, false>(p, stream);
  return vec ? launch_tree_typed<float, 4, true>(p, stream)
             : launch_tree_typed<float, 1, false>(p, stream);
}

}  // namespace sv
