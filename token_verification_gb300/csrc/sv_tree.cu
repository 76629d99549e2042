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
// One thread-block cluster per request.  Each step reduces the current node's
// row and, speculatively, the rows of all its children in one batch of loads
// (the cluster's warps split every row of the set into 1024-element chunks;
// exact argmax, lowest index on ties); CTAs exchange their partial results
// through distributed shared memory after one cluster barrier, and every CTA
// derives the same outcome from the same data, so all of them run the same
// number of steps.  The node's argmax picks the child; that child's argmax is
// already known and picks the grandchild, which the next step starts from:
// one step resolves two levels of the walk.  Only the rows of the walked
// nodes and their children are read.
#include <cooperative_groups.h>

#include "sv_common.cuh"
#include "sv_launch.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kTreeThreads = 128;
constexpr int kTreeWarps = kTreeThreads / kWarp;
constexpr int kRowBatch = 4;  // rows of the step's set whose chunks a warp loads together

__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The lowest child of `node` whose token is `tok` (0 if none); a warp-wide
// call, the same answer in every lane.
__device__ __forceinline__ int child_with_token(const short* s_par, const int* s_tok, int N,
                                                int node, int tok) {
  for (int c0 = 1; c0 <= N; c0 += kWarp) {
    const int c = c0 + lane_id();
    const unsigned hit =
        __ballot_sync(0xffffffffu, c <= N && s_par[c] == node && s_tok[c] == tok);
    if (hit) return c0 + __ffs(hit) - 1;
  }
  return 0;
}

template <typename T, int VEC>
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
  __shared__ int s_row[kMaxTreeNodes + 1];  // the step's rows: the node, then its children
  __shared__ int s_nrow;
  __shared__ float2 s_warp[kTreeWarps][kMaxTreeNodes + 1];
  __shared__ float2 s_cta[2][kMaxTreeNodes + 1];  // this CTA's result per row (two steps' worth)
  __shared__ int s_arg[kMaxTreeNodes + 1];         // the cluster's argmax per row (INT_MAX: bad)
  __shared__ int s_path[kMaxTreeNodes + 1];
  __shared__ int s_out[kMaxTreeNodes + 1];

  pdl_begin();
  // every CTA of the cluster loads the same tree and reaches the same verdict
  constexpr int kPer = (kMaxTreeNodes + kTreeThreads - 1) / kTreeThreads;
  int tok[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = 1 + threadIdx.x + i * kTreeThreads;
    tok[i] = n <= p.N ? __ldg(p.tokens + (long long)b * p.N + n - 1) : 0;
  }
  const bool tree_ok = load_tree(p.parent + (long long)b * p.parent_stride, p.N, p.D1 - 1, s_par,
                                 s_depth, s_anc);
  int bad = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = 1 + threadIdx.x + i * kTreeThreads;
    if (n <= p.N) {
      s_tok[n] = tok[i];
      bad |= (tok[i] < 0 || tok[i] >= p.V);
    }
  }
  bad = __syncthreads_or(bad);
  int status = !tree_ok ? kBadTree : (bad ? kBadToken : 0);
  int node = 0, depth = 0, parity = 0;
  const T* base = reinterpret_cast<const T*>(p.target) + (long long)b * (p.N + 1) * p.V;
  while (!status) {
    __syncthreads();  // the previous step's reads of s_row / s_arg are done
    if (warp == 0) {  // the set: the node, then its children in increasing id
      int n_set = 1;
      if (lane == 0) s_row[0] = node;
      for (int c0 = 1; c0 <= p.N; c0 += kWarp) {
        const int c = c0 + lane;
        const bool kid = c <= p.N && s_par[c] == node;
        const unsigned m = __ballot_sync(0xffffffffu, kid);
        if (kid) s_row[n_set + __popc(m & ((1u << lane) - 1u))] = c;
        n_set += __popc(m);
      }
      if (lane == 0) s_nrow = n_set;
    }
    __syncthreads();
    const int nrow = s_nrow;
    // each warp reduces its chunks of every row of the set, kRowBatch rows'
    // loads in flight at once
    for (int r0 = 0; r0 < nrow; r0 += kRowBatch) {
      float2 best[kRowBatch];
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j) best[j] = make_float2(-INFINITY, __int_as_float(0x7fffffff));
      bool first = true;
      for (int c = gw; c < p.NC; c += W) {
        typename L::Raw raw[kRowBatch][L::NV];
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j)
          if (r0 + j < nrow) load_chunk<T, VEC>(base + (long long)s_row[r0 + j] * p.V, p.V, c, raw[j]);
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j)
          if (r0 + j < nrow) {
            const float2 r = chunk_argmax<T, VEC>(raw[j], c * kChunk);
            if (first || r.x > best[j].x || (r.x != r.x && best[j].x == best[j].x)) best[j] = r;
          }
        first = false;
      }
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j)
          if (r0 + j < nrow) s_warp[warp][r0 + j] = best[j];
    }
    __syncthreads();
    // this CTA's result per row, then the cluster's
    for (int r = warp; r < nrow; r += kTreeWarps) {
      float2 v = lane < kTreeWarps ? s_warp[lane][r]
                                   : make_float2(-INFINITY, __int_as_float(0x7fffffff));
      v = warp_combine_argmax(v);
      if (lane == 0) s_cta[parity][r] = v;
    }
    cluster.sync();
    for (int r = warp; r < nrow; r += kTreeWarps) {
      float2 v = make_float2(-INFINITY, __int_as_float(0x7fffffff));
      if (lane < CL) v = *cluster.map_shared_rank(&s_cta[parity][r], lane);
      v = warp_combine_argmax(v);
      if (lane == 0) s_arg[r] = is_finite(v.x) ? __float_as_int(v.y) : 0x7fffffff;
    }
    __syncthreads();
    // the node's argmax picks the child; the child's (already reduced) picks
    // the grandchild, where the next step starts
    const int a = s_arg[0];
    if (a == 0x7fffffff) {
      status = kBadLogits;
      break;
    }
    if (threadIdx.x == 0) {
      s_path[depth] = node;
      s_out[depth] = a;
    }
    ++depth;
    const int c = child_with_token(s_par, s_tok, p.N, node, a);
    if (!c) break;
    int rc = 1;  // the child's place in the set (children follow in increasing id)
    while (s_row[rc] != c) ++rc;
    const int ac = s_arg[rc];
    if (ac == 0x7fffffff) {
      status = kBadLogits;
      break;
    }
    if (threadIdx.x == 0) {
      s_path[depth] = c;
      s_out[depth] = ac;
    }
    ++depth;
    const int g = child_with_token(s_par, s_tok, p.N, c, ac);
    if (!g) break;
    node = g;
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

template <typename T, int VEC>
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tree_kernel<T, VEC>, p);
}

}  // namespace

cudaError_t launch_tree(int dtype, bool vec, const TreeParams& p, cudaStream_t stream) {
  if (dtype == kBF16)
    return vec ? launch_tree_typed<uint16_t, 8>(p, stream) : launch_tree_typed<uint16_t, 1>(p, stream);
  return vec ? launch_tree_typed<float, 4>(p, stream) : launch_tree_typed<float, 1>(p, stream);
}

}  // namespace sv
