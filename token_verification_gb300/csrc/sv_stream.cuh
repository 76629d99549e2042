// sv_stream.cuh - kernel A's streaming read of the logits (included by the
// translation units that launch it).
//
// Method ("【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §2.1 "算法骨架"):
// every verification rule needs, per row, the tempered softmax's maximum and
// sum (or the argmax) and the draft token's logit, which kernel A provides as
// one 8-byte record per 1024-logit chunk.
#pragma once
#include <type_traits>

#include "sv_rows.cuh"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// kernel A: chunk records (a single streaming read of the logits)
// ---------------------------------------------------------------------------

// The row of a stream item and what the chunk reductions need to know.
struct Item {
  int rowid, c0, nch, x;  // x: the row's draft token (sampling modes), else -1
  bool need;
};

template <int MODE>
__device__ __forceinline__ Item decode_item(const VerifyParams& p, uint32_t it) {
  Item k;
  if (p.flat) {  // items across row boundaries (tree calls: no draft tokens)
    const uint32_t g0 = it * (uint32_t)p.item_chunks;
    const uint32_t row = fast_div(g0, p.div_nc);
    k.rowid = (int)row;
    k.c0 = (int)(g0 - row * (uint32_t)p.NC);
    k.nch = min(p.item_chunks, p.total_chunks - (int)g0);
    k.need = true;
    k.x = -1;
    return k;
  }
  const uint32_t row = fast_div(it, p.div_tpr);  // total items < 2^31
  const int part = (int)(it - row * (uint32_t)p.TPR);
  const int b = (int)fast_div(row, p.div_r);
  const int r = (int)(row - (uint32_t)b * (uint32_t)p.R);
  const int Kb = p.draft_lens ? __ldg(p.draft_lens + b) : p.K;
  k.rowid = (int)row;
  k.c0 = part * p.item_chunks;
  k.nch = min(p.item_chunks, p.NC - k.c0);
  k.need = row_needed(p, r, Kb);
  const int i = r > p.K ? r - p.K - 1 : r;
  k.x = (MODE != kGreedy && p.draft_tokens && k.need && i < Kb)
            ? __ldg(p.draft_tokens + (long long)b * p.K + i)
            : -1;
  return k;
}

// Register-tile variant (scalar path: any V, any alignment): warps stride
// over items of G chunks.
template <int MODE, typename T, int VEC>
__global__ void __launch_bounds__(kThreads, 2) verify_rows_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  constexpr int G = L::G;
  // Launched early (programmatic dependent launch): wait for the predecessor,
  // then let the finalize kernel launch - it reads the call's inputs before
  // its own wait, which is safe once everything before this kernel is done.
  pdl_wait();
  pdl_launch_dependents();
  const int lane = lane_id();
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long t = gw; t < p.total_tasks; t += nw) {
    const Item k = decode_item<MODE>(p, (uint32_t)t);
    if (!k.need) continue;
    const T* row = item_row<T>(p, k.rowid);
    const uint32_t* mrow = item_mask(p, k.rowid);
    typename L::Raw raw[G][L::NV];
    uint32_t word[G];
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (g < k.nch) {
        load_chunk<T, VEC>(row, p.V, k.c0 + g, raw[g]);
        if (mrow) word[g] = mask_word(mrow, p.mask_words, k.c0 + g);
      }
    float2* rec = p.rec + (long long)k.rowid * p.NC;
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (g < k.nch) {
        if (mrow) allow_only_chunk<T, VEC>(raw[g], word[g]);
        record_draft_logit<T, VEC>(p, raw[g], k.c0 + g, k.rowid, k.x);
        float2 out;
        if constexpr (MODE == kTreeSample)
          out = tree_chunk_record<T, VEC>(p, raw[g], k.rowid, k.c0 + g);
        else
          out = chunk_record<MODE, T, VEC>(
              raw[g], k.c0 + g, p.cc, MODE == kOneHot ? k.x : -1,
              MODE == kTypical ? p.ent + (long long)k.rowid * p.NC + k.c0 + g : nullptr);
        if (lane == 0) rec[k.c0 + g] = out;
      }
  }
}

// Streaming variant (vector paths).  Warp 0, lane 0 is the producer: it
// takes items from the call's work counter (an item = up to kConsumers
// consecutive chunks of one row, 30 KB of bf16), and copies each item with
// one cp.async.bulk into the next of kStages shared-memory stages, together
// with the item's description.  Each consumer warp w reduces chunk w of every
// stage into one record.  A stage has a "full" mbarrier (completed by the
// copy) and an "empty" one (completed when all consumers are done with it).
// Per-request work happens in the finalize kernel, whose last CTA returns the
// work counter to zero.  After the last item the producer publishes an end
// marker.
#ifndef SV_STREAM_STAGES_BF16
#define SV_STREAM_STAGES_BF16 3
#endif
#ifndef SV_STREAM_STAGES_F32
#define SV_STREAM_STAGES_F32 3
#endif
constexpr int kStreamThreads = 512;
constexpr int kConsumers = kStreamThreads / kWarp - 1;  // 15

// Shared memory: kStages logit stages, their (full, empty) barrier pairs,
// their item descriptions and, for masked calls, the stages' mask words
// (32 words per chunk).
template <typename T>
struct Stream {
  static constexpr int kChunkBytes = kChunk * (int)sizeof(T);
  static constexpr int kStageBytes = kConsumers * kChunkBytes;
  static constexpr int kMaskChunkBytes = kChunk / 8;
  static constexpr int kMaskStageBytes = kConsumers * kMaskChunkBytes;
  static constexpr int kStages = sizeof(T) == 2 ? SV_STREAM_STAGES_BF16 : SV_STREAM_STAGES_F32;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kMetaOffset = kBarOffset + kStages * 16;
  static constexpr int kMaskOffset = kMetaOffset + kStages * 16;
  static constexpr int smem_bytes(bool masked) {
    return kMaskOffset + (masked ? kStages * kMaskStageBytes : 0);
  }
};

// One logit of a staged chunk (shared-memory byte address of the chunk),
// widened to fp32.
__device__ __forceinline__ float stage_logit(uint32_t chunk, int i, const uint16_t*) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(chunk + 2u * (uint32_t)i));
  return __uint_as_float((uint32_t)v << 16);
}
__device__ __forceinline__ float stage_logit(uint32_t chunk, int i, const float*) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(chunk + 4u * (uint32_t)i));
  return v;
}

// A chunk whose grammar mask allows at most kSparseAllowed of its tokens
// (structured output): the same record as the dense path - {max over the
// allowed tokens (NaN wins), sum of 2^((l - max) c) over them leaving out
// mask_x}, the typical calls' entropy accumulator, the draft token's logit -
// from the allowed logits alone, read from the stage.  Lane l takes the
// tokens of its mask word (32 l .. 32 l + 31 of the chunk); bits past V are
// dropped.
constexpr int kSparseAllowed = 128;

template <int MODE, typename T>
__device__ __forceinline__ float2 sparse_chunk_record(const VerifyParams& p, uint32_t chunk, int c,
                                                      uint32_t word, int rowid, int x,
                                                      float* ent) {
  const int lane = lane_id();
  const T* tag = nullptr;
  float lm = -INFINITY;
  for (uint32_t b = word; b; b &= b - 1u) lm = max_nan(lm, stage_logit(chunk, lane * kWarp + __ffs(b) - 1, tag));
  const float cm = warp_max_nan(lm);
  const int xo = x - c * kChunk;  // the draft token's logit (-inf where disallowed)
  if (xo >= 0 && xo < kChunk && lane == (xo >> 5))
    p.lx[rowid] = ((word >> (xo & 31)) & 1u) ? stage_logit(chunk, xo, tag) : -INFINITY;
  if (!is_finite(cm)) {
    if (ent && lane == 0) *ent = 0.f;
    return make_float2(cm == -INFINITY ? -INFINITY : qnan(), 0.f);
  }
  const float nb = -cm * p.cc;
  float s = 0.f, et = 0.f;
  for (uint32_t b = word; b; b &= b - 1u) {
    const int i = lane * kWarp + __ffs(b) - 1;
    if (MODE == kOneHot && i == xo) continue;
    const float a = fmaf(stage_logit(chunk, i, tag), p.cc, nb);
    const float w = ex2(a);
    s += w;
    if (ent) et = fmaf(w, fmaxf(a, -256.f), et);
  }
  if (ent) {
    et = warp_sum(et);
    if (lane == 0) *ent = et;
  }
  return make_float2(cm, warp_sum(s));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <int MODE, typename T, int VEC, bool kMasked>
__global__ void __launch_bounds__(kStreamThreads, 2) verify_stream_kernel(const VerifyParams p) {
  using L = Lane<T, VEC>;
  using ST = Stream<T>;
  constexpr int S = ST::kStages;
  extern __shared__ __align__(128) unsigned char smem[];
  // Launched early (programmatic dependent launch): wait for the predecessor,
  // then let the finalize kernel launch - it reads the call's inputs before
  // its own wait, which is safe once everything before this kernel is done.
  pdl_wait();
  pdl_launch_dependents();
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t base = smem_u32(smem);
  auto stage_of = [&](int s) { return base + s * ST::kStageBytes; };
  auto full_of = [&](int s) { return base + ST::kBarOffset + s * 16; };
  auto empty_of = [&](int s) { return full_of(s) + 8; };
  auto mask_of = [&](int s) { return base + ST::kMaskOffset + s * ST::kMaskStageBytes; };
  int4* meta = reinterpret_cast<int4*>(smem + ST::kMetaOffset);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_of(s), 1);
      mbar_init(empty_of(s), kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t total = (uint32_t)p.total_tasks;

  // Warp 0, lane 0: the producer.
  auto producer = [&]() {
    uint32_t k = 0;  // stages issued
    bool ok = true;
    auto acquire = [&](int s) {  // wait until stage s may be refilled
      return k < (uint32_t)S || mbar_wait(empty_of(s), ((k / S) - 1) & 1u, p.wait_ns);
    };
    // Items are taken from the call's work counter one at a time, the next
    // one's index fetched while the current one is copied, so every CTA
    // finishes within about one item of the others whatever its share of
    // the bandwidth; the grid goes through the rows in order.
    uint32_t next = atomicAdd(p.work, 1u);
    const unsigned long long evict_first = l2_evict_first_policy();
    while (ok) {
      const uint32_t it = next;
      if (it >= total) break;
      next = atomicAdd(p.work, 1u);
      const Item item = decode_item<MODE>(p, it);
      if (!item.need) continue;
      const int s = (int)(k % S);
      if (!acquire(s)) {
        ok = false;
        atomicOr(p.err, 1);
        break;
      }
      meta[s] = make_int4(item.rowid, item.c0, item.nch, item.x);
      const T* src = item_row<T>(p, item.rowid) + (long long)item.c0 * kChunk;
      uint32_t bytes =
          (uint32_t)(min(item.nch * kChunk, p.V - item.c0 * kChunk) * (int)sizeof(T));
      if (p.flat) {  // through the item's last chunk, rows being contiguous
        int cl = item.c0 + item.nch - 1, rows = 0;
        while (cl >= p.NC) {
          cl -= p.NC;
          ++rows;
        }
        bytes = (uint32_t)(((long long)rows * p.V + min((cl + 1) * kChunk, p.V) -
                            (long long)item.c0 * kChunk) *
                           (long long)sizeof(T));
      }
      if (p.mask_bulk) {  // the item's mask words travel with its logits
        const int w0 = item.c0 * kWarp;
        const uint32_t mbytes = (uint32_t)(min(item.nch * kWarp, p.mask_words - w0) * 4);
        mbar_arrive_expect_tx(full_of(s), bytes + mbytes);
        bulk_copy_hint(stage_of(s), src, bytes, full_of(s), evict_first);
        bulk_copy(mask_of(s), item_mask(p, item.rowid) + w0, mbytes, full_of(s));
      } else {
        mbar_arrive_expect_tx(full_of(s), bytes);
        bulk_copy_hint(stage_of(s), src, bytes, full_of(s), evict_first);
      }
      ++k;
    }
    // end marker (a stage whose full barrier completes without a copy)
    const int s = (int)(k % S);
    bool marked = false;
    if (ok && acquire(s)) {
      meta[s] = make_int4(-1, 0, 0, -1);
      mbar_arrive(full_of(s));
      marked = true;
    } else if (ok) {
      atomicOr(p.err, 1);
    }
    // No copy may be in flight when this thread leaves: wait until the last
    // copy into each slot has landed.  The marker reused the slot of copy
    // k - S, whose consumption acquire() already waited for; a parity wait
    // on that slot would now name a phase two completions back.
    for (uint32_t j = (k > (uint32_t)S ? k - S : 0) + (marked && k >= (uint32_t)S ? 1 : 0); j < k;
         ++j)
      mbar_wait(full_of((int)(j % S)), (j / S) & 1u);
  };

  // Warps 1..15: consumer w reduces chunk w of every stage.
  auto consumer = [&](const int w) {
    for (uint32_t k = 0;; ++k) {
      const int s = (int)(k % S);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(full_of(s), (k / S) & 1u, p.wait_ns));
      if (!ok) {  // the producer or a copy stopped: leave (the call reports a timeout)
        if (lane == 0) atomicOr(p.err, 1);
        break;
      }
      const int4 m = meta[s];
      if (m.x < 0) break;  // end marker
      if (kMasked && MODE != kTreeSample && w < m.z) {  // grammar-masked calls (a separate instantiation)
        const int c = m.y + w;
        const uint32_t chunk = stage_of(s) + w * ST::kChunkBytes;
        float* ent = MODE == kTypical ? p.ent + (long long)m.x * p.NC + c : nullptr;
        uint32_t word = 0;
        if (c * kWarp + lane < p.mask_words)
          word = p.mask_bulk ? reinterpret_cast<const uint32_t*>(
                                   smem + ST::kMaskOffset + s * ST::kMaskStageBytes +
                                   w * ST::kMaskChunkBytes)[lane]
                             : __ldg(item_mask(p, m.x) + c * kWarp + lane);
        const int first = c * kChunk + lane * kWarp;  // this word's first token
        if (first + kWarp > p.V) word &= first >= p.V ? 0u : (1u << (p.V - first)) - 1u;
        float2 out;
        if (MODE != kGreedy &&
            __reduce_add_sync(0xffffffffu, (unsigned)__popc(word)) <= (unsigned)kSparseAllowed) {
          out = sparse_chunk_record<MODE, T>(p, chunk, c, word, m.x, m.w, ent);
        } else {
          typename L::Raw raw[L::NV];
          load_chunk_smem<T, VEC>(chunk, p.V, c, raw);
          allow_only_chunk<T, VEC>(raw, word);
          record_draft_logit<T, VEC>(p, raw, c, m.x, m.w);
          out = chunk_record<MODE, T, VEC>(raw, c, p.cc, MODE == kOneHot ? m.w : -1, ent);
        }
        if (lane == 0) p.rec[(long long)m.x * p.NC + c] = out;
      } else if (w < m.z) {
        int c = m.y + w, row = m.x;
        uint32_t off = w * ST::kChunkBytes;
        if (!kMasked && p.flat && c >= p.NC) {  // past the end of the item's first row
          while (c >= p.NC) {
            c -= p.NC;
            ++row;
          }
          off = (uint32_t)((((long long)(row - m.x) * p.V) + (long long)(c - m.y) * kChunk) *
                           (long long)sizeof(T));
        }
        typename L::Raw raw[L::NV];
        load_chunk_smem<T, VEC>(stage_of(s) + off, p.V, c, raw);
        record_draft_logit<T, VEC>(p, raw, c, row, m.w);
        float2 out;
        if constexpr (MODE == kTreeSample)
          out = tree_chunk_record<T, VEC>(p, raw, row, c);
        else
          out = chunk_record<MODE, T, VEC>(
              raw, c, p.cc, MODE == kOneHot ? m.w : -1,
              MODE == kTypical ? p.ent + (long long)row * p.NC + c : nullptr);
        if (lane == 0) p.rec[(long long)row * p.NC + c] = out;
      }
      // this warp's values from the stage are consumed: hand it back
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_of(s));
    }
  };

  if (warp == 0) {
    if (lane == 0) producer();
  } else {
    consumer(warp - 1);
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
// Launches kernel A's streaming variant (vector paths) for a call.
template <int MODE, typename T, int VEC>
cudaError_t launch_stream(const VerifyParams& p, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  VerifyParams pc = p;
  void* args[] = {&pc};
    constexpr int smem_max = Stream<T>::smem_bytes(true);
    const int smem = Stream<T>::smem_bytes(p.mask_bulk != 0);
    const void* fn = reinterpret_cast<const void*>(verify_stream_kernel<MODE, T, VEC, false>);
    if constexpr (MODE != kTreeSample)
      if (p.mask) fn = reinterpret_cast<const void*>(verify_stream_kernel<MODE, T, VEC, true>);
    static PerDevice once[2];
    int occ = 1;
    err = per_device(once[p.mask ? 1 : 0], &occ, [&](int& v) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem_max);
      if (e != cudaSuccess) return e;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, kStreamThreads, smem_max) !=
              cudaSuccess ||
          v < 1)
        v = 1;
      return cudaSuccess;
    });
    if (err != cudaSuccess) return err;
    const long long cap = (long long)di.sms * occ;
    const int grid = (int)(p.total_tasks < cap ? p.total_tasks : cap);
    // Chained to the previous call's finalize kernel by programmatic dependent
    // launch, except behind dense-draft calls: there it measured slower
    // (one-hot B256 K5: +2.8%, dense B64 K3: -3%), so dense calls launch it
    // plainly.
    if (MODE != kDense) {
      err = launch_pdl(fn, dim3(grid), dim3(kStreamThreads), s, args, smem);
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(kStreamThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = s;
      err = cudaLaunchKernelExC(&cfg, fn, args);
    }
    if (err != cudaSuccess) return err;
  return cudaSuccess;
}

}  // namespace
}  // namespace sv
