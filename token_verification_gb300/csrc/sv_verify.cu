// sv_verify.cu - kernel A of the verification calls: one streaming read of
// the logits.
//
// Method ("【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §2.1 "算法骨架"):
// for each request, accept draft x_i with probability min(1, p_i(x_i) /
// q_i(x_i)) in position order; at the first rejection n draw from
// norm(max(0, p_n - q_n)); if all drafts are accepted draw the extra token
// from the last position's p.  Greedy rule (§11 of the same page): accept
// while x_i equals the target argmax.  Every one of these needs, per row, the
// tempered softmax's maximum and sum (or the argmax) and the draft token's
// logit, which this kernel provides.
//
// Kernel A (verify_stream_kernel; verify_rows_kernel on the scalar path;
//   both in sv_stream.cuh) reads every needed logit once and reduces each
//   1024-logit chunk of a row to one 8-byte record.  One producer thread per
//   CTA copies items of 15 consecutive chunks (30 KB of bf16) into a ring of
//   shared-memory stages with cp.async.bulk; each of the 15 consumer warps
//   reduces one chunk of every stage.  The only shared state is a work
//   counter from which the producers take their items.  This file launches
//   it per mode; the per-request work (tests, draws, packed output) is
//   kernel F's (sv_finalize.cu); filtered calls use kernel A' (sv_filter.cu)
//   instead.
#include "sv_stream.cuh"

namespace sv {
namespace {

template <int MODE, typename T, int VEC>
cudaError_t launch_records(const VerifyParams& p, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  VerifyParams pc = p;
  void* args[] = {&pc};
  // A: chunk records
  if (p.filter) {
    err = launch_filter(MODE, sizeof(T) == 2 ? kBF16 : kF32, VEC > 1, p, s);
    if (err != cudaSuccess) return err;
  } else if constexpr (VEC * sizeof(T) == 16) {
    err = launch_stream<MODE, T, VEC>(p, s);
    if (err != cudaSuccess) return err;
  } else {
    static PerDevice once;
    int occ = 1;
    err = per_device(once, &occ, [&](int& v) {
      v = blocks_per_sm(verify_rows_kernel<MODE, T, VEC>);
      return cudaSuccess;
    });
    if (err != cudaSuccess) return err;
    const int warps_per_cta = kThreads / kWarp;
    const long long want = (p.total_tasks + warps_per_cta - 1) / warps_per_cta;
    const long long cap = (long long)di.sms * occ;
    const int grid = (int)(want < cap ? want : cap);
    err = launch_pdl(reinterpret_cast<const void*>(verify_rows_kernel<MODE, T, VEC>), dim3(grid),
                     dim3(kThreads), s, args);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace

int chunks_per_task(int dtype, bool vec) {
  if (vec) return kConsumers;
  return Lane<float, 1>::G;
}

cudaError_t launch_records(int mode, int dtype, bool vec, const VerifyParams& p,
                           cudaStream_t stream) {
  auto typed = [&](auto mode_tag) -> cudaError_t {
    constexpr int M = decltype(mode_tag)::value;
    if (dtype == kBF16)
      return vec ? launch_records<M, uint16_t, 8>(p, stream)
                 : launch_records<M, uint16_t, 1>(p, stream);
    return vec ? launch_records<M, float, 4>(p, stream) : launch_records<M, float, 1>(p, stream);
  };
  switch (mode) {
    case kOneHot: return typed(std::integral_constant<int, kOneHot>());
    case kDense: return typed(std::integral_constant<int, kDense>());
    case kTypical: return typed(std::integral_constant<int, kTypical>());
    case kTreeSample: return typed(std::integral_constant<int, kTreeSample>());
    default: return typed(std::integral_constant<int, kGreedy>());
  }
}

}  // namespace sv
