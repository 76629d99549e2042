// sv_noalloc.cu - spec_verify_sample without a caller-provided workspace.
//
// Some callers cannot allocate device memory: an inference runtime that
// reserves the whole device for its own pool and hands a plugin only its
// input and output buffers, or a code path on which a cudaMalloc (which may
// synchronise the device) is not allowed.  For them this entry point takes
// its scratch from one file-scope device array of SV_NOALLOC_SCRATCH_BYTES,
// which every GPU that loads the library holds until the process exits.  It
// calls no cudaMalloc, cudaFree or allocating library routine.
#include "../../include/spec_verify.h"
#include "sv_launch.h"

namespace {

// The scratch.  In host code this name only stands for the array: its
// device address comes from cudaGetSymbolAddress, with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch on the current device, looked up on every
// call: the lookup queues no work, and an address cached across calls would
// go stale if a device reset made the runtime load the module again.
cudaError_t scratch_address(void** out) {
  void* ptr = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (err != cudaSuccess) return err;
  *out = ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" sv_status spec_verify_sample_noalloc(
    const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
    const float* uniforms, float temperature, int32_t* out_tokens, int32_t* out_accept_len,
    sv_dtype dtype, int B, int K, int V, const int32_t* draft_lens, int32_t* out_cu_accept,
    int32_t* out_packed, int32_t* out_batch_id, float* out_accept_prob, int32_t* out_status,
    sv_stream_t stream) {
  const size_t need = spec_verify_workspace_size(B, K, V);
  if (need > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;  // the problem does not fit
  void* scratch = nullptr;
  if (B > 0 && need > 0) {
    if (scratch_address(&scratch) != cudaSuccess) return SV_ERR_CUDA;
    // The array keeps whatever the previous call left; the counters and flags
    // that must read zero when a call starts are cleared here (the region
    // laid out for dense drafts, which covers every mode's).
    const size_t zero = sv::workspace_layout(B, K, V).zero_bytes;
    if (cudaMemsetAsync(scratch, 0, zero, (cudaStream_t)stream) != cudaSuccess) return SV_ERR_CUDA;
  }
  return spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                            out_tokens, out_accept_len, dtype, B, K, V, draft_lens, out_cu_accept,
                            out_packed, out_batch_id, out_accept_prob, out_status, scratch,
                            scratch ? (size_t)SV_NOALLOC_SCRATCH_BYTES : 0, stream);
}
