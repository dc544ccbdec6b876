// sparse_mla_decode_noalloc: sparse_mla_decode for callers that cannot
// allocate GPU memory.
//
// sparse_mla_decode splits each token's keys across CTAs and needs a scratch
// workspace for the partial results of the splits, which its caller
// allocates. Some callers cannot: a serving engine that hands the whole GPU
// memory to its own pool at start-up and must not see an allocation outside
// it, a step replayed from a fixed launch sequence in which no allocator
// call may appear, or a plain C caller with no device allocator of its own.
// This entry point takes the scratch from one array in device memory that
// belongs to the library, so the caller passes only inputs and outputs and
// nothing is allocated by the call.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace nvmla {
nvmla_status record_error(nvmla_status s, const char* msg);
}

namespace {

// The library's split scratch: reserved on a device when this library's
// code is loaded there (on first use of this entry point under CUDA's lazy
// module loading) and held until the process exits. Nothing in it has to
// start at zero: every call writes each partial before its merge reads it.
// A call whose pipeline wait timed out (NVMLA_ERRW_WAIT_TIMEOUT) may merge
// stale partials, but its output is invalid in any case.
constexpr size_t kScratchBytes = size_t{16} << 20;
__device__ __align__(256) unsigned char nvmla_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per
// device and kept: it belongs to the device's primary context, so a
// cudaDeviceReset (which destroys that context and unloads this module)
// leaves a stale address; the header tells callers not to call again after
// one.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, nvmla_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = ptr;
  }
  *out = g_scratch[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t sparse_mla_decode_noalloc_max_scratch(void) { return kScratchBytes; }

nvmla_status sparse_mla_decode_noalloc(const void* q_latent, const void* q_rope, const uint8_t* cache,
                                       int64_t num_pages, const int32_t* block_table, int32_t num_seqs,
                                       int32_t max_pages_per_seq, const int32_t* topk_idx, int32_t topk,
                                       const int32_t* q_seq_idx, const int32_t* seq_lens, int32_t T, int32_t H,
                                       float sm_scale, void* out, float* lse, int32_t* err_word,
                                       nvmla_stream_t stream) {
  // the same split choice as sparse_mla_decode with a full workspace, so the
  // two calls give the same bits
  const size_t need = sparse_mla_decode_workspace_size(T, H, topk);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "sparse_mla_decode_noalloc: T = %d, H = %d, topk = %d needs %zu bytes of split scratch, more than "
             "the %zu the library holds; call sparse_mla_decode with a workspace instead",
             T, H, topk, need, kScratchBytes);
    return nvmla::record_error(NVMLA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "sparse_mla_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      return nvmla::record_error(NVMLA_ERR_CUDA, msg);
    }
  }
  return sparse_mla_decode(q_latent, q_rope, cache, num_pages, block_table, num_seqs, max_pages_per_seq, topk_idx,
                           topk, q_seq_idx, seq_lens, T, H, sm_scale, out, lse, scratch, need, err_word, stream);
}

}  // extern "C"
