// C ABI of the library: argument validation, kernel selection and launch.
// Every check that can fail runs before anything is enqueued, so an error
// status means nothing was launched. See include/nvmla.h for the contract.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "common.cuh"

namespace nvmla {

cudaError_t launch_pack(const void*, int64_t, const void*, int64_t, const int32_t*, int64_t, uint8_t*, int64_t,
                        int32_t, int32_t*, cudaStream_t);
cudaError_t launch_stage_dequant(const uint8_t*, const RowSelect&, int, uint8_t*, int32_t*, int32_t*,
                                 cudaStream_t);
cudaError_t launch_decode_mma(int fmt, const void*, const void*, const uint8_t*, const RowSelect&,
                              const int32_t*, int, int, int, float, void*, float*, void*, int, int32_t*,
                              cudaStream_t);
int mma_default_splits(int T, int H, int topk, int num_sms);
size_t mma_workspace_bytes(int T, int H, int splits);

cudaError_t launch_fp8_pack(const void*, int64_t, const void*, int64_t, const int32_t*, int64_t, uint8_t*, int64_t,
                            int32_t*, cudaStream_t);
cudaError_t launch_topk_select(const float*, int64_t, int32_t, const int32_t*, int32_t, int32_t, int32_t*,
                               cudaStream_t);

// tcgen05 path (decode_tc.cu)
bool tc_supported(int H);
bool tc_fp8_rows_supported(int H);
int tc_default_splits(int T, int H, int topk, int num_sms);
int tc_max_splits();
size_t tc_workspace_bytes(int T, int H, int splits);
cudaError_t launch_decode_tc(int fmt, const void*, const void*, const uint8_t*, const RowSelect&, const int32_t*,
                             int, int, int, float, void*, float*, void*, int, int32_t*, cudaStream_t,
                             uint32_t p_wait_ns, int force_p_timeout);

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

// Launch accounting: every successful enqueue adds its kernel count.
nvmla_status counted(cudaError_t e, int kernels, const char* what);

nvmla_status fail(nvmla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
nvmla_status fail(nvmla_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

nvmla_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return NVMLA_OK;
  return fail(NVMLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

nvmla_status counted(cudaError_t e, int kernels, const char* what) {
  if (e != cudaSuccess) return cuda_status(e, what);
  g_launches.fetch_add(static_cast<uint64_t>(kernels), std::memory_order_relaxed);
  return NVMLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SM count of the current device, queried once per device (concurrent
// callers may each query it; all store the same value); without a device,
// the 152 of a GB300, so that host-only callers (split counts, workspace
// sizes) see the shapes the device would use
int num_sms() {
  static std::atomic<int> cached[kMaxHostDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxHostDevices) {
    cudaGetLastError();
    return 152;
  }
  const int known = cached[dev].load(std::memory_order_relaxed);
  if (known > 0) return known;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

struct DecodeShape {
  int T, H, topk;
};

nvmla_status check_shape(int32_t T, int32_t H, int32_t topk, float sm_scale) {
  if (T < 0) return fail(NVMLA_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  if (T > NVMLA_MAX_TOKENS) return fail(NVMLA_ERR_UNSUPPORTED, "T = %d exceeds %d", T, NVMLA_MAX_TOKENS);
  if (H <= 0 || H % 16 != 0) return fail(NVMLA_ERR_UNSUPPORTED, "H = %d must be a positive multiple of 16", H);
  if (H > NVMLA_MAX_HEADS) return fail(NVMLA_ERR_UNSUPPORTED, "H = %d exceeds %d", H, NVMLA_MAX_HEADS);
  if (topk < 1 || topk > NVMLA_MAX_TOPK) return fail(NVMLA_ERR_UNSUPPORTED, "topk = %d must be in [1, %d]", topk, NVMLA_MAX_TOPK);
  if (!std::isfinite(sm_scale)) return fail(NVMLA_ERR_INVALID_ARG, "sm_scale must be finite");
  if (static_cast<int64_t>(T) * topk >= (int64_t{1} << 31)) return fail(NVMLA_ERR_UNSUPPORTED, "T * topk too large");
  return NVMLA_OK;
}

nvmla_status check_queries(const void* q_latent, const void* q_rope, const void* out, const float* lse) {
  if (!q_latent || !q_rope || !out || !lse) return fail(NVMLA_ERR_INVALID_ARG, "null q_latent/q_rope/out/lse");
  if (!aligned(q_latent, 16) || !aligned(q_rope, 16)) return fail(NVMLA_ERR_INVALID_ARG, "q_latent and q_rope must be 16-byte aligned");
  if (!aligned(out, 16)) return fail(NVMLA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(NVMLA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  return NVMLA_OK;
}

nvmla_status check_cache(const uint8_t* cache, int64_t num_pages, const int32_t* block_table, int32_t num_seqs,
                         int32_t max_pages, const int32_t* topk_idx) {
  if (!cache || !block_table || !topk_idx) return fail(NVMLA_ERR_INVALID_ARG, "null cache/block_table/topk_idx");
  if (!aligned(cache, 32)) return fail(NVMLA_ERR_INVALID_ARG, "cache must be 32-byte aligned");
  if (num_pages < 1) return fail(NVMLA_ERR_INVALID_ARG, "num_pages = %lld must be >= 1", (long long)num_pages);
  if (num_pages * NVMLA_PAGE_TOKENS >= (int64_t{1} << 31)) return fail(NVMLA_ERR_UNSUPPORTED, "cache has 2^31 slots or more");
  if (num_seqs < 1 || max_pages < 1) return fail(NVMLA_ERR_INVALID_ARG, "num_seqs and max_pages_per_seq must be >= 1");
  if (!aligned(block_table, 4) || !aligned(topk_idx, 4)) return fail(NVMLA_ERR_INVALID_ARG, "index arrays must be 4-byte aligned");
  return NVMLA_OK;
}

// A layer of a block-major multi-layer cache ([num_blocks][num_layers][64]
// rows): its rows start layer * 64 rows in, and blocks lie 64 * num_layers
// rows apart. One layer per cache is num_layers = 1, layer = 0.
constexpr int32_t kMaxLayers = 4096;
nvmla_status check_layers(int64_t num_blocks, int32_t num_layers, int32_t layer) {
  if (num_layers < 1 || num_layers > kMaxLayers)
    return fail(NVMLA_ERR_INVALID_ARG, "num_layers = %d must be in [1, %d]", num_layers, kMaxLayers);
  if (layer < 0 || layer >= num_layers)
    return fail(NVMLA_ERR_INVALID_ARG, "layer = %d must be in [0, num_layers = %d)", layer, num_layers);
  if (num_blocks >= (int64_t{1} << 40) / num_layers)
    return fail(NVMLA_ERR_UNSUPPORTED, "num_blocks * num_layers too large");
  return NVMLA_OK;
}
int64_t layer_offset(int32_t layer) { return static_cast<int64_t>(layer) * NVMLA_PAGE_TOKENS * NVMLA_ROW_BYTES; }

int pick_impl(const nvmla_decode_options* opts, int H) {
  const int want = opts ? opts->impl : NVMLA_IMPL_AUTO;
  if (want == NVMLA_IMPL_MMA) return NVMLA_IMPL_MMA;
  if (want == NVMLA_IMPL_TCGEN05) return NVMLA_IMPL_TCGEN05;
  return tc_supported(H) ? NVMLA_IMPL_TCGEN05 : NVMLA_IMPL_MMA;
}

bool tc_fp8_supported(int H) { return tc_fp8_rows_supported(H); }

int pick_impl_fp8(const nvmla_decode_options* opts, int H) {
  const int want = opts ? opts->impl : NVMLA_IMPL_AUTO;
  if (want == NVMLA_IMPL_MMA) return NVMLA_IMPL_MMA;
  if (want == NVMLA_IMPL_TCGEN05) return NVMLA_IMPL_TCGEN05;
  return tc_fp8_supported(H) ? NVMLA_IMPL_TCGEN05 : NVMLA_IMPL_MMA;
}

// The test hook that makes the tcgen05 kernel's wait for P^T give up at once.
int force_timeout(const nvmla_decode_options* opts) {
  return (opts && (opts->debug_flags & NVMLA_DEBUG_FORCE_WAIT_TIMEOUT)) ? 1 : 0;
}

// Split count for the mma kernel that fits the workspace (explicit requests
// must fit; the heuristic falls back to fewer splits).
int impl_tile(int impl) { return impl == NVMLA_IMPL_TCGEN05 ? 128 : 64; }

int default_splits(int impl, int T, int H, int topk) {
  return impl == NVMLA_IMPL_TCGEN05 ? tc_default_splits(T, H, topk, num_sms()) : mma_default_splits(T, H, topk, num_sms());
}

size_t workspace_bytes(int impl, int T, int H, int splits) {
  return impl == NVMLA_IMPL_TCGEN05 ? tc_workspace_bytes(T, H, splits) : mma_workspace_bytes(T, H, splits);
}

nvmla_status pick_splits(int impl, const nvmla_decode_options* opts, int T, int H, int topk, size_t ws_bytes,
                         const void* ws, int* splits) {
  const int tiles = (topk + impl_tile(impl) - 1) / impl_tile(impl);
  int s = (opts && opts->num_splits > 0) ? opts->num_splits : default_splits(impl, T, H, topk);
  if (s > tiles) s = tiles;
  if (s < 1) s = 1;
  const bool explicit_req = opts && opts->num_splits > 0;
  auto too_small = [&](int n) {
    const size_t need = workspace_bytes(impl, T, H, n);
    return need > 0 && (!ws || need > ws_bytes);
  };
  if (s > 1 && too_small(s)) {
    if (explicit_req)
      return fail(NVMLA_ERR_WORKSPACE, "num_splits = %d needs %zu workspace bytes, got %zu", s,
                  workspace_bytes(impl, T, H, s), ws ? ws_bytes : size_t(0));
    while (s > 1 && too_small(s)) --s;
  }
  if (impl == NVMLA_IMPL_TCGEN05 && s > tc_max_splits())
    return fail(NVMLA_ERR_UNSUPPORTED, "num_splits = %d exceeds the %d CTAs a cluster can hold on this device", s,
                tc_max_splits());
  if (ws && !aligned(ws, 16)) return fail(NVMLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  *splits = s;
  return NVMLA_OK;
}

}  // namespace

// Records `msg` as the calling thread's last error and returns `s` (for the
// entry points defined in other translation units).
nvmla_status record_error(nvmla_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace nvmla

using namespace nvmla;

extern "C" {

const char* nvmla_status_string(nvmla_status s) {
  switch (s) {
    case NVMLA_OK: return "NVMLA_OK";
    case NVMLA_ERR_INVALID_ARG: return "NVMLA_ERR_INVALID_ARG";
    case NVMLA_ERR_UNSUPPORTED: return "NVMLA_ERR_UNSUPPORTED";
    case NVMLA_ERR_CUDA: return "NVMLA_ERR_CUDA";
    case NVMLA_ERR_WORKSPACE: return "NVMLA_ERR_WORKSPACE";
  }
  return "NVMLA_UNKNOWN_STATUS";
}

const char* nvmla_last_error(void) { return g_last_error.c_str(); }

int32_t nvmla_version(void) { return 200; }

uint64_t nvmla_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t nvmla_build_flags(void) {
#ifdef NVMLA_DEBUG_BOUNDS
  return NVMLA_BUILD_DEBUG_BOUNDS;
#else
  return 0;
#endif
}

namespace {
nvmla_status pack_impl(const void* latent_bf16, int64_t latent_stride, const void* rope_bf16, int64_t rope_stride,
                       const int32_t* slot_mapping, int64_t n_tokens, uint8_t* cache, int64_t num_blocks,
                       int32_t num_layers, int32_t layer, int32_t* err_word, nvmla_stream_t stream) {
  if (n_tokens < 0) return fail(NVMLA_ERR_INVALID_ARG, "n_tokens = %lld must be >= 0", (long long)n_tokens);
  if (n_tokens == 0) return NVMLA_OK;
  if (!latent_bf16 || !rope_bf16 || !slot_mapping || !cache)
    return fail(NVMLA_ERR_INVALID_ARG, "null latent/rope/slot_mapping/cache");
  if (!aligned(latent_bf16, 16) || latent_stride < NVMLA_LATENT_DIM || latent_stride % 8 != 0)
    return fail(NVMLA_ERR_INVALID_ARG, "latent must be 16-byte aligned with a stride >= 512 and a multiple of 8");
  if (!aligned(rope_bf16, 4) || rope_stride < NVMLA_ROPE_DIM || rope_stride % 2 != 0)
    return fail(NVMLA_ERR_INVALID_ARG, "rope must be 4-byte aligned with an even stride >= 64");
  if (!aligned(slot_mapping, 4)) return fail(NVMLA_ERR_INVALID_ARG, "slot_mapping must be 4-byte aligned");
  if (!aligned(cache, 32)) return fail(NVMLA_ERR_INVALID_ARG, "cache must be 32-byte aligned");
  if (num_blocks < 1) return fail(NVMLA_ERR_INVALID_ARG, "num_pages = %lld must be >= 1", (long long)num_blocks);
  nvmla_status s = check_layers(num_blocks, num_layers, layer);
  if (s != NVMLA_OK) return s;
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  return counted(launch_pack(latent_bf16, latent_stride, rope_bf16, rope_stride, slot_mapping, n_tokens,
                             cache + layer_offset(layer), num_blocks, NVMLA_PAGE_TOKENS * num_layers, err_word,
                             reinterpret_cast<cudaStream_t>(stream)),
                 1, "nvfp4_mla_pack launch");
}
}  // namespace

nvmla_status nvfp4_mla_pack(const void* latent_bf16, int64_t latent_stride, const void* rope_bf16,
                            int64_t rope_stride, const int32_t* slot_mapping, int64_t n_tokens, uint8_t* cache,
                            int64_t num_pages, int32_t* err_word, nvmla_stream_t stream) {
  return pack_impl(latent_bf16, latent_stride, rope_bf16, rope_stride, slot_mapping, n_tokens, cache, num_pages, 1, 0,
                   err_word, stream);
}

nvmla_status nvfp4_mla_pack_layered(const void* latent_bf16, int64_t latent_stride, const void* rope_bf16,
                                    int64_t rope_stride, const int32_t* slot_mapping, int64_t n_tokens,
                                    uint8_t* cache, int64_t num_blocks, int32_t num_layers, int32_t layer,
                                    int32_t* err_word, nvmla_stream_t stream) {
  return pack_impl(latent_bf16, latent_stride, rope_bf16, rope_stride, slot_mapping, n_tokens, cache, num_blocks,
                   num_layers, layer, err_word, stream);
}

size_t sparse_mla_decode_workspace_size_ex(int32_t T, int32_t H, int32_t topk, const nvmla_decode_options* opts) {
  if (T <= 0 || H <= 0 || H % 16 != 0 || H > NVMLA_MAX_HEADS || topk < 1 || topk > NVMLA_MAX_TOPK) return 0;
  const int impl = pick_impl(opts, H);
  if (impl == NVMLA_IMPL_TCGEN05 && !tc_supported(H)) return 0;
  const int tiles = (topk + impl_tile(impl) - 1) / impl_tile(impl);
  int s = (opts && opts->num_splits > 0) ? opts->num_splits : default_splits(impl, T, H, topk);
  if (s > tiles) s = tiles;
  if (s < 1) s = 1;
  return workspace_bytes(impl, T, H, s);
}

int32_t sparse_mla_decode_splits(int32_t T, int32_t H, int32_t topk, const nvmla_decode_options* opts) {
  if (T <= 0 || H <= 0 || H % 16 != 0 || H > NVMLA_MAX_HEADS || topk < 1 || topk > NVMLA_MAX_TOPK) return 0;
  const int impl = pick_impl(opts, H);
  if (impl == NVMLA_IMPL_TCGEN05 && !tc_supported(H)) return 0;
  const int tiles = (topk + impl_tile(impl) - 1) / impl_tile(impl);
  int s = (opts && opts->num_splits > 0) ? opts->num_splits : default_splits(impl, T, H, topk);
  if (s > tiles) s = tiles;
  if (s < 1) s = 1;
  return s;
}

size_t sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t topk) {
  return sparse_mla_decode_workspace_size_ex(T, H, topk, nullptr);
}

size_t sparse_mla_decode_fp8rows_workspace_size(int32_t T, int32_t H, int32_t topk, const nvmla_decode_options* opts) {
  if (T <= 0 || H <= 0 || H % 16 != 0 || H > NVMLA_MAX_HEADS || topk < 1 || topk > NVMLA_MAX_TOPK) return 0;
  const int impl = pick_impl_fp8(opts, H);
  if (impl == NVMLA_IMPL_TCGEN05 && !tc_fp8_supported(H)) return 0;
  const int tiles = (topk + impl_tile(impl) - 1) / impl_tile(impl);
  int s = (opts && opts->num_splits > 0) ? opts->num_splits : default_splits(impl, T, H, topk);
  if (s > tiles) s = tiles;
  if (s < 1) s = 1;
  return workspace_bytes(impl, T, H, s);
}

namespace {
nvmla_status decode_impl(const void* q_latent, const void* q_rope, const uint8_t* cache, int64_t num_blocks,
                         int32_t num_layers, int32_t layer, const int32_t* block_table, int32_t num_seqs,
                         int32_t max_pages_per_seq, const int32_t* topk_idx, int32_t topk, const int32_t* q_seq_idx,
                         const int32_t* seq_lens, int32_t T, int32_t H, float sm_scale, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, int32_t* err_word,
                         const nvmla_decode_options* opts, nvmla_stream_t stream) {
  nvmla_status s = check_shape(T, H, topk, sm_scale);
  if (s != NVMLA_OK || T == 0) return s;
  if ((s = check_queries(q_latent, q_rope, out, lse)) != NVMLA_OK) return s;
  if ((s = check_cache(cache, num_blocks, block_table, num_seqs, max_pages_per_seq, topk_idx)) != NVMLA_OK) return s;
  if ((s = check_layers(num_blocks, num_layers, layer)) != NVMLA_OK) return s;
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  if (opts && (opts->impl < 0 || opts->impl > NVMLA_IMPL_TCGEN05 || opts->num_splits < 0 ||
               (opts->debug_flags & ~NVMLA_DEBUG_FORCE_WAIT_TIMEOUT) != 0))
    return fail(NVMLA_ERR_INVALID_ARG, "bad options");
  RowSelect sel{topk_idx, block_table, q_seq_idx, seq_lens, num_blocks * NVMLA_PAGE_TOKENS, topk, max_pages_per_seq,
                num_seqs, NVMLA_PAGE_TOKENS * num_layers};
  const uint8_t* rows = cache + layer_offset(layer);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int impl = pick_impl(opts, H);
  if (impl == NVMLA_IMPL_TCGEN05 && !tc_supported(H))
    return fail(NVMLA_ERR_UNSUPPORTED, "the tcgen05 kernel needs H a multiple of 64 (H = %d)", H);
  int splits = 1;
  if ((s = pick_splits(impl, opts, T, H, topk, workspace_bytes, workspace, &splits)) != NVMLA_OK) return s;
  if (impl == NVMLA_IMPL_TCGEN05) {
    return counted(launch_decode_tc(0, q_latent, q_rope, rows, sel, nullptr, T, H, topk, sm_scale, out, lse,
                                    workspace, splits, err_word, st, 0, force_timeout(opts)),
                   1, "sparse_mla_decode (tcgen05) launch");
  }
  return counted(launch_decode_mma(0, q_latent, q_rope, rows, sel, nullptr, T, H, topk, sm_scale, out, lse,
                                   workspace, splits, err_word, st),
                 splits > 1 ? 2 : 1, "sparse_mla_decode (mma) launch");
}
}  // namespace

nvmla_status sparse_mla_decode_ex(const void* q_latent, const void* q_rope, const uint8_t* cache, int64_t num_pages,
                                  const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq,
                                  const int32_t* topk_idx, int32_t topk, const int32_t* q_seq_idx,
                                  const int32_t* seq_lens, int32_t T, int32_t H, float sm_scale, void* out,
                                  float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                  const nvmla_decode_options* opts, nvmla_stream_t stream) {
  return decode_impl(q_latent, q_rope, cache, num_pages, 1, 0, block_table, num_seqs, max_pages_per_seq, topk_idx,
                     topk, q_seq_idx, seq_lens, T, H, sm_scale, out, lse, workspace, workspace_bytes, err_word, opts,
                     stream);
}

nvmla_status sparse_mla_decode_layered(const void* q_latent, const void* q_rope, const uint8_t* cache,
                                       int64_t num_blocks, int32_t num_layers, int32_t layer,
                                       const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq,
                                       const int32_t* topk_idx, int32_t topk, const int32_t* q_seq_idx,
                                       const int32_t* seq_lens, int32_t T, int32_t H, float sm_scale, void* out,
                                       float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                       const nvmla_decode_options* opts, nvmla_stream_t stream) {
  return decode_impl(q_latent, q_rope, cache, num_blocks, num_layers, layer, block_table, num_seqs, max_pages_per_seq,
                     topk_idx, topk, q_seq_idx, seq_lens, T, H, sm_scale, out, lse, workspace, workspace_bytes,
                     err_word, opts, stream);
}

nvmla_status sparse_mla_decode(const void* q_latent, const void* q_rope, const uint8_t* cache, int64_t num_pages,
                               const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq,
                               const int32_t* topk_idx, int32_t topk, const int32_t* q_seq_idx,
                               const int32_t* seq_lens, int32_t T, int32_t H, float sm_scale, void* out, float* lse,
                               void* workspace, size_t workspace_bytes, int32_t* err_word, nvmla_stream_t stream) {
  return sparse_mla_decode_ex(q_latent, q_rope, cache, num_pages, block_table, num_seqs, max_pages_per_seq, topk_idx,
                              topk, q_seq_idx, seq_lens, T, H, sm_scale, out, lse, workspace, workspace_bytes,
                              err_word, nullptr, stream);
}

nvmla_status fp8_mla_pack(const void* latent_bf16, int64_t latent_stride, const void* rope_bf16, int64_t rope_stride,
                          const int32_t* slot_mapping, int64_t n_tokens, uint8_t* cache, int64_t num_pages,
                          int32_t* err_word, nvmla_stream_t stream) {
  if (n_tokens < 0) return fail(NVMLA_ERR_INVALID_ARG, "n_tokens = %lld must be >= 0", (long long)n_tokens);
  if (n_tokens == 0) return NVMLA_OK;
  if (!latent_bf16 || !rope_bf16 || !slot_mapping || !cache)
    return fail(NVMLA_ERR_INVALID_ARG, "null latent/rope/slot_mapping/cache");
  if (!aligned(latent_bf16, 16) || latent_stride < NVMLA_LATENT_DIM || latent_stride % 8 != 0)
    return fail(NVMLA_ERR_INVALID_ARG, "latent must be 16-byte aligned with a stride >= 512 and a multiple of 8");
  if (!aligned(rope_bf16, 4) || rope_stride < NVMLA_ROPE_DIM || rope_stride % 2 != 0)
    return fail(NVMLA_ERR_INVALID_ARG, "rope must be 4-byte aligned with an even stride >= 64");
  if (!aligned(slot_mapping, 4)) return fail(NVMLA_ERR_INVALID_ARG, "slot_mapping must be 4-byte aligned");
  if (!aligned(cache, 32)) return fail(NVMLA_ERR_INVALID_ARG, "cache must be 32-byte aligned");
  if (num_pages < 1) return fail(NVMLA_ERR_INVALID_ARG, "num_pages = %lld must be >= 1", (long long)num_pages);
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  return counted(launch_fp8_pack(latent_bf16, latent_stride, rope_bf16, rope_stride, slot_mapping, n_tokens, cache,
                                 num_pages, err_word, reinterpret_cast<cudaStream_t>(stream)),
                 1, "fp8_mla_pack launch");
}

nvmla_status sparse_mla_decode_fp8cache(const void* q_latent, const void* q_rope, const uint8_t* cache,
                                        int64_t num_pages, const int32_t* block_table, int32_t num_seqs,
                                        int32_t max_pages_per_seq, const int32_t* topk_idx, int32_t topk,
                                        const int32_t* q_seq_idx, const int32_t* seq_lens, int32_t T, int32_t H,
                                        float sm_scale, void* out, float* lse, void* workspace,
                                        size_t workspace_bytes, int32_t* err_word, const nvmla_decode_options* opts,
                                        nvmla_stream_t stream) {
  nvmla_status s = check_shape(T, H, topk, sm_scale);
  if (s != NVMLA_OK || T == 0) return s;
  if ((s = check_queries(q_latent, q_rope, out, lse)) != NVMLA_OK) return s;
  if ((s = check_cache(cache, num_pages, block_table, num_seqs, max_pages_per_seq, topk_idx)) != NVMLA_OK) return s;
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  if (opts && (opts->impl < 0 || opts->impl > NVMLA_IMPL_TCGEN05 || opts->num_splits < 0 ||
               (opts->debug_flags & ~NVMLA_DEBUG_FORCE_WAIT_TIMEOUT) != 0))
    return fail(NVMLA_ERR_INVALID_ARG, "bad options");
  if ((opts && opts->impl == NVMLA_IMPL_MMA) || !tc_supported(H))
    return fail(NVMLA_ERR_UNSUPPORTED, "the FP8-cache decode runs on the tcgen05 kernel: H a multiple of 64 (H = %d)",
                H);
  nvmla_decode_options o{NVMLA_IMPL_TCGEN05, opts ? opts->num_splits : 0, 0};
  int splits = 1;
  if ((s = pick_splits(NVMLA_IMPL_TCGEN05, &o, T, H, topk, workspace_bytes, workspace, &splits)) != NVMLA_OK) return s;
  RowSelect sel{topk_idx, block_table, q_seq_idx, seq_lens, num_pages * NVMLA_PAGE_TOKENS, topk, max_pages_per_seq,
                num_seqs, NVMLA_PAGE_TOKENS};
  return counted(launch_decode_tc(2, q_latent, q_rope, cache, sel, nullptr, T, H, topk, sm_scale, out, lse, workspace,
                                  splits, err_word, reinterpret_cast<cudaStream_t>(stream), 0, force_timeout(opts)),
                 1, "sparse_mla_decode_fp8cache launch");
}

nvmla_status nvmla_topk_select(const float* scores, int64_t row_stride, int32_t ncols, const int32_t* lengths,
                               int32_t T, int32_t topk, int32_t* topk_idx, nvmla_stream_t stream) {
  if (T < 0) return fail(NVMLA_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  if (topk < 1 || topk > NVMLA_MAX_TOPK)
    return fail(NVMLA_ERR_UNSUPPORTED, "topk = %d must be in [1, %d]", topk, NVMLA_MAX_TOPK);
  if (T > NVMLA_MAX_TOKENS) return fail(NVMLA_ERR_UNSUPPORTED, "T = %d exceeds %d", T, NVMLA_MAX_TOKENS);
  if (ncols < 0) return fail(NVMLA_ERR_INVALID_ARG, "ncols = %d must be >= 0", ncols);
  if (ncols > NVMLA_MAX_TOPK_COLS) return fail(NVMLA_ERR_UNSUPPORTED, "ncols = %d exceeds %d", ncols, NVMLA_MAX_TOPK_COLS);
  if (row_stride < ncols) return fail(NVMLA_ERR_INVALID_ARG, "row_stride must be >= ncols");
  if (T == 0) return NVMLA_OK;
  if ((!scores && ncols > 0) || !topk_idx) return fail(NVMLA_ERR_INVALID_ARG, "null scores/topk_idx");
  if (!aligned(scores, 4) || !aligned(topk_idx, 4) || (lengths && !aligned(lengths, 4)))
    return fail(NVMLA_ERR_INVALID_ARG, "scores, lengths and topk_idx must be 4-byte aligned");
  return counted(launch_topk_select(scores, row_stride, ncols, lengths, T, topk, topk_idx,
                                    reinterpret_cast<cudaStream_t>(stream)),
                 1, "nvmla_topk_select launch");
}

nvmla_status nvfp4_stage_dequant_fp8(const uint8_t* cache, int64_t num_pages, const int32_t* block_table,
                                     int32_t num_seqs, int32_t max_pages_per_seq, const int32_t* topk_idx,
                                     int32_t topk, const int32_t* q_seq_idx, const int32_t* seq_lens, int32_t T,
                                     uint8_t* fp8_rows, int32_t* row_idx, int32_t* err_word, nvmla_stream_t stream) {
  if (T < 0) return fail(NVMLA_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  if (topk < 1 || topk > NVMLA_MAX_TOPK) return fail(NVMLA_ERR_UNSUPPORTED, "topk = %d must be in [1, %d]", topk, NVMLA_MAX_TOPK);
  if (T == 0) return NVMLA_OK;
  nvmla_status s = check_cache(cache, num_pages, block_table, num_seqs, max_pages_per_seq, topk_idx);
  if (s != NVMLA_OK) return s;
  if (!fp8_rows || !row_idx) return fail(NVMLA_ERR_INVALID_ARG, "null fp8_rows/row_idx");
  if (!aligned(fp8_rows, 16) || !aligned(row_idx, 4)) return fail(NVMLA_ERR_INVALID_ARG, "fp8_rows must be 16-byte aligned");
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  RowSelect sel{topk_idx, block_table, q_seq_idx, seq_lens, num_pages * NVMLA_PAGE_TOKENS, topk, max_pages_per_seq,
                num_seqs, NVMLA_PAGE_TOKENS};
  return counted(launch_stage_dequant(cache, sel, T, fp8_rows, row_idx, err_word, reinterpret_cast<cudaStream_t>(stream)),
                 1, "nvfp4_stage_dequant_fp8 launch");
}

nvmla_status sparse_mla_decode_fp8rows(const void* q_latent, const void* q_rope, const uint8_t* fp8_rows,
                                       const int32_t* row_idx, int32_t topk, int32_t T, int32_t H, float sm_scale,
                                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                                       int32_t* err_word, const nvmla_decode_options* opts, nvmla_stream_t stream) {
  nvmla_status s = check_shape(T, H, topk, sm_scale);
  if (s != NVMLA_OK || T == 0) return s;
  if ((s = check_queries(q_latent, q_rope, out, lse)) != NVMLA_OK) return s;
  if (!fp8_rows || !row_idx) return fail(NVMLA_ERR_INVALID_ARG, "null fp8_rows/row_idx");
  if (!aligned(fp8_rows, 16) || !aligned(row_idx, 4)) return fail(NVMLA_ERR_INVALID_ARG, "fp8_rows must be 16-byte aligned");
  if (err_word && !aligned(err_word, 4)) return fail(NVMLA_ERR_INVALID_ARG, "err_word must be 4-byte aligned");
  if (opts && (opts->impl < 0 || opts->impl > NVMLA_IMPL_TCGEN05 || opts->num_splits < 0 ||
               (opts->debug_flags & ~NVMLA_DEBUG_FORCE_WAIT_TIMEOUT) != 0))
    return fail(NVMLA_ERR_INVALID_ARG, "bad options");
  RowSelect sel{};
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int impl = pick_impl_fp8(opts, H);
  if (impl == NVMLA_IMPL_TCGEN05 && !tc_fp8_supported(H))
    return fail(NVMLA_ERR_UNSUPPORTED, "no tcgen05 kernel for FP8 rows with H = %d", H);
  int splits = 1;
  if ((s = pick_splits(impl, opts, T, H, topk, workspace_bytes, workspace, &splits)) != NVMLA_OK) return s;
  if (impl == NVMLA_IMPL_TCGEN05) {
    return counted(launch_decode_tc(1, q_latent, q_rope, fp8_rows, sel, row_idx, T, H, topk, sm_scale, out, lse,
                                    workspace, splits, err_word, st, 0, 0),
                   splits > 1 ? 2 : 1, "sparse_mla_decode_fp8rows (tcgen05) launch");
  }
  return counted(launch_decode_mma(1, q_latent, q_rope, fp8_rows, sel, row_idx, T, H, topk, sm_scale, out, lse,
                                   workspace, splits, err_word, st),
                 splits > 1 ? 2 : 1, "sparse_mla_decode_fp8rows (mma) launch");
}

}  // extern "C"
