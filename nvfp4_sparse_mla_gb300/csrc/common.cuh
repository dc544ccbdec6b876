// Shared device helpers of the NVFP4 sparse-MLA kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "format.h"
#include "nvmla.h"

namespace nvmla {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- conversions

// Two E2M1 codes (one byte: low nibble first) per f16x2, four bytes at once.
// The hardware conversion is exact: every E2M1 value is an fp16 value.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

// Four E4M3 bytes -> two f16x2.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xffffu));
  hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// (a, b) -> two E4M3 bytes, a in the low byte; round to nearest even,
// saturating to +-448 (the sign of zero is kept).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// scale byte -> f16x2 with the scale in both halves (exact)
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(byte | (byte << 8)));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- memory

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// (the memory clobbers keep the compiler from moving shared-memory accesses
// across the copies and the waits)
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void report_error(int32_t* err_word, int32_t flag, int32_t count) {
  if (err_word) {
    atomicOr(err_word, flag);
    atomicAdd(err_word + 1, count);
  }
}

// Byte offset of the row of cache slot s (block s / 64, token s % 64) when
// consecutive blocks lie page_rows rows apart: 64 for a cache that holds one
// layer, 64 L when each block keeps the rows of L layers together
// (block-major, layer-next: the layer's own rows then start at layer * 64).
__host__ __device__ __forceinline__ int64_t cache_row_offset(int64_t s, int32_t page_rows,
                                                             int row_bytes = kRowBytes) {
  return ((s >> 6) * page_rows + (s & 63)) * row_bytes;
}

// Physical cache slot of slot k of query token t, or -1 (padding or a bad
// entry; bad entries are reported once, by the caller's choice of thread).
// A token whose sequence index lies outside [0, num_seqs) has no valid slot.
struct RowSelect {
  const int32_t* topk_idx;
  const int32_t* block_table;
  const int32_t* q_seq_idx;
  const int32_t* seq_lens;
  int64_t num_slots;
  int32_t topk;
  int32_t max_pages;
  int32_t num_seqs;
  int32_t page_rows;  // rows from one block to the next (cache_row_offset)

  __device__ __forceinline__ int64_t slot(int t, int k, int32_t* err_word, bool report) const {
    const int32_t p = __ldg(topk_idx + static_cast<int64_t>(t) * topk + k);
    if (p == -1) return -1;
    const int32_t b = q_seq_idx ? __ldg(q_seq_idx + t) : 0;
    if (b < 0 || b >= num_seqs) {
      if (report) report_error(err_word, NVMLA_ERRW_BAD_INDEX, 1);
      return -1;
    }
    int64_t limit = static_cast<int64_t>(max_pages) * kPage;
    if (seq_lens) {
      const int64_t L = __ldg(seq_lens + b);
      limit = L < limit ? L : limit;
    }
    if (p < 0 || p >= limit) {
      if (report) report_error(err_word, NVMLA_ERRW_BAD_INDEX, 1);
      return -1;
    }
    const int64_t page = __ldg(block_table + static_cast<int64_t>(b) * max_pages + (p >> 6));
    const int64_t s = page * kPage + (p & 63);
    if (page < 0 || s >= num_slots) {
      if (report) report_error(err_word, NVMLA_ERRW_BAD_SLOT, 1);
      return -1;
    }
    return s;
  }
};

// ---------------------------------------------------------------- launch shape

constexpr int kMaxHostDevices = 64;

// Blocks of `kernel` (with `threads` threads and `smem` bytes of dynamic
// shared memory a block) that the current device holds at once: its SM
// count times the blocks resident per SM. Queried once per device and kept
// in `cache` (one slot per device, shared by concurrent callers: each
// computes the same value); 0 if the device or the query fails.
template <typename Kernel>
inline int resident_blocks(Kernel kernel, int threads, size_t smem, std::atomic<int> (&cache)[kMaxHostDevices]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxHostDevices) return 0;
  const int known = cache[dev].load(std::memory_order_relaxed);
  if (known > 0) return known;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || sms <= 0 ||
      per_sm <= 0) {
    cudaGetLastError();  // no sticky error from a failed query
    return 0;
  }
  cache[dev].store(sms * per_sm, std::memory_order_relaxed);
  return sms * per_sm;
}

// Grid of a grid-stride kernel: the blocks the work needs, at most one full
// wave of resident blocks (all of them when the query fails).
template <typename Kernel>
inline int grid_blocks(int64_t needed, Kernel kernel, int threads, size_t smem, std::atomic<int> (&cache)[kMaxHostDevices]) {
  const int64_t wave = resident_blocks(kernel, threads, smem, cache);
  int64_t b = needed < 1 ? 1 : needed;
  if (wave > 0 && b > wave) b = wave;
  return static_cast<int>(b < 0x7fffffff ? b : 0x7fffffff);
}

}  // namespace nvmla
