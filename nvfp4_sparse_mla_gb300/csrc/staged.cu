// Staged baseline, stage 1: unpack the selected NVFP4 rows into a temporary
// 576-byte FP8 buffer in GPU memory.
//
// "Prime Inference open-model serving" (mo.ai.kr), section "KV 캐시와 데이터
// 전송": before the native kernel, compressed data was unpacked into a
// temporary FP8 buffer ahead of an existing attention kernel, adding a
// conversion plus a GPU-memory write and read. "Prime Intellect unveils
// Prime Inference", section "4-bit caches open the way", says the same. The
// FP8 row is 512 latent + 64 RoPE E4M3 bytes ("Prime Inference: Fast,
// Reliable Serving for Frontier Open Models", section "Making room for
// low-latency decode").
//
// One warp per selected slot (t, k): lane l turns latent group l (8 code
// bytes + its scale) into 16 E4M3 bytes: E2M1 x E4M3 is exact in fp16, then
// one round-to-nearest-even saturating conversion to E4M3 (lossy: the product
// has up to 6 significant bits and reaches 2688). Lanes 0-3 copy the RoPE
// bytes. Rows of masked slots are not written; row_idx says which are valid.
#include "common.cuh"

namespace nvmla {

constexpr int kStageWarps = 8;

__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

__global__ void __launch_bounds__(kStageWarps * 32)
stage_dequant_kernel(const uint8_t* __restrict__ cache, RowSelect sel, int T, uint8_t* __restrict__ fp8_rows,
                     int32_t* __restrict__ row_idx, int32_t* err_word) {
  const int lane = threadIdx.x & 31;
  const int64_t total = static_cast<int64_t>(T) * sel.topk;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kStageWarps;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kStageWarps + (threadIdx.x >> 5); w < total; w += nwarps) {
    const int t = static_cast<int>(w / sel.topk), k = static_cast<int>(w % sel.topk);
    const int64_t slot = sel.slot(t, k, err_word, lane == 0);
    if (lane == 0) row_idx[w] = slot >= 0 ? k : -1;
    if (slot < 0) continue;
    const uint8_t* src = cache + cache_row_offset(slot, sel.page_rows);
    uint8_t* dst = fp8_rows + w * kFp8RowBytes;
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    const uint32_t s2 = e4m3_to_f16x2_bcast(__ldg(src + kScaleOff + lane));
    uint32_t h[4], q[4];
    e2m1x8_to_f16x8(c.x, h);
    q[0] = f16x2_to_e4m3x2(hmul2_u32(h[0], s2)) | (f16x2_to_e4m3x2(hmul2_u32(h[1], s2)) << 16);
    q[1] = f16x2_to_e4m3x2(hmul2_u32(h[2], s2)) | (f16x2_to_e4m3x2(hmul2_u32(h[3], s2)) << 16);
    e2m1x8_to_f16x8(c.y, h);
    q[2] = f16x2_to_e4m3x2(hmul2_u32(h[0], s2)) | (f16x2_to_e4m3x2(hmul2_u32(h[1], s2)) << 16);
    q[3] = f16x2_to_e4m3x2(hmul2_u32(h[2], s2)) | (f16x2_to_e4m3x2(hmul2_u32(h[3], s2)) << 16);
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
    if (lane < 4) {
      reinterpret_cast<uint4*>(dst + kLatent)[lane] = __ldg(reinterpret_cast<const uint4*>(src + kRopeOff) + lane);
    }
  }
}

cudaError_t launch_stage_dequant(const uint8_t* cache, const RowSelect& sel, int T, uint8_t* fp8_rows,
                                 int32_t* row_idx, int32_t* err_word, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(T) * sel.topk;
  static std::atomic<int> wave[kMaxHostDevices];
  const int blocks = grid_blocks((total + kStageWarps - 1) / kStageWarps, stage_dequant_kernel, kStageWarps * 32, 0, wave);
  stage_dequant_kernel<<<blocks, kStageWarps * 32, 0, stream>>>(cache, sel, T, fp8_rows, row_idx, err_word);
  return cudaGetLastError();
}

}  // namespace nvmla
