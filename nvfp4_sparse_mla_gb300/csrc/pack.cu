// nvfp4_mla_pack: quantise new tokens into 352-byte NVFP4 cache rows.
//
// "Prime Inference: Fast, Reliable Serving for Frontier Open Models",
// section "Making room for low-latency decode": the 512-value latent is
// stored as 4-bit values with one FP8 scale per 16 values, the 64-value RoPE
// part stays FP8, 352 bytes per row.
//
// One warp per token at a time, each warp taking every nwarps-th token and
// fetching its next token's values while it quantises the current one (the
// grid gives every warp at least two tokens, at most one wave). Lane l owns
// latent group l (16 values = 32 bytes of bf16, read as two 16-byte loads,
// so a warp reads the token's 1 KiB latent fully coalesced) and RoPE values
// 2l, 2l+1. The group's scale and codes are computed in registers without
// any shuffle, and each lane stores its own bytes of the 352-byte row: 8
// code bytes, 1 scale byte and 2 RoPE bytes (the warp's three stores cover
// 256, 32 and 64 contiguous bytes).
//
// Rounding, bit-exact with the definition:
//  * scale = E4M3(amax / 6): fp32 division correctly rounded (__fdiv_rn), then
//    the hardware's round-to-nearest-even saturating E4M3 conversion. amax is
//    a bf16 value (8 significant bits); amax/6 is either exact or has an
//    infinite binary expansion, so the fp32 rounding can never create or
//    break an E4M3 tie: the two roundings equal one.
//  * codes: |v| is compared with S times the E2M1 midpoints 0.25, 0.75, 1.25,
//    1.75, 2.5, 3.5, 5; at a midpoint the strict or non-strict comparison
//    sends the value to the even code. The comparisons run two values at a
//    time in bf16x2 on the input itself: each product has at most 7
//    significant bits and so is exact in bf16.
#include "common.cuh"

namespace nvmla {
// read-only loads issued where they stand (volatile: the compiler does not
// sink them to their first use)
__device__ __forceinline__ uint4 ldg_nc_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int32_t ldg_nc_s32i(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}


constexpr int kPackWarps = 8;

__global__ void __launch_bounds__(kPackWarps * 32)
nvfp4_pack_kernel(const __nv_bfloat16* __restrict__ latent, int64_t lat_stride,
                  const __nv_bfloat16* __restrict__ rope, int64_t rope_stride,
                  const int32_t* __restrict__ slot_mapping, int64_t n_tokens,
                  uint8_t* __restrict__ cache, int64_t num_slots, int32_t page_rows, int32_t* err_word) {
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kPackWarps;

  // a token's values are requested together with its slot (one memory
  // round trip, not two), and the warp's next token's before this one is
  // quantised; a token that is skipped leaves them unused
  struct In {
    uint4 a, b;
    uint32_t rw;
    int32_t slot;
  };
  auto fetch = [&](int64_t n) {
    In v;
    const uint4* src = reinterpret_cast<const uint4*>(latent + n * lat_stride + lane * 16);
    v.a = ldg_nc_u4(src);
    v.b = ldg_nc_u4(src + 1);
    v.rw = ldg_nc_u32(reinterpret_cast<const uint32_t*>(rope + n * rope_stride) + lane);
    v.slot = ldg_nc_s32i(slot_mapping + n);
    return v;
  };
  int64_t n = static_cast<int64_t>(blockIdx.x) * kPackWarps + wib;
  In cur;
  if (n < n_tokens) cur = fetch(n);
  for (; n < n_tokens; n += nwarps) {
    In nxt{};
    if (n + nwarps < n_tokens) nxt = fetch(n + nwarps);
    const uint4 a = cur.a, b = cur.b;
    const uint32_t rw = cur.rw;
    const int64_t slot = cur.slot;
    cur = nxt;
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) report_error(err_word, NVMLA_ERRW_PACK_SLOT, 1);
      continue;
    }
    // ---- latent group `lane`
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    // amax in bf16x2 (max ignores a NaN operand, as fmaxf does; an all-NaN
    // group gets 0)
    uint32_t mx = w[0] & 0x7fff7fffu;
#pragma unroll
    for (int i = 1; i < 8; ++i) asm("max.bf16x2 %0, %1, %2;" : "=r"(mx) : "r"(mx), "r"(w[i] & 0x7fff7fffu));
    const float amax = fmaxf(0.f, fmaxf(bf16_bits_to_f32(mx & 0xffffu), bf16_bits_to_f32(mx >> 16)));
    const float q = __fdiv_rn(amax, 6.0f);
    const uint32_t sbyte = f32x2_to_e4m3x2(q, 0.f) & 0xffu;
    const float S = __half2float(__ushort_as_half(static_cast<uint16_t>(e4m3x2_to_f16x2(static_cast<uint16_t>(sbyte)) & 0xffffu)));
    // codes two at a time in bf16x2, straight on the input. The thresholds
    // mid_k * S (mid = 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5: at most 3
    // significant bits; S: 4) are exact bf16 products. The code magnitude is
    // the count of thresholds below |v|, strictly for even k and non-strictly
    // for odd k, which sends a midpoint to the even code; the thresholds
    // increase with k, so the count is found by a binary search: |v| against
    // mid_3, then mid_1 or mid_5, then one of mid_0, 2, 4, 6, each compare
    // giving a per-half mask. A NaN compares false (code 0).
    const uint32_t s2 = (__float_as_uint(S) >> 16) * 0x10001u;
    uint32_t th[7];
    {
      constexpr uint32_t kMid2[7] = {0x3e803e80u, 0x3f403f40u, 0x3fa03fa0u, 0x3fe03fe0u,
                                     0x40204020u, 0x40604060u, 0x40a040a0u};
#pragma unroll
      for (int k = 0; k < 7; ++k) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(th[k]) : "r"(s2), "r"(kMid2[k]));
    }
    uint32_t codes[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wi = w[i];
      const uint32_t x2 = wi & 0x7fff7fffu;
      uint32_t b2, b1, b0;
      asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(b2) : "r"(x2), "r"(th[3]));
      const uint32_t t1 = (th[5] & b2) | (th[1] & ~b2);
      asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(b1) : "r"(x2), "r"(t1));
      const uint32_t ta = (th[6] & b1) | (th[4] & ~b1), tb = (th[2] & b1) | (th[0] & ~b1);
      const uint32_t t0 = (ta & b2) | (tb & ~b2);
      asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(b0) : "r"(x2), "r"(t0));
      uint32_t m2 = (b2 & 0x00040004u) | (b1 & 0x00020002u) | (b0 & 0x00010001u);
      m2 = (S == 0.f) ? 0u : m2;
      const uint32_t byte = (m2 & 0xfu) | ((m2 >> 12) & 0xf0u) | ((wi >> 12) & 0x8u) | ((wi >> 24) & 0x80u);
      codes[i >> 2] |= byte << (8 * (i & 3));
    }
    // ---- RoPE values 2*lane, 2*lane+1
    const uint16_t r8 = f32x2_to_e4m3x2(bf16_bits_to_f32(rw & 0xffffu), bf16_bits_to_f32(rw >> 16));
    // this lane's bytes straight to the row: its 8 code bytes, scale byte
    // and 2 RoPE bytes (the warp's stores cover 256, 32 and 64 contiguous
    // bytes)
    uint8_t* dst = cache + cache_row_offset(slot, page_rows);
    *reinterpret_cast<uint2*>(dst + 8 * lane) = make_uint2(codes[0], codes[1]);
    dst[kScaleOff + lane] = static_cast<uint8_t>(sbyte);
    *reinterpret_cast<uint16_t*>(dst + kRopeOff + 2 * lane) = r8;
  }
}

cudaError_t launch_pack(const void* latent, int64_t lat_stride, const void* rope, int64_t rope_stride,
                        const int32_t* slot_mapping, int64_t n_tokens, uint8_t* cache, int64_t num_pages,
                        int32_t page_rows, int32_t* err_word, cudaStream_t stream) {
  static std::atomic<int> wave[kMaxHostDevices];
  // at least two tokens a warp (the second is fetched during the first)
  const int blocks = grid_blocks((n_tokens + 2 * kPackWarps - 1) / (2 * kPackWarps), nvfp4_pack_kernel,
                                 kPackWarps * 32, 0, wave);
  nvfp4_pack_kernel<<<blocks, kPackWarps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(latent), lat_stride, static_cast<const __nv_bfloat16*>(rope),
      rope_stride, slot_mapping, n_tokens, cache, num_pages * kPage, page_rows, err_word);
  return cudaGetLastError();
}

// fp8_mla_pack: the FP8 cache the NVFP4 rows are compared with (576-byte
// rows: the 512 latent and 64 RoPE values each as one E4M3 byte, nearest
// even, saturating, no scale; "Prime Inference: Fast, Reliable Serving for
// Frontier Open Models", section "Making room for low-latency decode": 576
// bytes per token before the NVFP4 change). One warp per token: lane l owns
// latent values 16l .. 16l + 15 and RoPE values 2l, 2l + 1; the row is
// assembled in shared memory and written as 36 aligned 16-byte stores.
__global__ void __launch_bounds__(kPackWarps * 32)
fp8_pack_kernel(const __nv_bfloat16* __restrict__ latent, int64_t lat_stride, const __nv_bfloat16* __restrict__ rope,
                int64_t rope_stride, const int32_t* __restrict__ slot_mapping, int64_t n_tokens,
                uint8_t* __restrict__ cache, int64_t num_slots, int32_t* err_word) {
  __shared__ __align__(16) uint8_t rowbuf[kPackWarps][kFp8RowBytes];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  uint8_t* row = rowbuf[wib];
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kPackWarps;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * kPackWarps + wib; n < n_tokens; n += nwarps) {
    // values and slot in one round trip, as in nvfp4_pack_kernel
    const uint4* src = reinterpret_cast<const uint4*>(latent + n * lat_stride + lane * 16);
    const uint4 a = __ldg(src);
    const uint4 b = __ldg(src + 1);
    const uint32_t rw = __ldg(reinterpret_cast<const uint32_t*>(rope + n * rope_stride) + lane);
    const int64_t slot = __ldg(slot_mapping + n);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) report_error(err_word, NVMLA_ERRW_PACK_SLOT, 1);
      continue;
    }
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = f32x2_to_e4m3x2(bf16_bits_to_f32(w[2 * i] & 0xffffu), bf16_bits_to_f32(w[2 * i] >> 16));
      const uint32_t hi =
          f32x2_to_e4m3x2(bf16_bits_to_f32(w[2 * i + 1] & 0xffffu), bf16_bits_to_f32(w[2 * i + 1] >> 16));
      q[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(q[0], q[1], q[2], q[3]);
    *reinterpret_cast<uint16_t*>(row + kLatent + 2 * lane) =
        f32x2_to_e4m3x2(bf16_bits_to_f32(rw & 0xffffu), bf16_bits_to_f32(rw >> 16));
    __syncwarp();
    uint8_t* dst = cache + slot * kFp8RowBytes;
    for (int c = lane; c < kFp8RowBytes / 16; c += 32)
      reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(row)[c];
    __syncwarp();
  }
}

cudaError_t launch_fp8_pack(const void* latent, int64_t lat_stride, const void* rope, int64_t rope_stride,
                            const int32_t* slot_mapping, int64_t n_tokens, uint8_t* cache, int64_t num_pages,
                            int32_t* err_word, cudaStream_t stream) {
  static std::atomic<int> wave[kMaxHostDevices];
  const int blocks = grid_blocks((n_tokens + kPackWarps - 1) / kPackWarps, fp8_pack_kernel, kPackWarps * 32, 0, wave);
  fp8_pack_kernel<<<blocks, kPackWarps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(latent), lat_stride, static_cast<const __nv_bfloat16*>(rope), rope_stride,
      slot_mapping, n_tokens, cache, num_pages * kPage, err_word);
  return cudaGetLastError();
}

}  // namespace nvmla
