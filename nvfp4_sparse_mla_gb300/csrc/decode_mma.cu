// Sparse MLA decode, warp-level tensor-core kernel (mma.sync m16n8k16) with
// split-key partials and a separate merge kernel.
//
// What it computes: "Prime Inference: Fast, Reliable Serving for Frontier
// Open Models", section "A native NVFP4 sparse-MLA decode kernel" -- for each
// query token, only the rows the indexer selected are loaded, unpacked on
// chip and attended to with FP16 operands and FP32 accumulation; "Prime
// Intellect unveils Prime Inference", section "4-bit caches open the way",
// item 3 -- empty slots of the 2048-slot list contribute nothing.
//
// This is the general kernel: any head count that is a multiple of 16, both
// row formats (352-byte NVFP4 rows from the paged cache, or 576-byte FP8
// rows of the staged baseline). The tcgen05 kernel supersedes it where the
// head count makes the contraction a real dense one.
//
// Work split: grid (splits, T, head blocks of 64). A CTA owns one token, up
// to 64 heads and a contiguous range of the token's slots, processed in
// tiles of 64 rows:
//   1. cp.async gathers the tile's raw rows (16-byte pieces) into a double
//      buffer while the previous tile is computed;
//   2. all threads unpack the raw rows into an fp16 K tile [64][576] in
//      shared memory (E2M1 x E4M3 products are exact in fp16);
//   3. warp w takes 16 heads (w % 4) and half of the 512 value columns
//      (w / 4): S = Q K^T (36 k-steps), online softmax in fp32 with the
//      masked slots at -inf, O += P V with P rounded to fp16.
// Each CTA writes (O, m, l) for its slot range; the merge kernel combines
// the ranges (or, with one split, the CTA writes out/lse directly).
#include "common.cuh"

namespace nvmla {

constexpr int kKT = 64;            // rows per tile
constexpr int kQPad = 584;         // halves per smem row: 576 + 8 (bank spread)
constexpr int kRowB = kQPad * 2;   // 1168 bytes
constexpr int kMmaThreads = 256;

enum RowFormat { kNvfp4Paged = 0, kFp8Rows = 1 };

struct MmaParams {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;  // NVFP4 paged cache or FP8 rows
  RowSelect sel;         // NVFP4: index -> slot
  const int32_t* row_idx;  // FP8 rows: [T][topk]
  int T, H, topk;
  float sl2;  // sm_scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;   // [T][S][H][512]
  float* ws_ml;  // [T][S][H][2]
  int num_splits;
  int tiles_total;
  int32_t* err_word;
};

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int FMT>
struct Fmt;
template <>
struct Fmt<kNvfp4Paged> {
  static constexpr int kRaw = kRowBytes;
  static constexpr int kChunks = kRowBytes / 16;  // 22
};
template <>
struct Fmt<kFp8Rows> {
  static constexpr int kRaw = kFp8RowBytes;
  static constexpr int kChunks = kFp8RowBytes / 16;  // 36
};

template <int FMT>
__device__ __forceinline__ void unpack_tile(const uint8_t* raw, const int32_t* rows, __half* Ks, int nvalid_rows) {
  if constexpr (FMT == kNvfp4Paged) {
    // item = (row, part): parts 0..31 latent groups, 32..39 RoPE octets
    for (int i = threadIdx.x; i < kKT * 40; i += kMmaThreads) {
      const int r = i / 40, part = i % 40;
      uint4* dst;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      const uint8_t* src = raw + r * kRowBytes;
      const bool valid = r < nvalid_rows && rows[r] >= 0;
      if (part < 32) {
        dst = reinterpret_cast<uint4*>(Ks + r * kQPad + part * 16);
        if (valid) {
          const uint2 c = *reinterpret_cast<const uint2*>(src + part * 8);
          const uint32_t s2 = e4m3_to_f16x2_bcast(src[kScaleOff + part]);
          uint32_t h[4];
          e2m1x8_to_f16x8(c.x, h);
          v0 = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
          e2m1x8_to_f16x8(c.y, h);
          v1 = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
        }
        dst[0] = v0;
        dst[1] = v1;
      } else {
        const int q = part - 32;
        dst = reinterpret_cast<uint4*>(Ks + r * kQPad + kLatent + q * 8);
        if (valid) {
          const uint2 c = *reinterpret_cast<const uint2*>(src + kRopeOff + q * 8);
          e4m3x4_to_f16x4(c.x, v0.x, v0.y);
          e4m3x4_to_f16x4(c.y, v0.z, v0.w);
        }
        dst[0] = v0;
      }
    }
  } else {
    // item = (row, octet): 72 octets of E4M3 bytes per 576-byte row
    for (int i = threadIdx.x; i < kKT * 72; i += kMmaThreads) {
      const int r = i / 72, q = i % 72;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < nvalid_rows && rows[r] >= 0) {
        const uint2 c = *reinterpret_cast<const uint2*>(raw + r * kFp8RowBytes + q * 8);
        e4m3x4_to_f16x4(c.x, v.x, v.y);
        e4m3x4_to_f16x4(c.y, v.z, v.w);
      }
      *reinterpret_cast<uint4*>(Ks + r * kQPad + q * 8) = v;
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kMmaThreads, 1) decode_mma_kernel(MmaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kRaw = Fmt<FMT>::kRaw;
  constexpr int kChunks = Fmt<FMT>::kChunks;
  __half* Qs = reinterpret_cast<__half*>(smem);
  __half* Ks = reinterpret_cast<__half*>(smem + 64 * kRowB);
  uint8_t* raw = smem + 2 * 64 * kRowB;
  int32_t* rows = reinterpret_cast<int32_t*>(raw + 2 * kKT * kRaw);  // [keys of this CTA]

  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * 64;
  const int HB = min(64, p.H - h0);
  const int HG = HB / 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int tile_lo = (split * p.tiles_total) / p.num_splits;
  const int tile_hi = ((split + 1) * p.tiles_total) / p.num_splits;
  const int kbeg = tile_lo * kKT;
  const int kend = min(tile_hi * kKT, p.topk);
  const int nkeys = max(0, kend - kbeg);
  const int ntiles = (nkeys + kKT - 1) / kKT;

  // ---- rows of this CTA's slots (-1 = masked)
  for (int i = tid; i < nkeys; i += kMmaThreads) {
    int32_t r;
    if constexpr (FMT == kNvfp4Paged) {
      r = static_cast<int32_t>(p.sel.slot(t, kbeg + i, p.err_word, blockIdx.z == 0));
    } else {
      const int32_t idx = __ldg(p.row_idx + static_cast<int64_t>(t) * p.topk + kbeg + i);
      r = (idx >= 0 && idx < p.topk) ? t * p.topk + idx : -1;
      if (idx < -1 || idx >= p.topk) {
        if (blockIdx.z == 0) report_error(p.err_word, NVMLA_ERRW_BAD_INDEX, 1);
      }
    }
    rows[i] = r;
  }
  // ---- Q block -> fp16 smem
  for (int i = tid; i < HB * 72; i += kMmaThreads) {
    const int h = i / 72, c = i % 72;
    const int64_t qh = static_cast<int64_t>(t) * p.H + h0 + h;
    const uint4 v = c < 64 ? __ldg(reinterpret_cast<const uint4*>(p.q_latent + qh * kLatent) + c)
                           : __ldg(reinterpret_cast<const uint4*>(p.q_rope + qh * kRope) + (c - 64));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(bf16_bits_to_f32(w[j] & 0xffffu), bf16_bits_to_f32(w[j] >> 16));
    *reinterpret_cast<uint4*>(Qs + h * kQPad + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();

  auto issue = [&](int j) {
    uint8_t* dst = raw + (j & 1) * kKT * kRaw;
    const int base = j * kKT;
    const int n = min(kKT, nkeys - base);
    for (int c = tid; c < n * kChunks; c += kMmaThreads) {
      const int r = c / kChunks, q = c % kChunks;
      const int32_t row = rows[base + r];
      if (row >= 0) {
        const int64_t off = FMT == kNvfp4Paged ? cache_row_offset(row, p.sel.page_rows)
                                               : static_cast<int64_t>(row) * kRaw;
        cp_async_16(dst + r * kRaw + q * 16, p.cache + off + q * 16);
      }
    }
  };

  const int g = lane >> 2, t4 = lane & 3;
  const int hg = warp % 4, dvh = warp / 4;
  const bool active = hg < HG;
  float o[32][4];
#pragma unroll
  for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (ntiles > 0) issue(0);
  cp_async_commit();
  for (int j = 0; j < ntiles; ++j) {
    if (j + 1 < ntiles) issue(j + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int base = j * kKT;
    const int nrows = min(kKT, nkeys - base);
    unpack_tile<FMT>(raw + (j & 1) * kKT * kRaw, rows + base, Ks, nrows);
    __syncthreads();

    if (active) {
      // ---- S = Q K^T for 16 heads x 64 rows
      float s[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      const uint32_t qa = smem_u32(Qs + (hg * 16 + (lane & 15)) * kQPad + (lane >> 4) * 8);
      const uint32_t kb = smem_u32(Ks + ((lane >> 4) * 8 + (lane & 7)) * kQPad + ((lane >> 3) & 1) * 8);
#pragma unroll 4
      for (int kk = 0; kk < kDqk / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, qa + kk * 32);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, kb + np * 16 * kRowB + kk * 32);
          mma16816(s[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- mask + online softmax (log2 domain)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = 8 * n + 2 * t4 + e;
          const bool ok = key < nrows && rows[base + key] >= 0;
          s[n][e] = ok ? s[n][e] * p.sl2 : -INFINITY;
          s[n][e + 2] = ok ? s[n][e + 2] * p.sl2 : -INFINITY;
          mx0 = fmaxf(mx0, s[n][e]);
          mx1 = fmaxf(mx1, s[n][e + 2]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
      const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[n][e] = (mn0 == -INFINITY) ? 0.f : exp2f(s[n][e] - mn0);
          s[n][e + 2] = (mn1 == -INFINITY) ? 0.f : exp2f(s[n][e + 2] - mn1);
          rs0 += s[n][e];
          rs1 += s[n][e + 2];
        }
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      // ---- O += P V over this warp's 256 value columns
      const uint32_t vb = smem_u32(Ks + ((lane & 7) + ((lane >> 3) & 1) * 8) * kQPad + dvh * 256 + (lane >> 4) * 8);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t a0 = pack_f16x2(s[2 * ks][0], s[2 * ks][1]);
        const uint32_t a1 = pack_f16x2(s[2 * ks][2], s[2 * ks][3]);
        const uint32_t a2 = pack_f16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
        const uint32_t a3 = pack_f16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, vb + ks * 16 * kRowB + np * 32);
          mma16816(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  if (!active) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int hA = h0 + hg * 16 + g, hB = hA + 8;
  const int64_t rowA = static_cast<int64_t>(t) * p.H + hA, rowB = static_cast<int64_t>(t) * p.H + hB;
  if (p.num_splits == 1) {
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      const int dv = dvh * 256 + 8 * n + 2 * t4;
      *reinterpret_cast<__nv_bfloat162*>(p.out + rowA * kLatent + dv) = __floats2bfloat162_rn(o[n][0] * i0, o[n][1] * i0);
      *reinterpret_cast<__nv_bfloat162*>(p.out + rowB * kLatent + dv) = __floats2bfloat162_rn(o[n][2] * i1, o[n][3] * i1);
    }
    if (dvh == 0 && t4 == 0) {
      p.lse[rowA] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      p.lse[rowB] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
  } else {
    const int64_t pa = (static_cast<int64_t>(t) * p.num_splits + split) * p.H + hA;
    const int64_t pb = pa + 8;
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      const int dv = dvh * 256 + 8 * n + 2 * t4;
      *reinterpret_cast<float2*>(p.ws_o + pa * kLatent + dv) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(p.ws_o + pb * kLatent + dv) = make_float2(o[n][2], o[n][3]);
    }
    if (dvh == 0 && t4 == 0) {
      *reinterpret_cast<float2*>(p.ws_ml + pa * 2) = make_float2(m0, l0);
      *reinterpret_cast<float2*>(p.ws_ml + pb * 2) = make_float2(m1, l1);
    }
  }
}

// Merge split partials (O_i, m_i, l_i), m in log2 units:
//   M = max m_i, L = sum l_i 2^(m_i - M), out = sum O_i 2^(m_i - M) / L,
//   lse = (M + log2 L) ln 2.
__global__ void __launch_bounds__(128) merge_splits_kernel(const float* __restrict__ ws_o,
                                                           const float* __restrict__ ws_ml, int S, int H,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int th = blockIdx.x;  // t * H + h
  const int t = th / H, h = th % H;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ws_ml[((static_cast<int64_t>(t) * S + s) * H + h) * 2]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const int64_t ps = (static_cast<int64_t>(t) * S + s) * H + h;
      const float2 ml = *reinterpret_cast<const float2*>(ws_ml + ps * 2);
      if (ml.x == -INFINITY) continue;
      const float w = exp2f(ml.x - M);
      L += ml.y * w;
      const float4 v = reinterpret_cast<const float4*>(ws_o + ps * kLatent)[threadIdx.x];
      acc.x += v.x * w;
      acc.y += v.y * w;
      acc.z += v.z * w;
      acc.w += v.w * w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out + static_cast<int64_t>(th) * kLatent) + 2 * threadIdx.x;
  o2[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  o2[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  if (threadIdx.x == 0) lse[th] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

cudaError_t launch_merge(const float* ws_o, const float* ws_ml, int T, int S, int H, __nv_bfloat16* out, float* lse,
                         cudaStream_t stream) {
  merge_splits_kernel<<<T * H, 128, 0, stream>>>(ws_o, ws_ml, S, H, out, lse);
  return cudaGetLastError();
}

size_t mma_smem_bytes(int fmt, int topk_per_cta) {
  const int raw = fmt == kNvfp4Paged ? kRowBytes : kFp8RowBytes;
  return static_cast<size_t>(2 * 64 * kRowB) + 2 * kKT * raw + sizeof(int32_t) * ((topk_per_cta + 63) / 64 * 64);
}

int mma_default_splits(int T, int H, int topk, int num_sms) {
  const int hblocks = (H + 63) / 64;
  const int tiles = (topk + kKT - 1) / kKT;
  int s = num_sms / max(1, T * hblocks);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  return s;
}

size_t mma_workspace_bytes(int T, int H, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(T) * splits * H * (kLatent + 2) * sizeof(float);
}

cudaError_t launch_decode_mma(int fmt, const void* q_latent, const void* q_rope, const uint8_t* rows_src,
                              const RowSelect& sel, const int32_t* row_idx, int T, int H, int topk,
                              float sm_scale, void* out, float* lse, void* workspace, int splits,
                              int32_t* err_word, cudaStream_t stream) {
  MmaParams p;
  p.q_latent = static_cast<const __nv_bfloat16*>(q_latent);
  p.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
  p.cache = rows_src;
  p.sel = sel;
  p.row_idx = row_idx;
  p.T = T;
  p.H = H;
  p.topk = topk;
  p.sl2 = sm_scale * kLog2e;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.num_splits = splits;
  p.tiles_total = (topk + kKT - 1) / kKT;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = splits > 1 ? p.ws_o + static_cast<size_t>(T) * splits * H * kLatent : nullptr;
  p.err_word = err_word;
  const int max_tiles = (p.tiles_total + splits - 1) / splits;
  const size_t smem = mma_smem_bytes(fmt, max_tiles * kKT);
  dim3 grid(splits, T, (H + 63) / 64);
  cudaError_t e;
  if (fmt == kNvfp4Paged) {
    e = cudaFuncSetAttribute(decode_mma_kernel<kNvfp4Paged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_mma_kernel<kNvfp4Paged><<<grid, kMmaThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(decode_mma_kernel<kFp8Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_mma_kernel<kFp8Rows><<<grid, kMmaThreads, smem, stream>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  return launch_merge(p.ws_o, p.ws_ml, T, splits, H, p.out, lse, stream);
}

}  // namespace nvmla
