// nvmla_topk_select: the step upstream of the decode -- each query token's
// top-k positions by score, written as the fixed-length, -1 padded list the
// decode consumes ("Prime Intellect unveils Prime Inference", section "4-bit
// caches open the way", item 3: 2048-slot lists with the empty slots padded;
// "Prime Inference: Fast, Reliable Serving for Frontier Open Models", section
// "A native NVFP4 sparse-MLA decode kernel": the decode consumes the
// positions the sparse indexer selected). The indexer's scores come from
// trained weights the pages do not give, so the scores are an input here and
// only the selection is computed.
//
// Selection rule: the k = min(topk, length) largest scores, equal scores
// ranked by lower position; the chosen positions are written in increasing
// order, followed by -1 up to topk. -0.0 ranks as +0.0.
//
// One CTA per token: an exact radix select of the k-th largest key over the
// order-preserving 32-bit image of the scores (11 + 11 + 10 bits; the first
// pass over the whole row, the other two over the keys of the chosen bin,
// which are gathered into shared memory), then one ordered pass that writes
// every position above the threshold and the first `need` positions equal to
// it, using block-wide prefix counts.
#include "common.cuh"

namespace nvmla {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

// order-preserving image of a float: a > b (as reals) iff key(a) > key(b)
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;  // -0 ranks as +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inclusive prefix sum of v over the block's threads, in thread order; also
// returns the block total. Every thread of the block calls it.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kTopkWarps ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kTopkWarps) warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_tot[warp - 1] : 0u;
  total = warp_tot[kTopkWarps - 1];
  __syncthreads();  // warp_tot may be reused right after
  return before + x;
}

constexpr int kCand = 8192;  // candidates kept in shared memory after the first pass

// The histogram step of one radix pass over keys, and the choice of the bin
// that holds the rank-`need` key from the top (every thread calls it).
__device__ __forceinline__ void pick_bin(uint32_t* hist, int nb, uint32_t* warp_tot, uint32_t* found, uint32_t need) {
  // bins from the top: thread i holds bins nb-1-2i and nb-2-2i (nb <= 2048)
  const int tid = threadIdx.x;
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
  const uint32_t h0 = b0 >= 0 ? hist[b0] : 0u, h1 = b1 >= 0 ? hist[b1] : 0u;
  uint32_t total;
  const uint32_t incl = block_incl_scan(h0 + h1, warp_tot, total);
  const uint32_t above0 = incl - h0 - h1, above1 = above0 + h0;
  if (b0 >= 0 && need > above0 && need <= above0 + h0) {
    found[0] = static_cast<uint32_t>(b0);
    found[1] = above0;
    found[2] = h0;
  }
  if (b1 >= 0 && need > above1 && need <= above1 + h1) {
    found[0] = static_cast<uint32_t>(b1);
    found[1] = above1;
    found[2] = h1;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_select_kernel(const float* __restrict__ scores, int64_t stride,
                                                                   int32_t ncols, const int32_t* __restrict__ lengths,
                                                                   int32_t topk, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint32_t cand[];  // kCand keys, kCand positions, 4 x 2048 first-pass counts
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_tot[kTopkWarps];
  __shared__ uint32_t found[3];  // bin, count above it, count in it
  __shared__ uint32_t ncand;
  const int t = blockIdx.x, tid = threadIdx.x;
  const float* s = scores + static_cast<int64_t>(t) * stride;
  int32_t* o = out + static_cast<int64_t>(t) * topk;
  int L = lengths ? __ldg(lengths + t) : ncols;
  L = min(max(L, 0), ncols);
  const int k = min(topk, L);

  if (k == L) {
    // every position is chosen
    for (int i = tid; i < topk; i += kTopkThreads) o[i] = i < L ? i : -1;
    return;
  }
  // rows that start on a 16-byte boundary are read 4 scores at a time
  const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
  const int L4 = vec ? L / 4 : 0;
  const float4* s4 = reinterpret_cast<const float4*>(s);
  // apply f(valid, key, position) to every candidate of the row; the loops
  // run the same number of rounds in every lane of a warp (f may use warp
  // collectives), lanes past the end passing valid = false
  constexpr int kU = 4;  // 16-byte loads in flight per thread
  auto for_all = [&](auto&& f) {
    for (int b = 0; b < L4; b += kU * kTopkThreads) {
      float4 v[kU];
#pragma unroll
      for (int r = 0; r < kU; ++r) {
        const int i = b + r * kTopkThreads + tid;
        v[r] = i < L4 ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int r = 0; r < kU; ++r) {
        const int i = b + r * kTopkThreads + tid;
        const bool ok = i < L4;
        f(ok, score_key(v[r].x), 4 * i);
        f(ok, score_key(v[r].y), 4 * i + 1);
        f(ok, score_key(v[r].z), 4 * i + 2);
        f(ok, score_key(v[r].w), 4 * i + 3);
      }
    }
    for (int b = 4 * L4; b < L; b += kTopkThreads) {
      const int i = b + tid;
      const bool ok = i < L;
      f(ok, ok ? score_key(__ldg(s + i)) : 0u, i);
    }
  };
  auto hist_add = [&](bool ok, uint32_t bin) {
    if (ok) atomicAdd(&hist[bin], 1u);
  };

  // ---- radix select of the k-th largest key: bits 31-21 over the row,
  // then bits 20-10 and 9-0 over the keys of the chosen bin (from shared
  // memory when they fit, else over the row again)
  uint32_t need = static_cast<uint32_t>(k);  // rank wanted within the current prefix
  // (four copies of the first histogram, a quarter of the warps each: the
  // scores of a row crowd into few of its bins)
  uint32_t* hist4 = cand + 2 * kCand;
  for (int b = tid; b < 4 * 2048; b += kTopkThreads) hist4[b] = 0u;
  if (tid == 0) ncand = 0u;
  __syncthreads();
  uint32_t* mine = hist4 + 2048 * ((tid >> 5) & 3);
  for_all([&](bool ok, uint32_t u, int) {
    if (ok) atomicAdd(&mine[u >> 21], 1u);
  });
  __syncthreads();
  for (int b = tid; b < 2048; b += kTopkThreads) hist[b] = hist4[b] + hist4[2048 + b] + hist4[4096 + b] + hist4[6144 + b];
  __syncthreads();
  pick_bin(hist, 2048, warp_tot, found, need);
  uint32_t prefix = found[0] << 21, mask = 0xffe00000u;
  need -= found[1];
  const bool in_smem = found[2] <= static_cast<uint32_t>(kCand);
  __syncthreads();
  if (in_smem) {
    for_all([&](bool ok, uint32_t u, int i) {
      const bool in = ok && (u & mask) == prefix;
      const uint32_t bal = __ballot_sync(0xffffffffu, in);
      if (bal == 0u) return;
      const int lane = tid & 31, leader = __ffs(bal) - 1;
      uint32_t base = 0u;
      if (lane == leader) base = atomicAdd(&ncand, static_cast<uint32_t>(__popc(bal)));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (in) {
        const uint32_t c = base + __popc(bal & ((1u << lane) - 1u));
        cand[c] = u;
        cand[kCand + c] = static_cast<uint32_t>(i);
      }
    });
    __syncthreads();
  }
  const int nc = static_cast<int>(ncand);
#pragma unroll 1
  for (int pass = 1; pass < 3; ++pass) {
    const int sh = pass == 1 ? 10 : 0, nb = pass == 1 ? 2048 : 1024;
    for (int b = tid; b < nb; b += kTopkThreads) hist[b] = 0u;
    __syncthreads();
    auto count = [&](bool ok, uint32_t u, int) { hist_add(ok && (u & mask) == prefix, (u >> sh) & (nb - 1)); };
    if (in_smem) {
      for (int b = 0; b < nc; b += kTopkThreads) {
        const int c = b + tid;
        count(c < nc, c < nc ? cand[c] : 0u, 0);
      }
    } else {
      for_all(count);
    }
    __syncthreads();
    pick_bin(hist, nb, warp_tot, found, need);
    prefix |= found[0] << sh;
    mask |= static_cast<uint32_t>(nb - 1) << sh;
    need -= found[1];
    __syncthreads();
  }
  // prefix is the k-th largest key; `need` (>= 1) positions equal to it are
  // taken, the lowest first

  // ---- ordered collection: 16 consecutive positions per thread per round
  constexpr int kPer = 16;
  uint32_t base_gt = 0u, base_eq = 0u;
#pragma unroll 1
  for (int start = 0; start < L; start += kPer * kTopkThreads) {
    const int p0 = start + kPer * tid;
    uint32_t key[kPer];
    if (vec && p0 + kPer - 1 < L) {
#pragma unroll
      for (int q = 0; q < kPer / 4; ++q) {
        const float4 v = __ldg(s4 + (p0 >> 2) + q);
        key[4 * q] = score_key(v.x);
        key[4 * q + 1] = score_key(v.y);
        key[4 * q + 2] = score_key(v.z);
        key[4 * q + 3] = score_key(v.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) key[j] = p0 + j < L ? score_key(__ldg(s + p0 + j)) : 0u;
    }
    uint32_t gt = 0u, eq = 0u;  // bit j: position p0 + j
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (p0 + j < L) {
        gt |= (key[j] > prefix ? 1u : 0u) << j;
        eq |= (key[j] == prefix ? 1u : 0u) << j;
      }
    }
    const uint32_t c = __popc(gt) | (__popc(eq) << 16);
    uint32_t total;
    const uint32_t excl = block_incl_scan(c, warp_tot, total) - c;
    uint32_t g = base_gt + (excl & 0xffffu), e = base_eq + (excl >> 16);
    uint32_t sel = gt | eq;
    while (sel) {
      const int j = __ffs(sel) - 1;
      sel &= sel - 1u;
      const uint32_t below = (1u << j) - 1u;
      const uint32_t gj = g + __popc(gt & below), ej = e + __popc(eq & below);
      if (((gt >> j) & 1u) || ej < need) o[gj + min(ej, need)] = p0 + j;
    }
    base_gt += total & 0xffffu;
    base_eq += total >> 16;
  }
  for (int i = k + tid; i < topk; i += kTopkThreads) o[i] = -1;
}

cudaError_t launch_topk_select(const float* scores, int64_t stride, int32_t ncols, const int32_t* lengths, int32_t T,
                               int32_t topk, int32_t* out, cudaStream_t stream) {
  constexpr int kDyn = (2 * kCand + 4 * 2048) * 4;
  static bool attr_set[64] = {false};  // the attribute is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  topk_select_kernel<<<T, kTopkThreads, kDyn, stream>>>(scores, stride, ncols, lengths, topk, out);
  return cudaGetLastError();
}

}  // namespace nvmla
