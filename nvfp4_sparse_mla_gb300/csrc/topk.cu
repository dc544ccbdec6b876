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
// One cluster of kTopkCtas CTAs per token, CTA r owning a contiguous chunk of
// the row. An exact radix select of the k-th largest key over the
// order-preserving 32-bit image of the scores (11 + 11 + 10 bits): every CTA
// histograms its chunk (the first pass) or its own keys of the chosen bin
// (kept in shared memory; the other two passes), and reads the other CTAs'
// histograms through distributed shared memory, so that every CTA picks the
// same bin. Each CTA then knows how many of its positions lie above the
// threshold and how many equal it, learns the counts of the CTAs before it,
// and writes its chosen positions at their place in the list.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace nvmla {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCtas = 8;  // CTAs per token (a portable cluster)
constexpr int kCand = 4096;   // keys of the chosen bin a CTA keeps in shared memory

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

struct TopkShared {
  uint32_t hist[2048];       // this CTA's counts of the current pass
  uint32_t cand_key[kCand];  // this CTA's keys of the chosen first-pass bin
  uint32_t cand_pos[kCand];
  uint32_t warp_tot[kTopkWarps];
  uint32_t found[2];  // chosen bin, cluster-wide count above it
  uint32_t ncand;     // keys of the chosen bin in this CTA
  uint32_t overflow;  // some CTA of the cluster has more than kCand of them
  uint32_t counts[2];  // this CTA's positions above / equal to the threshold
};

// The cluster-wide histogram (the sum of `hist` over the cluster's CTAs) and
// the bin that holds the rank-`need` key from the top, into sh.found. Every
// thread of every CTA of the cluster calls it, once the histograms are
// complete cluster-wide.
__device__ __forceinline__ void pick_bin_cluster(cg::cluster_group& cluster, TopkShared& sh, int nb, uint32_t need) {
  const int tid = threadIdx.x;
  // bins from the top: thread i holds bins nb-1-2i and nb-2-2i (nb <= 2048)
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
  uint32_t h0 = 0u, h1 = 0u;
  for (int r = 0; r < kTopkCtas; ++r) {
    const uint32_t* rh = cluster.map_shared_rank(sh.hist, r);
    if (b0 >= 0) h0 += rh[b0];
    if (b1 >= 0) h1 += rh[b1];
  }
  uint32_t total;
  const uint32_t incl = block_incl_scan(h0 + h1, sh.warp_tot, total);
  const uint32_t above0 = incl - h0 - h1, above1 = above0 + h0;
  if (b0 >= 0 && need > above0 && need <= above0 + h0) {
    sh.found[0] = static_cast<uint32_t>(b0);
    sh.found[1] = above0;
  }
  if (b1 >= 0 && need > above1 && need <= above1 + h1) {
    sh.found[0] = static_cast<uint32_t>(b1);
    sh.found[1] = above1;
  }
  __syncthreads();
}

__global__ void __cluster_dims__(kTopkCtas, 1, 1) __launch_bounds__(kTopkThreads, 1)
    topk_select_kernel(const float* __restrict__ scores, int64_t stride, int32_t ncols,
                       const int32_t* __restrict__ lengths, int32_t topk, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int t = blockIdx.y, tid = threadIdx.x;
  const float* s = scores + static_cast<int64_t>(t) * stride;
  int32_t* o = out + static_cast<int64_t>(t) * topk;
  int L = lengths ? __ldg(lengths + t) : ncols;
  L = min(max(L, 0), ncols);
  const int k = min(topk, L);

  if (k == L) {
    // every position is chosen (the same decision in every CTA of the token,
    // before any cluster barrier)
    if (rank == 0)
      for (int i = tid; i < topk; i += kTopkThreads) o[i] = i < L ? i : -1;
    return;
  }
  // this CTA's chunk: positions [lo, hi), split at multiples of 4
  const int quads = (L + 3) / 4;
  const int lo = 4 * ((rank * quads) / kTopkCtas), hi = min(L, 4 * (((rank + 1) * quads) / kTopkCtas));
  // rows that start on a 16-byte boundary are read 4 scores at a time
  const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
  // apply f(key, position) to every position of the chunk
  auto for_chunk = [&](auto&& f) {
    if (vec) {
      const float4* s4 = reinterpret_cast<const float4*>(s);
      const int q_hi = hi / 4;
      constexpr int kU = 4;  // 16-byte loads in flight per thread
      for (int q0 = lo / 4; q0 < q_hi; q0 += kU * kTopkThreads) {
        float4 v[kU];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < q_hi) v[r] = __ldg(s4 + q);
        }
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < q_hi) {
            f(score_key(v[r].x), 4 * q);
            f(score_key(v[r].y), 4 * q + 1);
            f(score_key(v[r].z), 4 * q + 2);
            f(score_key(v[r].w), 4 * q + 3);
          }
        }
      }
      for (int i = 4 * q_hi + tid; i < hi; i += kTopkThreads) f(score_key(__ldg(s + i)), i);
    } else {
      for (int i = lo + tid; i < hi; i += kTopkThreads) f(score_key(__ldg(s + i)), i);
    }
  };

  // ---- pass 1: key bits 31-21 over the chunk
  for (int b = tid; b < 2048; b += kTopkThreads) sh.hist[b] = 0u;
  if (tid == 0) {
    sh.ncand = 0u;
    sh.overflow = 0u;
  }
  __syncthreads();
  for_chunk([&](uint32_t u, int) { atomicAdd(&sh.hist[u >> 21], 1u); });
  cluster.sync();
  uint32_t need = static_cast<uint32_t>(k);  // rank wanted within the current prefix
  pick_bin_cluster(cluster, sh, 2048, need);
  const uint32_t bin1 = sh.found[0];
  uint32_t prefix = bin1 << 21, mask = 0xffe00000u;
  need -= sh.found[1];
  // the chunk's positions in bins above the chosen one are all chosen
  uint32_t n_above = 0u;
  for (int b = static_cast<int>(bin1) + 1 + tid; b < 2048; b += kTopkThreads) n_above += sh.hist[b];
  {
    uint32_t tot;
    block_incl_scan(n_above, sh.warp_tot, tot);
    n_above = tot;
  }
  if (tid == 0 && sh.hist[bin1] > static_cast<uint32_t>(kCand)) {
    for (int r = 0; r < kTopkCtas; ++r) atomicExch(cluster.map_shared_rank(&sh.overflow, r), 1u);
  }
  cluster.sync();  // every CTA is done with the first histograms; overflow is final
  const bool keep = sh.overflow == 0u;  // the same in every CTA of the cluster
  // the chunk's keys of the chosen bin, in shared memory
  if (keep) {
    for_chunk([&](uint32_t u, int i) {
      if ((u & mask) == prefix) {
        const uint32_t c = atomicAdd(&sh.ncand, 1u);
        sh.cand_key[c] = u;
        sh.cand_pos[c] = static_cast<uint32_t>(i);
      }
    });
  }
  __syncthreads();
  const int nc = static_cast<int>(sh.ncand);

  // ---- passes 2 and 3: bits 20-10, then 9-0, over the chosen bin's keys
#pragma unroll 1
  for (int pass = 1; pass < 3; ++pass) {
    const int sb = pass == 1 ? 10 : 0, nb = pass == 1 ? 2048 : 1024;
    for (int b = tid; b < nb; b += kTopkThreads) sh.hist[b] = 0u;
    __syncthreads();
    auto count = [&](uint32_t u, int) {
      if ((u & mask) == prefix) atomicAdd(&sh.hist[(u >> sb) & (nb - 1)], 1u);
    };
    if (keep) {
      for (int c = tid; c < nc; c += kTopkThreads) count(sh.cand_key[c], 0);
    } else {
      for_chunk(count);
    }
    cluster.sync();
    pick_bin_cluster(cluster, sh, nb, need);
    prefix |= sh.found[0] << sb;
    mask |= static_cast<uint32_t>(nb - 1) << sb;
    need -= sh.found[1];
    cluster.sync();  // every CTA is done reading the others' histograms
  }
  // prefix is the k-th largest key; `need` (>= 1) positions equal to it are
  // taken, the lowest first

  // ---- this CTA's positions above / equal to the threshold, then the
  // counts of the CTAs before it
  uint32_t n_gt = 0u, n_eq = 0u;
  if (keep) {
    for (int c = tid; c < nc; c += kTopkThreads) {
      n_gt += sh.cand_key[c] > prefix ? 1u : 0u;
      n_eq += sh.cand_key[c] == prefix ? 1u : 0u;
    }
  } else {
    for_chunk([&](uint32_t u, int) {
      n_gt += u > prefix ? 1u : 0u;
      n_eq += u == prefix ? 1u : 0u;
    });
  }
  {
    uint32_t tg, te;
    block_incl_scan(n_gt, sh.warp_tot, tg);
    block_incl_scan(n_eq, sh.warp_tot, te);
    // (with the chosen bin's keys kept, the bins above it hold the rest of
    // the chunk's keys above the threshold)
    if (tid == 0) {
      sh.counts[0] = tg + (keep ? n_above : 0u);
      sh.counts[1] = te;
    }
  }
  cluster.sync();
  uint32_t base_gt = 0u, base_eq = 0u;
  for (int r = 0; r < rank; ++r) {
    const uint32_t* rc = cluster.map_shared_rank(sh.counts, r);
    base_gt += rc[0];
    base_eq += rc[1];
  }
  cluster.sync();  // no CTA leaves while another reads its counts

  // ---- ordered collection over the chunk: 16 consecutive positions per
  // thread per round
  constexpr int kPer = 16;
#pragma unroll 1
  for (int start = lo; start < hi; start += kPer * kTopkThreads) {
    const int p0 = start + kPer * tid;
    uint32_t key[kPer];
    if (vec && p0 + kPer <= hi) {
#pragma unroll
      for (int q = 0; q < kPer / 4; ++q) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(s + p0) + q);
        key[4 * q] = score_key(v.x);
        key[4 * q + 1] = score_key(v.y);
        key[4 * q + 2] = score_key(v.z);
        key[4 * q + 3] = score_key(v.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) key[j] = p0 + j < hi ? score_key(__ldg(s + p0 + j)) : 0u;
    }
    uint32_t gt = 0u, eq = 0u;  // bit j: position p0 + j
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (p0 + j < hi) {
        gt |= (key[j] > prefix ? 1u : 0u) << j;
        eq |= (key[j] == prefix ? 1u : 0u) << j;
      }
    }
    const uint32_t c = __popc(gt) | (__popc(eq) << 16);
    uint32_t total;
    const uint32_t excl = block_incl_scan(c, sh.warp_tot, total) - c;
    const uint32_t g = base_gt + (excl & 0xffffu), e = base_eq + (excl >> 16);
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
  if (rank == kTopkCtas - 1)
    for (int i = k + tid; i < topk; i += kTopkThreads) o[i] = -1;
}

cudaError_t launch_topk_select(const float* scores, int64_t stride, int32_t ncols, const int32_t* lengths, int32_t T,
                               int32_t topk, int32_t* out, cudaStream_t stream) {
  constexpr int kDyn = static_cast<int>(sizeof(TopkShared));
  static bool attr_set[64] = {false};  // the attribute is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  topk_select_kernel<<<dim3(kTopkCtas, T), kTopkThreads, kDyn, stream>>>(scores, stride, ncols, lengths, topk, out);
  return cudaGetLastError();
}

}  // namespace nvmla
