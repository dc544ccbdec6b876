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
// the row; the k-th largest key is found exactly, over the order-preserving
// 32-bit image of the scores. Rows whose chunks fit in shared memory (up to
// 8 x kResKeys positions, the decode's 200K rows among them) take
// topk_resident_kernel, described at its definition below: one exchange of
// the candidates above a bound every CTA can certify. Longer rows take
// topk_select_kernel, a radix select whose chunk walks read global memory
// where the chunk does not fit:
//  * first pass, bits 31-21: each CTA histograms its chunk (keeping the keys
//    in shared memory where they fit) and adds its non-zero bins into rank
//    0's cluster histogram (remote shared-memory atomics); rank 0 picks the
//    bin holding the k-th largest key and writes it into every CTA;
//  * each thread lists the chunk offsets of its keys at or above that bin
//    (every position that can still be chosen; the chunk is walked again
//    where a list would overflow);
//  * the keys of the bin, cluster-wide, usually a few thousand: every CTA
//    copies its own into a pool in rank 0, which finishes the select on them
//    alone (bits 20-10, then 9-0) and sends each CTA the threshold and the
//    counts of chosen positions in the chunks before its own; with more of
//    them than the pool holds, the last two passes run cluster-wide like the
//    first and the CTAs exchange their counts;
//  * each CTA marks its chosen positions in bitmaps of its chunk and writes
//    them in order at their place in the list (or walks the chunk again in
//    order where it does not fit in shared memory).
#include <cooperative_groups.h>

#include <cstddef>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace nvmla {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCtas = 8;  // CTAs per token (a portable cluster)

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

constexpr int kChunkKeys = 32 * 1024;     // a chunk of up to this many keys stays in shared memory
constexpr int kPool = 8 * 1024;           // keys of the first pass's bin rank 0 collects from the cluster
constexpr int kList = 8;                  // chunk offsets a thread lists after the first pass
constexpr int kBmWords = kChunkKeys / 32;  // words of a bitmap of the chunk
static_assert(kBmWords == kTopkThreads, "one bitmap word per thread");

struct TopkShared {
  uint32_t hist[2048];     // this CTA's counts of the current pass
  uint32_t cl_hist[2048];  // rank 0: the cluster's counts of the current pass
  uint32_t bm_gt[kBmWords];  // chosen positions above / equal to the threshold, by chunk offset
  uint32_t bm_eq[kBmWords];
  uint32_t warp_tot[kTopkWarps];
  uint32_t part[kTopkWarps][2 * kTopkCtas];  // rank 0: per warp, pool keys above / equal by source rank
  uint32_t found[3];  // written by rank 0: chosen bin, cluster-wide count above it, count in it
  // written by rank 0 (pool path): threshold key, equal keys taken, and the
  // chosen positions above / equal to it in the chunks before this one
  uint32_t res[4];
  uint32_t lower[kTopkCtas][2];  // counts above / equal written by each lower rank (cluster-wide path)
  uint32_t seg[kTopkCtas][3];    // rank 0: each rank's pool start and length, and its count above the bin
  // per thread (column), the chunk offsets of its keys at or above the first
  // pass's bin
  uint32_t list[kList][kTopkThreads];
  uint32_t few[32];              // rank 0: the last few keys of the select
  uint32_t nfew;
  uint32_t pool_n;               // rank 0: pool slots handed out
  uint32_t slot;                 // this CTA's pool slots used
  uint32_t base;                 // this CTA's pool start
  alignas(16) uint32_t pool[kPool];
  alignas(16) uint32_t keys[kChunkKeys];  // the chunk's keys, when they fit
};
static_assert(offsetof(TopkShared, keys) % 16 == 0, "chunk keys are read 16 bytes at a time");
static_assert(sizeof(TopkShared) <= 227 * 1024, "shared memory of one CTA");

// Cluster barrier in two halves; every thread of every CTA of the cluster
// executes both, in the same order. Arrive releases and wait acquires this
// thread's shared (local and remote) and global memory accesses at cluster
// scope.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ void cluster_barrier() {
  cluster_arrive();
  cluster_wait();
}

// this CTA's non-zero counts of bins [0, nb) into rank 0's cluster histogram
__device__ __forceinline__ void push_hist(cg::cluster_group& cluster, TopkShared& sh, int nb) {
  uint32_t* dst = cluster.map_shared_rank(sh.cl_hist, 0);
  for (int b = threadIdx.x; b < nb; b += kTopkThreads) {
    const uint32_t v = sh.hist[b];
    if (v != 0u) atomicAdd(dst + b, v);
  }
}

// Every thread of one CTA: the bin of `h` (nb <= 2048 bins) that holds the
// rank-`need` key from the top, the count above it and the count in it, as
// seen by the one thread that finds it (need must lie in 1 .. sum of h).
// Returns true on that thread. Each bin is cleared after it is read.
__device__ __forceinline__ bool pick_bin(uint32_t* warp_tot, uint32_t* h, int nb, uint32_t need, uint32_t& bin,
                                         uint32_t& above, uint32_t& count) {
  const int tid = threadIdx.x;
  // bins from the top: thread i holds bins nb-1-2i and nb-2-2i
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
  const uint32_t h0 = b0 >= 0 ? h[b0] : 0u;
  const uint32_t h1 = b1 >= 0 ? h[b1] : 0u;
  uint32_t total;
  const uint32_t incl = block_incl_scan(h0 + h1, warp_tot, total);
  const uint32_t above0 = incl - h0 - h1, above1 = above0 + h0;
  if (b0 >= 0) h[b0] = 0u;
  if (b1 >= 0) h[b1] = 0u;
  if (b0 >= 0 && need > above0 && need <= above0 + h0) {
    bin = static_cast<uint32_t>(b0);
    above = above0;
    count = h0;
    return true;
  }
  if (b1 >= 0 && need > above1 && need <= above1 + h1) {
    bin = static_cast<uint32_t>(b1);
    above = above1;
    count = h1;
    return true;
  }
  return false;
}

// Rank 0, every thread, once the cluster histogram is complete: the chosen
// bin, written into every CTA's `found`; the cluster histogram is cleared
// for the next pass.
__device__ __forceinline__ void pick_broadcast(cg::cluster_group& cluster, TopkShared& sh, int nb, uint32_t need) {
  uint32_t bin, above, count;
  if (pick_bin(sh.warp_tot, sh.cl_hist, nb, need, bin, above, count)) {
    for (int r = 0; r < kTopkCtas; ++r) {
      uint32_t* f = cluster.map_shared_rank(sh.found, r);
      f[0] = bin;
      f[1] = above;
      f[2] = count;
    }
  }
}

__global__ void __cluster_dims__(kTopkCtas, 1, 1) __launch_bounds__(kTopkThreads, 1)
    topk_select_kernel(const float* __restrict__ scores, int64_t stride, int32_t ncols,
                       const int32_t* __restrict__ lengths, int32_t topk, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  const int len = hi - lo;
  // rows that start on a 16-byte boundary are read 4 scores at a time
  const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
  // the chunk's keys are kept in shared memory by the first pass
  const bool in_smem = len <= kChunkKeys;
  // apply f(key, chunk offset) to every key of the chunk (any order); from
  // shared memory after the first pass where the chunk fits
  auto for_chunk = [&](auto&& f) {
    if (in_smem) {
      const int n4 = len / 4;
      for (int q = tid; q < n4; q += kTopkThreads) {
        const uint4 v = reinterpret_cast<const uint4*>(sh.keys)[q];
        f(v.x, 4 * q);
        f(v.y, 4 * q + 1);
        f(v.z, 4 * q + 2);
        f(v.w, 4 * q + 3);
      }
      for (int i = 4 * n4 + tid; i < len; i += kTopkThreads) f(sh.keys[i], i);
    } else if (vec) {
      const float4* s4 = reinterpret_cast<const float4*>(s + lo);
      const int n4 = len / 4;
      constexpr int kU = 4;  // 16-byte loads in flight per thread
      for (int q0 = 0; q0 < n4; q0 += kU * kTopkThreads) {
        float4 v[kU];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < n4) v[r] = __ldg(s4 + q);
        }
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < n4) {
            f(score_key(v[r].x), 4 * q);
            f(score_key(v[r].y), 4 * q + 1);
            f(score_key(v[r].z), 4 * q + 2);
            f(score_key(v[r].w), 4 * q + 3);
          }
        }
      }
      for (int i = 4 * n4 + tid; i < len; i += kTopkThreads) f(score_key(__ldg(s + lo + i)), i);
    } else {
      for (int i = tid; i < len; i += kTopkThreads) f(score_key(__ldg(s + lo + i)), i);
    }
  };

  // ---- pass 1: key bits 31-21 over the chunk
  for (int b = tid; b < 2048; b += kTopkThreads) {
    sh.hist[b] = 0u;
    if (rank == 0) sh.cl_hist[b] = 0u;
  }
  for (int w = tid; w < kBmWords; w += kTopkThreads) {
    sh.bm_gt[w] = 0u;
    sh.bm_eq[w] = 0u;
  }
  if (tid == 0) {
    sh.pool_n = 0u;
    sh.slot = 0u;
    sh.nfew = 0u;
    // (rank 0 overwrites it; in range whatever happens)
    sh.found[0] = sh.found[1] = sh.found[2] = 0u;
  }
  __syncthreads();
  // rank 0's cleared histogram and pool counter are released here and
  // acquired before the first remote add: the first pass's loads run in
  // between
  cluster_arrive();
  {
    // (for_chunk's global walk, also storing the keys)
    auto hist1 = [&](uint32_t u, int i) {
      atomicAdd(&sh.hist[u >> 21], 1u);
      if (in_smem) sh.keys[i] = u;
    };
    if (vec) {
      const float4* s4 = reinterpret_cast<const float4*>(s + lo);
      const int n4 = len / 4;
      constexpr int kU = 4;
      for (int q0 = 0; q0 < n4; q0 += kU * kTopkThreads) {
        float4 v[kU];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < n4) v[r] = __ldg(s4 + q);
        }
#pragma unroll
        for (int r = 0; r < kU; ++r) {
          const int q = q0 + r * kTopkThreads + tid;
          if (q < n4) {
            const uint4 u = make_uint4(score_key(v[r].x), score_key(v[r].y), score_key(v[r].z), score_key(v[r].w));
            atomicAdd(&sh.hist[u.x >> 21], 1u);
            atomicAdd(&sh.hist[u.y >> 21], 1u);
            atomicAdd(&sh.hist[u.z >> 21], 1u);
            atomicAdd(&sh.hist[u.w >> 21], 1u);
            if (in_smem) reinterpret_cast<uint4*>(sh.keys)[q] = u;
          }
        }
      }
      for (int i = 4 * n4 + tid; i < len; i += kTopkThreads) hist1(score_key(__ldg(s + lo + i)), i);
    } else {
      for (int i = tid; i < len; i += kTopkThreads) hist1(score_key(__ldg(s + lo + i)), i);
    }
  }
  __syncthreads();
  cluster_wait();
  push_hist(cluster, sh, 2048);
  cluster_barrier();
  if (rank == 0) pick_broadcast(cluster, sh, 2048, static_cast<uint32_t>(k));
  cluster_barrier();
  const uint32_t bin1 = sh.found[0], cnt1 = sh.found[2];
  uint32_t need = static_cast<uint32_t>(k) - sh.found[1];  // rank wanted within the bin
  uint32_t prefix = bin1 << 21, mask = 0xffe00000u;
  uint32_t base_gt = 0u, base_eq = 0u;

  const bool pooled = cnt1 <= static_cast<uint32_t>(kPool);  // the same in every CTA
  const uint32_t mine = sh.hist[bin1];                          // this CTA's keys of the bin
  if (pooled && warp == 0) {
    // this CTA's pool segment (one remote atomic, its latency under the
    // listing below) and its count of keys above the bin
    uint32_t a = 0u;
    for (int b = static_cast<int>(bin1) + 1 + lane; b < 2048; b += 32) a += sh.hist[b];
    a = __reduce_add_sync(0xffffffffu, a);
    if (lane == 0) {
      const uint32_t b = atomicAdd(cluster.map_shared_rank(&sh.pool_n, 0), mine);
      sh.base = b;
      uint32_t* sg = cluster.map_shared_rank(&sh.seg[0][0], 0) + 3 * rank;
      sg[0] = b;
      sg[1] = mine;
      sg[2] = a;
    }
  }

  // ---- each thread lists its keys at or above the bin (every position
  // that can still be chosen): short lists, or the chunk is walked instead
  const uint32_t key_lo = bin1 << 21;
  uint32_t nl = 0u, nb1 = 0u;  // keys this thread found at or above the bin, and in it
  if (in_smem) {
    auto note = [&](uint32_t u, int off) {
      if (u >= key_lo) {
        if (nl < static_cast<uint32_t>(kList)) sh.list[nl][tid] = static_cast<uint32_t>(off);
        ++nl;
        nb1 += (u >> 21) == bin1 ? 1u : 0u;
      }
    };
    const int n4 = len / 4;
    for (int q = tid; q < n4; q += kTopkThreads) {
      const uint4 v = reinterpret_cast<const uint4*>(sh.keys)[q];
      note(v.x, 4 * q);
      note(v.y, 4 * q + 1);
      note(v.z, 4 * q + 2);
      note(v.w, 4 * q + 3);
    }
    for (int i = 4 * n4 + tid; i < len; i += kTopkThreads) note(sh.keys[i], i);
  }
  // one block scan: this thread's first slot among the CTA's keys of the
  // bin (low half; the CTA has fewer than 2^16 keys when it lists them) and
  // the number of lists that overflowed (high half)
  uint32_t scan_tot;
  const uint32_t packed = (nb1 & 0xffffu) | (nl > static_cast<uint32_t>(kList) ? 0x10000u : 0u);
  const uint32_t scan_excl = block_incl_scan(packed, sh.warp_tot, scan_tot) - packed;
  const bool listed = in_smem && (scan_tot >> 16) == 0u;

  if (pooled) {
    // ---- the bin's keys into rank 0's pool
    uint32_t* pool0 = cluster.map_shared_rank(sh.pool, 0) + sh.base;
    if (listed) {
      uint32_t at = scan_excl & 0xffffu;
      for (uint32_t j = 0; j < nl; ++j) {
        const uint32_t u = sh.keys[sh.list[j][tid]];
        if ((u >> 21) == bin1) {
          if (at < mine) pool0[at] = u;  // exactly `mine` of them
          ++at;
        }
      }
    }
    // otherwise a warp-uniform walk over the chunk's quads, slots taken a
    // warp at a time
    const int nq = listed ? 0 : (len + 3) / 4;
    for (int q0 = 32 * warp; q0 < nq; q0 += kTopkThreads) {
      const int q = q0 + lane, off = 4 * q;
      uint32_t key[4] = {0u, 0u, 0u, 0u};
      if (q < nq) {
        if (in_smem && off + 4 <= len) {
          const uint4 v = reinterpret_cast<const uint4*>(sh.keys)[q];
          key[0] = v.x;
          key[1] = v.y;
          key[2] = v.z;
          key[3] = v.w;
        } else if (!in_smem && vec && off + 4 <= len) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(s + lo + off));
          key[0] = score_key(v.x);
          key[1] = score_key(v.y);
          key[2] = score_key(v.z);
          key[3] = score_key(v.w);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (off + e < len) key[e] = in_smem ? sh.keys[off + e] : score_key(__ldg(s + lo + off + e));
        }
      }
      uint32_t m = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) m |= (q < nq && off + e < len && (key[e] >> 21) == bin1 ? 1u : 0u) << e;
      if (__any_sync(0xffffffffu, m != 0u)) {
        // this lane's slot among the warp's keys of the bin, in lane order
        const uint32_t c = static_cast<uint32_t>(__popc(m));
        const uint32_t c0 = __ballot_sync(0xffffffffu, c & 1u), c1 = __ballot_sync(0xffffffffu, c & 2u),
                       c2 = __ballot_sync(0xffffffffu, c & 4u);
        const uint32_t below = (1u << lane) - 1u;
        const uint32_t pre = __popc(c0 & below) + 2u * __popc(c1 & below) + 4u * __popc(c2 & below);
        const uint32_t tot = __popc(c0) + 2u * __popc(c1) + 4u * __popc(c2);
        uint32_t at = 0u;
        if (lane == 0) at = atomicAdd(&sh.slot, tot);
        at = __shfl_sync(0xffffffffu, at, 0) + pre;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((m >> e) & 1u) {
            if (at < mine) pool0[at] = key[e];  // exactly `mine` of them
            ++at;
          }
        }
      }
    }
    cluster_barrier();
    if (rank == 0) {
      // ---- the select within the pool (bits 20-10, then 9-0), then each
      // rank's counts of chosen positions
      const int np = static_cast<int>(cnt1);
#pragma unroll 1
      for (int pass = 1; pass < 3; ++pass) {
        const int sb = pass == 1 ? 10 : 0, nb = pass == 1 ? 2048 : 1024;
        if (pass == 2 && sh.found[2] <= 32u) {
          // at most 32 keys share the top 22 bits: their ranks, counted by
          // one warp, give the threshold
          for (int i = tid; i < np; i += kTopkThreads) {
            const uint32_t u = sh.pool[i];
            if ((u & mask) == prefix) {
              const uint32_t c = atomicAdd(&sh.nfew, 1u);
              if (c < 32u) sh.few[c] = u;
            }
          }
          __syncthreads();
          if (warp == 0) {
            const uint32_t nf = min(sh.nfew, 32u);
            const uint32_t u = static_cast<uint32_t>(lane) < nf ? sh.few[lane] : 0u;
            uint32_t n_gt = 0u, n_ge = 0u;
            for (uint32_t j = 0; j < nf; ++j) {
              const uint32_t v = sh.few[j];
              n_gt += v > u ? 1u : 0u;
              n_ge += v >= u ? 1u : 0u;
            }
            // (lanes holding equal keys write the same values)
            if (static_cast<uint32_t>(lane) < nf && n_gt < need && need <= n_ge) {
              sh.found[0] = u;
              sh.found[1] = n_gt;
            }
          }
          __syncthreads();
          prefix = sh.found[0];
          mask = 0xffffffffu;
          need -= sh.found[1];
          break;
        }
        for (int b = tid; b < nb; b += kTopkThreads) sh.hist[b] = 0u;
        __syncthreads();
        for (int i = tid; i < np; i += kTopkThreads) {
          const uint32_t u = sh.pool[i];
          if ((u & mask) == prefix) atomicAdd(&sh.hist[(u >> sb) & (nb - 1)], 1u);
        }
        __syncthreads();
        uint32_t bin, ab, cnt;
        if (pick_bin(sh.warp_tot, sh.hist, nb, need, bin, ab, cnt)) {
          sh.found[0] = bin;
          sh.found[1] = ab;
          sh.found[2] = cnt;
        }
        __syncthreads();
        prefix |= sh.found[0] << sb;
        mask |= static_cast<uint32_t>(nb - 1) << sb;
        need -= sh.found[1];
        __syncthreads();  // found is rewritten by the next pass
      }
      // pool keys above / equal to the threshold, by the rank they came from
      uint32_t gt[kTopkCtas], eq[kTopkCtas];
#pragma unroll
      for (int r = 0; r < kTopkCtas; ++r) gt[r] = eq[r] = 0u;
      for (int i = tid; i < np; i += kTopkThreads) {
        const uint32_t u = sh.pool[i];
        const uint32_t g = u > prefix ? 1u : 0u, e = u == prefix ? 1u : 0u;
#pragma unroll
        for (int r = 0; r < kTopkCtas; ++r) {
          const bool from = static_cast<uint32_t>(i) - sh.seg[r][0] < sh.seg[r][1];
          gt[r] += from ? g : 0u;
          eq[r] += from ? e : 0u;
        }
      }
#pragma unroll
      for (int r = 0; r < kTopkCtas; ++r) {
        const uint32_t wg = __reduce_add_sync(0xffffffffu, gt[r]), we = __reduce_add_sync(0xffffffffu, eq[r]);
        if (lane == 0) {
          sh.part[warp][2 * r] = wg;
          sh.part[warp][2 * r + 1] = we;
        }
      }
      __syncthreads();
      if (tid < 2 * kTopkCtas) {
        uint32_t v = 0u;
        for (int w = 0; w < kTopkWarps; ++w) v += sh.part[w][tid];
        sh.warp_tot[tid] = v;  // [2r]: above, [2r + 1]: equal, from rank r's pool keys
      }
      __syncthreads();
      if (tid < kTopkCtas) {
        uint32_t bg = 0u, be = 0u;
        for (int r = 0; r < tid; ++r) {
          bg += sh.seg[r][2] + sh.warp_tot[2 * r];
          be += sh.warp_tot[2 * r + 1];
        }
        uint32_t* d = cluster.map_shared_rank(sh.res, tid);
        d[0] = prefix;
        d[1] = need;
        d[2] = bg;
        d[3] = be;
      }
    }
    cluster_barrier();  // the last: no CTA touches another's shared memory after it
    prefix = sh.res[0];
    need = sh.res[1];
    base_gt = sh.res[2];
    base_eq = sh.res[3];
  } else {
    // ---- passes 2 and 3 cluster-wide: bits 20-10, then 9-0, of the bin's keys
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
      const int sb = pass == 1 ? 10 : 0, nb = pass == 1 ? 2048 : 1024;
      for (int b = tid; b < nb; b += kTopkThreads) sh.hist[b] = 0u;
      __syncthreads();
      for_chunk([&](uint32_t u, int) {
        if ((u & mask) == prefix) atomicAdd(&sh.hist[(u >> sb) & (nb - 1)], 1u);
      });
      __syncthreads();
      push_hist(cluster, sh, nb);
      cluster_barrier();
      if (rank == 0) pick_broadcast(cluster, sh, nb, need);
      cluster_barrier();
      prefix |= sh.found[0] << sb;
      mask |= static_cast<uint32_t>(nb - 1) << sb;
      need -= sh.found[1];
    }
    // this CTA's positions above / equal to the threshold, into every higher
    // rank; then the counts of the ranks below this one
    uint32_t n_gt = 0u, n_eq = 0u;
    for_chunk([&](uint32_t u, int) {
      n_gt += u > prefix ? 1u : 0u;
      n_eq += u == prefix ? 1u : 0u;
    });
    uint32_t tg, te;
    block_incl_scan(n_gt, sh.warp_tot, tg);
    block_incl_scan(n_eq, sh.warp_tot, te);
    if (tid > rank && tid < kTopkCtas) {
      uint32_t* d = cluster.map_shared_rank(&sh.lower[0][0], tid);
      d[2 * rank] = tg;
      d[2 * rank + 1] = te;
    }
    cluster_barrier();  // the last: no CTA touches another's shared memory after it
    for (int r = 0; r < rank; ++r) {
      base_gt += sh.lower[r][0];
      base_eq += sh.lower[r][1];
    }
  }
  // prefix is the k-th largest key; `need` (>= 1) positions equal to it are
  // taken cluster-wide, the lowest first; base_gt / base_eq count the chosen
  // positions above / equal to it in the chunks before this one

  if (in_smem) {
    // ---- ordered collection from bitmaps of the chunk: thread i holds
    // chunk offsets 32i .. 32i + 31
    auto mark = [&](uint32_t u, uint32_t off) {
      if (u > prefix) atomicOr(&sh.bm_gt[off >> 5], 1u << (off & 31));
      if (u == prefix) atomicOr(&sh.bm_eq[off >> 5], 1u << (off & 31));
    };
    if (listed) {
      for (uint32_t j = 0; j < nl; ++j) {
        const uint32_t off = sh.list[j][tid];
        mark(sh.keys[off], off);
      }
    } else {
      for_chunk([&](uint32_t u, int off) { mark(u, static_cast<uint32_t>(off)); });
    }
    __syncthreads();
    const uint32_t gw = sh.bm_gt[tid], ew = sh.bm_eq[tid];
    const uint32_t c = __popc(gw) | (__popc(ew) << 16);
    uint32_t total;
    const uint32_t excl = block_incl_scan(c, sh.warp_tot, total) - c;
    const uint32_t g = base_gt + (excl & 0xffffu), e = base_eq + (excl >> 16);
    uint32_t sel = gw | ew;
    while (sel) {
      const int j = __ffs(sel) - 1;
      sel &= sel - 1u;
      const uint32_t below = (1u << j) - 1u;
      const uint32_t gj = g + __popc(gw & below), ej = e + __popc(ew & below);
      const uint32_t at = gj + min(ej, need);  // < k when the counts are right; checked all the same
      if ((((gw >> j) & 1u) || ej < need) && at < static_cast<uint32_t>(k)) o[at] = lo + 32 * tid + j;
    }
  } else {
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
        const uint32_t at = gj + min(ej, need);
        if ((((gt >> j) & 1u) || ej < need) && at < static_cast<uint32_t>(k)) o[at] = p0 + j;
      }
      base_gt += total & 0xffffu;
      base_eq += total >> 16;
    }
  }
  if (rank == kTopkCtas - 1)
    for (int i = k + tid; i < topk; i += kTopkThreads) o[i] = -1;
}

// ---------------------------------------------------------------------------
// Rows whose eighths fit in shared memory (the decode's 200K-position rows):
// one exchange of candidates instead of rounds of histograms.
//  * each CTA requests its whole chunk at once, keeps the scores in shared
//    memory and notes each thread's largest score;
//  * each CTA picks its own cut b_r: the q-th largest of its per-thread
//    maxima, q = 3 ceil(k / 8) / 2, so that at least q of its keys lie at or
//    above it (a few hundred on scores like the indexer's);
//  * each CTA lists its keys >= b_r in position order (compared as floats
//    against the score of b_r; NaN scores are listed whatever their key, and
//    every later step compares keys) and copies the list into a segment of
//    its own in every CTA's pool, with b_r, its count and its largest key;
//    after one cluster barrier each CTA holds, for V = max_r b_r, every key
//    >= V of the row. If at least k of them are >= V, the k-th largest key
//    T is >= V and every key that can be chosen
//    is in the pool: each CTA finds T over the pool alone (radix passes from
//    the highest bit where V and the row's largest key differ), counts the
//    chosen keys of the chunks before its own, and writes its chosen
//    positions from its own list;
//  * otherwise (a segment overflowed, or fewer than k keys >= V: bunched
//    winners, heavy ties) the select runs cluster-wide over every key: three
//    radix passes whose histograms every CTA adds into every CTA, one
//    exchange of the per-chunk counts, and an ordered walk of the chunk.
// Block-wide steps use one-barrier scans: the 32 warp totals are summed by
// each warp with a warp reduction instead of a second scan.
constexpr int kResKeys = 32 * 1024;  // longest chunk this kernel takes
constexpr int kSeg = 1024;           // pool keys per source rank
static_assert(kResKeys / kTopkThreads <= 32, "a thread's positions of an ordered walk fit one mask");
static_assert(kSeg <= kTopkThreads, "one listed key per thread in the output step");
static_assert(kTopkWarps == 32, "one warp total per lane");

struct ResShared {
  alignas(16) uint32_t vals[kResKeys];          // the chunk's scores (bits), by chunk offset
  alignas(16) uint32_t pool[kTopkCtas * kSeg];  // rank r's keys >= b_r at [r * kSeg, r * kSeg + seg_n[r])
  uint32_t lpos[kSeg];                          // chunk offsets of this CTA's listed keys, in order
  uint32_t hist[2048];                          // this CTA's counts (zero between uses)
  uint32_t cl_hist[3][2048];                    // fallback: the cluster's counts of pass j
  uint32_t scan[kTopkWarps];
  uint32_t cut[kTopkCtas];     // written by rank r: b_r
  uint32_t top[kTopkCtas];     // written by rank r: its largest key
  uint32_t seg_n[kTopkCtas];   // written by rank r: its keys >= b_r
  uint32_t cnt[kTopkCtas][2];  // fallback, written by rank r: its keys above / equal to the threshold
  uint32_t base[2];            // chosen keys above / equal to the threshold in the chunks before this one
  uint32_t found[4];
  uint32_t few[32];
  uint32_t nfew;
  uint32_t cmax, cmin;         // largest and smallest per-thread maximum (keys)
  uint32_t lmax;               // largest listed key
};
static_assert(sizeof(ResShared) <= 227 * 1024, "shared memory of one CTA");

// Exclusive prefix sum of v over the block's threads, in thread order, and
// the block total; one block barrier. `scan` is written before the barrier
// and read after it: a barrier must separate two uses of the same array.
__device__ __forceinline__ uint32_t block_excl_scan1(uint32_t v, uint32_t* scan, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scan[warp] = x;
  __syncthreads();
  const uint32_t wt = scan[lane];
  total = __reduce_add_sync(0xffffffffu, wt);
  return __reduce_add_sync(0xffffffffu, lane < warp ? wt : 0u) + x - v;
}

// Every thread of one CTA: in the nb-bin histogram h (nb <= 2048, a power of
// two), the bin that holds the rank-`need` key from the top, the count above
// it and its count, on every thread, and the histogram's total; `bin` is
// valid only when 1 <= need <= total. Each bin is cleared after it is read.
// Two block barriers.
__device__ __forceinline__ uint32_t pick_bin1(ResShared& sh, uint32_t* h, int nb, uint32_t need, uint32_t& bin,
                                              uint32_t& above, uint32_t& count) {
  const int tid = threadIdx.x;
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;  // bins from the top
  const uint32_t h0 = b0 >= 0 ? h[b0] : 0u;
  const uint32_t h1 = b1 >= 0 ? h[b1] : 0u;
  uint32_t total;
  const uint32_t above0 = block_excl_scan1(h0 + h1, sh.scan, total), above1 = above0 + h0;
  if (b0 >= 0) h[b0] = 0u;
  if (b1 >= 0) h[b1] = 0u;
  if (b0 >= 0 && need > above0 && need <= above1) {
    sh.found[0] = static_cast<uint32_t>(b0);
    sh.found[1] = above0;
    sh.found[2] = h0;
  }
  if (b1 >= 0 && need > above1 && need <= above1 + h1) {
    sh.found[0] = static_cast<uint32_t>(b1);
    sh.found[1] = above1;
    sh.found[2] = h1;
  }
  __syncthreads();
  bin = sh.found[0];
  above = sh.found[1];
  count = sh.found[2];
  // (found is next written after the barrier of the next scan, which every
  // thread reaches only after these reads)
  return total;
}

// Mask of the bits above the highest bit where a and b differ (all bits when
// they are equal), and that bit (-1 when equal).
__device__ __forceinline__ int common_high_bits(uint32_t a, uint32_t b, uint32_t& mask) {
  const int hb = a == b ? -1 : 31 - __clz(a ^ b);
  mask = hb >= 31 ? 0u : 0xffffffffu << (hb + 1);
  return hb;
}

// Wait until the first r + 1 of n committed copy groups have landed (r is a
// compile-time constant in the unrolled loops that call it).
template <int N>
__device__ __forceinline__ void cp_async_wait_dyn(int r) {
  if constexpr (N > 0) {
    if (r == 0) {
      cp_async_wait<N - 1>();
    } else {
      cp_async_wait_dyn<N - 1>(r - 1);
    }
  }
}

// The float whose key is `key` (for keys of a float: key(-0) gives +0).
__device__ __forceinline__ float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__global__ void __cluster_dims__(kTopkCtas, 1, 1) __launch_bounds__(kTopkThreads, 1)
    topk_resident_kernel(const float* __restrict__ scores, int64_t stride, int32_t ncols,
                         const int32_t* __restrict__ lengths, int32_t topk, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  ResShared& sh = *reinterpret_cast<ResShared*>(topk_smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* s = scores + static_cast<int64_t>(t) * stride;
  int32_t* o = out + static_cast<int64_t>(t) * topk;
  int L = lengths ? __ldg(lengths + t) : ncols;
  L = min(max(L, 0), ncols);
  const int k = min(topk, L);
  if (k == L) {
    if (rank == 0)
      for (int i = tid; i < topk; i += kTopkThreads) o[i] = i < L ? i : -1;
    return;
  }
  const int quads = (L + 3) / 4;
  const int lo = 4 * ((rank * quads) / kTopkCtas), hi = min(L, 4 * (((rank + 1) * quads) / kTopkCtas));
  const int len = hi - lo;  // <= kResKeys (host check on the row length)
  const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;

  // ---- the whole chunk requested first, straight into shared memory by
  // 16-byte asynchronous copies where the row is aligned (one commit group
  // per round of the block's threads; no registers and no L1 lines held);
  // shared memory is cleared while it is on its way
  constexpr int kU = kResKeys / 4 / kTopkThreads;
  const float4* s4 = reinterpret_cast<const float4*>(s + lo);
  const int n4 = vec ? len / 4 : 0;
#pragma unroll
  for (int r = 0; r < kU; ++r) {
    const int q = r * kTopkThreads + tid;
    if (q < n4) cp_async_16(sh.vals + 4 * q, s4 + q);
    cp_async_commit();
  }
  for (int b = tid; b < 2048; b += kTopkThreads) sh.hist[b] = 0u;
  if (tid == 0) {
    sh.nfew = 0u;
    sh.cmax = 0u;
    sh.cmin = 0xffffffffu;
    sh.lmax = 0u;
    sh.base[0] = sh.base[1] = 0u;
  }
  __syncthreads();
  // released here, acquired before the first remote access; the loads run
  // in between
  cluster_arrive();

  // ---- this thread's largest score (as a float: NaN scores are passed
  // over, which only lowers the cut), each round once its copies landed
  float fmx = -INFINITY;
  bool any = false;
#pragma unroll
  for (int r = 0; r < kU; ++r) {
    cp_async_wait_dyn<kU>(r);
    const int q = r * kTopkThreads + tid;
    if (q < n4) {
      const float4 x = reinterpret_cast<const float4*>(sh.vals)[q];  // (this thread's own copy)
      fmx = fmaxf(fmx, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
      any = true;
    }
  }
  for (int i = 4 * n4 + tid; i < len; i += kTopkThreads) {  // the tail, or every score of an unaligned row
    const float x = __ldg(s + lo + i);
    sh.vals[i] = __float_as_uint(x);
    fmx = fmaxf(fmx, x);
    any = true;
  }
  const uint32_t tmax = any ? score_key(fmx) : 0u;
  {
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, tmax);
    const uint32_t wmin = __reduce_min_sync(0xffffffffu, any ? tmax : 0xffffffffu);
    if (lane == 0) {
      atomicMax(&sh.cmax, wmax);
      atomicMin(&sh.cmin, wmin);
    }
  }
  const uint32_t holders = __syncthreads_count(any ? 1 : 0);  // also: keys, cmax and cmin are complete

  // ---- this CTA's cut: the q-th largest per-thread maximum, to the low
  // edge of its bin in one 11-bit digit below the bits that the largest and
  // smallest maxima share (0 with fewer than q maxima)
  const uint32_t q = (3u * static_cast<uint32_t>((k + kTopkCtas - 1) / kTopkCtas) + 1u) / 2u;
  uint32_t cut = 0u;
  if (holders >= q) {
    uint32_t pmask;
    const int hb = common_high_bits(sh.cmin, sh.cmax, pmask);
    if (hb < 0) {
      cut = sh.cmax;
    } else {
      const int w = min(11, hb + 1), sb = hb + 1 - w, nb = 1 << w;
      if (any) atomicAdd(&sh.hist[(tmax >> sb) & (nb - 1)], 1u);
      __syncthreads();
      uint32_t bin, ab, cnt;
      pick_bin1(sh, sh.hist, nb, q, bin, ab, cnt);
      cut = (sh.cmax & pmask) | (bin << sb);
    }
  }

  // ---- this chunk's keys >= cut, listed in position order (thread i walks
  // chunk offsets [per i, per (i + 1)), per a multiple of 4)
  const int per = ((len + kTopkThreads - 1) / kTopkThreads + 3) & ~3;
  const int p0 = min(tid * per, len), p1 = min(p0 + per, len);
  uint32_t nlist;  // this chunk's keys >= cut
  uint32_t* seg = sh.pool + rank * kSeg;
  {
    // key >= cut <=> score >= cf for every score but NaN; !(x < cf) also
    // lists NaN scores, whose keys the later steps compare
    const float cf = key_score(cut);
    uint32_t fm = 0u;  // bit j: chunk offset p0 + j
    if (p1 - p0 == per) {
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4) {
        if (j4 < per) {
          const float4 x = *reinterpret_cast<const float4*>(sh.vals + p0 + j4);
          fm |= ((!(x.x < cf) ? 1u : 0u) | (!(x.y < cf) ? 2u : 0u) | (!(x.z < cf) ? 4u : 0u) | (!(x.w < cf) ? 8u : 0u))
                << j4;
        }
      }
    } else {
      for (int j = 0; j < p1 - p0; ++j) fm |= (!(__uint_as_float(sh.vals[p0 + j]) < cf) ? 1u : 0u) << j;
    }
    uint32_t at = block_excl_scan1(__popc(fm), sh.scan, nlist);
    uint32_t mymax = 0u;
    while (fm) {
      const int j = __ffs(fm) - 1;
      fm &= fm - 1u;
      const uint32_t u = score_key(__uint_as_float(sh.vals[p0 + j]));
      mymax = max(mymax, u);
      if (at < static_cast<uint32_t>(kSeg)) {
        seg[at] = u;
        sh.lpos[at] = static_cast<uint32_t>(p0 + j);
      }
      ++at;
    }
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, mymax);
    if (lane == 0 && wmax != 0u) atomicMax(&sh.lmax, wmax);
  }
  __syncthreads();
  // ---- the list into every other CTA's pool, with the cut, the count and
  // the largest key into every CTA
  cluster_wait();
  {
    const int nu = (static_cast<int>(min(nlist, static_cast<uint32_t>(kSeg))) + 3) / 4;
    for (int u = tid; u < nu; u += kTopkThreads) {
      const uint4 x = reinterpret_cast<const uint4*>(seg)[u];
#pragma unroll
      for (int r = 0; r < kTopkCtas; ++r)
        if (r != rank) reinterpret_cast<uint4*>(cluster.map_shared_rank(seg, r))[u] = x;
    }
    if (tid < kTopkCtas) {
      cluster.map_shared_rank(sh.seg_n, tid)[rank] = nlist;
      cluster.map_shared_rank(sh.cut, tid)[rank] = cut;
      cluster.map_shared_rank(sh.top, tid)[rank] = sh.lmax;
    }
  }
  cluster_barrier();  // every pool is complete

  // V, the row's largest key (the largest listed one) and whether every
  // list fit, by warp reductions over lanes 0-7
  const uint32_t hn = lane < kTopkCtas ? sh.seg_n[lane] : 0u;
  const uint32_t V = __reduce_max_sync(0xffffffffu, lane < kTopkCtas ? sh.cut[lane] : 0u);
  const uint32_t vmax = __reduce_max_sync(0xffffffffu, lane < kTopkCtas ? sh.top[lane] : 0u);
  bool fast = __reduce_max_sync(0xffffffffu, hn) <= static_cast<uint32_t>(kSeg);
  // this thread's slot of every segment, and which of them hold keys >= V
  uint32_t pk[kTopkCtas];
  uint32_t vm = 0u;
#pragma unroll
  for (int m = 0; m < kTopkCtas; ++m) {
    pk[m] = sh.pool[m * kSeg + tid];
    vm |= (static_cast<uint32_t>(tid) < __shfl_sync(0xffffffffu, hn, m) && pk[m] >= V ? 1u : 0u) << m;
  }
  // (every CTA computes the same V, vmax, fast, and below the same pool
  // histograms, so every CTA takes the same path)

  uint32_t prefix = 0u, mask = 0u, need = static_cast<uint32_t>(k);
  if (fast) {
    // ---- the k-th largest key among the pool's keys >= V (all of the row's
    // keys >= V), every CTA on its own copy; they lie in [V, vmax] and share
    // the bits above the highest bit where V and vmax differ
    int hb = common_high_bits(V, vmax, mask);
    prefix = vmax & mask;
    bool first = true;
    // (the first pass always runs: it also counts the keys >= V; with
    // V == vmax it is a one-bit pass that changes nothing else)
#pragma unroll 1
    while (first || hb >= 0) {
      const int w = hb >= 0 ? min(11, hb + 1) : 1, sb = hb >= 0 ? hb + 1 - w : 0, nb = 1 << w;
#pragma unroll
      for (int m = 0; m < kTopkCtas; ++m)
        if (((vm >> m) & 1u) && (pk[m] & mask) == prefix) atomicAdd(&sh.hist[(pk[m] >> sb) & (nb - 1)], 1u);
      __syncthreads();
      uint32_t bin, ab, cnt;
      const uint32_t total = pick_bin1(sh, sh.hist, nb, need, bin, ab, cnt);
      if (first && total < need) {  // fewer than k keys >= V
        fast = false;
        break;
      }
      first = false;
      prefix |= bin << sb;
      mask |= static_cast<uint32_t>(nb - 1) << sb;
      need -= ab;
      hb = sb - 1;
      if (hb >= 0 && cnt <= 32u) {
        // at most 32 keys left in the bin: warp a ranks key a against all
#pragma unroll
        for (int m = 0; m < kTopkCtas; ++m) {
          if (((vm >> m) & 1u) && (pk[m] & mask) == prefix) {
            const uint32_t c = atomicAdd(&sh.nfew, 1u);
            if (c < 32u) sh.few[c] = pk[m];
          }
        }
        __syncthreads();
        const uint32_t nf = min(sh.nfew, 32u);
        if (static_cast<uint32_t>(warp) < nf) {
          const uint32_t ua = sh.few[warp];
          const uint32_t ub = static_cast<uint32_t>(lane) < nf ? sh.few[lane] : 0u;
          const bool inb = static_cast<uint32_t>(lane) < nf;
          const uint32_t n_gt = __popc(__ballot_sync(0xffffffffu, inb && ub > ua));
          const uint32_t n_ge = __popc(__ballot_sync(0xffffffffu, inb && ub >= ua));
          // (warps holding equal keys write the same values)
          if (lane == 0 && n_gt < need && need <= n_ge) {
            sh.found[0] = ua;
            sh.found[3] = n_gt;
          }
        }
        __syncthreads();
        prefix = sh.found[0];
        mask = 0xffffffffu;
        need -= sh.found[3];
        break;
      }
    }
  }
  if (fast) {
    // ---- chosen keys of the chunks before this one (all >= T >= V: in the pool)
    uint32_t g = 0u, e = 0u;
#pragma unroll
    for (int m = 0; m < kTopkCtas; ++m) {
      const bool in = m < rank && ((vm >> m) & 1u);
      g += in && pk[m] > prefix ? 1u : 0u;
      e += in && pk[m] == prefix ? 1u : 0u;
    }
    const uint32_t wg = __reduce_add_sync(0xffffffffu, g), we = __reduce_add_sync(0xffffffffu, e);
    if (lane == 0 && (wg | we) != 0u) {
      atomicAdd(&sh.base[0], wg);
      atomicAdd(&sh.base[1], we);
    }
    // ---- this chunk's chosen positions, from its list (position order)
    const bool in = static_cast<uint32_t>(tid) < nlist;
    const uint32_t u = in ? seg[tid] : 0u;
    const bool gt = in && u > prefix, eq = in && u == prefix;
    uint32_t total;
    const uint32_t c = (gt ? 1u : 0u) | (eq ? 0x10000u : 0u);
    const uint32_t excl = block_excl_scan1(c, sh.scan, total);  // (its barrier also completes base)
    const uint32_t gj = sh.base[0] + (excl & 0xffffu), ej = sh.base[1] + (excl >> 16);
    const uint32_t at = gj + min(ej, need);  // < k when the counts are right; checked all the same
    if ((gt || (eq && ej < need)) && at < static_cast<uint32_t>(k)) o[at] = lo + static_cast<int>(sh.lpos[tid]);
  } else {
    // ---- the select cluster-wide over every key of the row: each pass's
    // histogram added into every CTA's, then every CTA picks the same bin
    prefix = 0u;
    mask = 0u;
    need = static_cast<uint32_t>(k);
    for (int b = tid; b < 3 * 2048; b += kTopkThreads) (&sh.cl_hist[0][0])[b] = 0u;
    for (int b = tid; b < 2048; b += kTopkThreads) sh.hist[b] = 0u;
    cluster_barrier();  // every CTA's counts are cleared before the first remote add
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int sb = pass == 0 ? 21 : pass == 1 ? 10 : 0, nb = pass == 2 ? 1024 : 2048;
      for (int i = tid; i < len; i += kTopkThreads) {
        const uint32_t u = score_key(__uint_as_float(sh.vals[i]));
        if ((u & mask) == prefix) atomicAdd(&sh.hist[(u >> sb) & (nb - 1)], 1u);
      }
      __syncthreads();
      for (int b = tid; b < nb; b += kTopkThreads) {
        const uint32_t x = sh.hist[b];
        if (x != 0u) {
          sh.hist[b] = 0u;
#pragma unroll
          for (int r = 0; r < kTopkCtas; ++r) atomicAdd(cluster.map_shared_rank(sh.cl_hist[pass], r) + b, x);
        }
      }
      cluster_barrier();
      uint32_t bin, ab, cnt;
      pick_bin1(sh, sh.cl_hist[pass], nb, need, bin, ab, cnt);
      prefix |= bin << sb;
      mask |= static_cast<uint32_t>(nb - 1) << sb;
      need -= ab;
    }
    // this chunk's keys above / equal to the threshold, into every CTA
    uint32_t n_gt = 0u, n_eq = 0u;
    for (int i = tid; i < len; i += kTopkThreads) {
      const uint32_t u = score_key(__uint_as_float(sh.vals[i]));
      n_gt += u > prefix ? 1u : 0u;
      n_eq += u == prefix ? 1u : 0u;
    }
    uint32_t tg;
    block_excl_scan1(n_gt | (n_eq << 16), sh.scan, tg);  // (each count <= kResKeys < 2^16)
    if (tid < kTopkCtas) {
      uint32_t* d = cluster.map_shared_rank(&sh.cnt[0][0], tid) + 2 * rank;
      d[0] = tg & 0xffffu;
      d[1] = tg >> 16;
    }
    cluster_barrier();  // the last access to another CTA's memory on this path
    uint32_t base_gt = 0u, base_eq = 0u;
    for (int r = 0; r < rank; ++r) {
      base_gt += sh.cnt[r][0];
      base_eq += sh.cnt[r][1];
    }
    // ---- ordered output: thread i walks chunk offsets [per i, per (i + 1))
    uint32_t gw = 0u, ew = 0u;  // bit j: chunk offset p0 + j
    for (int j = 0; j < p1 - p0; ++j) {
      const uint32_t u = score_key(__uint_as_float(sh.vals[p0 + j]));
      gw |= (u > prefix ? 1u : 0u) << j;
      ew |= (u == prefix ? 1u : 0u) << j;
    }
    uint32_t total;
    const uint32_t c = __popc(gw) | (__popc(ew) << 16);
    const uint32_t excl = block_excl_scan1(c, sh.scan, total);
    const uint32_t g = base_gt + (excl & 0xffffu), e = base_eq + (excl >> 16);
    uint32_t sel = gw | ew;
    while (sel) {
      const int j = __ffs(sel) - 1;
      sel &= sel - 1u;
      const uint32_t below = (1u << j) - 1u;
      const uint32_t gj = g + __popc(gw & below), ej = e + __popc(ew & below);
      const uint32_t at = gj + min(ej, need);
      if ((((gw >> j) & 1u) || ej < need) && at < static_cast<uint32_t>(k)) o[at] = lo + p0 + j;
    }
  }
  if (rank == kTopkCtas - 1)
    for (int i = k + tid; i < topk; i += kTopkThreads) o[i] = -1;
}

cudaError_t launch_topk_select(const float* scores, int64_t stride, int32_t ncols, const int32_t* lengths, int32_t T,
                               int32_t topk, int32_t* out, cudaStream_t stream) {
  // rows whose longest chunk fits in shared memory take the resident kernel
  const int64_t quads = (static_cast<int64_t>(ncols) + 3) / 4;
  const bool resident = 4 * ((quads + kTopkCtas - 1) / kTopkCtas) <= kResKeys;
  const int dyn = resident ? static_cast<int>(sizeof(ResShared)) : static_cast<int>(sizeof(TopkShared));
  const void* fn = resident ? reinterpret_cast<const void*>(topk_resident_kernel)
                            : reinterpret_cast<const void*>(topk_select_kernel);
  // the attribute is set once per device and kernel; a caller that sees the
  // flag (acquire) also sees the attribute set by the caller that raised it
  // (release)
  static std::atomic<bool> attr_set[2][kMaxHostDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::atomic<bool>* flag = (dev >= 0 && dev < kMaxHostDevices) ? &attr_set[resident ? 1 : 0][dev] : nullptr;
  if (!flag || !flag->load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    if (flag) flag->store(true, std::memory_order_release);
  }
  if (resident)
    topk_resident_kernel<<<dim3(kTopkCtas, T), kTopkThreads, dyn, stream>>>(scores, stride, ncols, lengths, topk, out);
  else
    topk_select_kernel<<<dim3(kTopkCtas, T), kTopkThreads, dyn, stream>>>(scores, stride, ncols, lengths, topk, out);
  return cudaGetLastError();
}

}  // namespace nvmla
