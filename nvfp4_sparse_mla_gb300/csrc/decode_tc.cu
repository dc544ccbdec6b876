// Sparse MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: "Prime Inference: Fast, Reliable Serving for Frontier
// Open Models", section "A native NVFP4 sparse-MLA decode kernel" -- for each
// query token only the rows the indexer selected are loaded, unpacked on chip
// and attended to with FP16 operands and FP32 accumulation, with no FP8
// staging buffer in GPU memory. "Prime Intellect unveils Prime Inference",
// section "4-bit caches open the way": item 1 (one warp group unpacks rows
// while others compute scores and accumulate), item 3 (empty slots of the
// 2048-slot list contribute nothing).
//
// Design on sm_103a (one CTA = one token x 64 heads x a range of its slots):
//
//   warp 8  gather:  computes each slot's cache row from the index list and
//                    the block table, then moves the 352-byte rows into a
//                    double-buffered raw tile in shared memory with one
//                    cp.async.bulk per row (the TMA engine does the gather).
//   warps 0-3 unpack: turn raw rows into fp16 operand chunks (E2M1 x E4M3 is
//                    exact in fp16) in a two-slot ring, 128B-swizzled in the
//                    tcgen05 canonical layouts: K chunks (128 rows x 64 dims,
//                    K-major) for QK, V chunks (64 rows x 128 value dims,
//                    MN-major) for PV. The latent is unpacked twice (as K and
//                    as V): the 72 KB query block and the raw tiles leave no
//                    room to keep a whole fp16 tile resident.
//   warp 9  MMA:     one thread issues tcgen05.mma. Both contractions keep
//                    M = 128 by putting rows (keys) or value dims in M:
//                      S^T[128 rows, 64 heads]  = K[128 x 576] . Q^T
//                      O^T[512 dims, 64 heads] += V^T[512 x 128] . P^T
//                    S^T is double-buffered in TMEM (2 x 64 columns), O^T
//                    takes 4 x 64 columns.
//   warps 4-7 softmax: thread = row (TMEM lane). Per-head maxima and sums
//                    are reduced across rows with a transposing butterfly and
//                    shared memory; P^T goes to shared memory as fp16. The
//                    running maximum is only raised when a tile exceeds it by
//                    more than 2^8 (P stays below 256, safe in fp16), and
//                    only then is O^T rescaled in TMEM.
//
// Key splits: several CTAs share a token; each writes (O, m, l) partials and a
// merge kernel combines them, or a single CTA writes out/lse directly.
// Every wait is bounded: on timeout the CTA sets NVMLA_ERRW_WAIT_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and exits.
#include "common.cuh"

namespace nvmla {

namespace tc {

constexpr int kTile = 128;  // rows per tile (MMA M for QK)
constexpr int kHeads = 64;  // heads per CTA (MMA N)
constexpr int kThreads = 320;
constexpr int kProducerWarps = 4;  // warps 0-3
constexpr int kSoftmaxWarp0 = 4;   // warps 4-7
constexpr int kGatherWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRing = 2;
constexpr int kChunkBytes = 16384;
constexpr int kKChunks = 9;  // 8 latent + 1 RoPE chunk of 64 dims
constexpr int kVChunks = 8;  // 4 blocks of 128 value dims x 2 halves of 64 rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T buffers: [0,64) and [64,128)
constexpr uint32_t kColO = 128;   // O^T blocks: [128 + 64 j, +64)
constexpr float kTau = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr uint32_t kSpinLimit = 1u << 22;

// shared memory map (bytes)
constexpr int kOffQ = 0;                                   // 9 x 8 KB
constexpr int kOffRaw = kOffQ + 9 * 8192;                  // 2 x 45056
constexpr int kRawBytes = kTile * kRowBytes;               // 45056
constexpr int kOffRing = kOffRaw + 2 * kRawBytes;          // 2 x 16 KB
constexpr int kOffPT = kOffRing + kRing * kChunkBytes;     // 16 KB
constexpr int kOffSlots = kOffPT + kChunkBytes;            // 2 x 128 int32
constexpr int kOffRed = kOffSlots + 2 * kTile * 4;         // 4 x 64 fp32 (maxima)
constexpr int kOffRedSum = kOffRed + 4 * kHeads * 4;       // 4 x 64 fp32 (sums)
constexpr int kOffM = kOffRedSum + 4 * kHeads * 4;         // 64 fp32
constexpr int kOffL = kOffM + kHeads * 4;                  // 64 fp32
constexpr int kOffAlpha = kOffL + kHeads * 4;              // 64 fp32
constexpr int kOffBar = kOffAlpha + kHeads * 4;            // barriers
enum Bar {
  kBarRawFull = 0,    // 2
  kBarRawEmpty = 2,   // 2
  kBarRingFull = 4,   // 2
  kBarRingEmpty = 6,  // 2
  kBarSFull = 8,      // 2
  kBarSFree = 10,     // 2
  kBarPFull = 12,
  kBarPFree = 13,
  kBarODone = 14,
  kBarQReady = 15,
  kBarDrain = 16,
  kNumBars = 17
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // room to align the base to 1 KB

struct Params {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;
  RowSelect sel;
  int T, H, topk;
  float sl2;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;
  float* ws_ml;
  int num_splits;
  int tiles_total;
  int32_t* err_word;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false (and
// raises the CTA's abort flag) on timeout or when another role aborted.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err_word) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (i > 32) __nanosleep(64);
  }
  if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) report_error(err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  return false;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// shared-memory matrix descriptor: start, leading/stride byte offsets,
// version 1 (sm_100 family), 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t{1} << 46) | (uint64_t{2} << 61);
}

// instruction descriptor, kind::f16: fp16 A/B, fp32 D, M = 128, N = 64
__host__ __device__ constexpr uint32_t idesc_f16(bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((64u >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define NVMLA_TMEM_LD16(taddr, r, o)                                                                          \
  asm volatile(                                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
      : "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]),       \
        "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]), "=r"(r[o + 11]),     \
        "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15])                                    \
      : "r"(taddr))

#define NVMLA_TMEM_ST16(taddr, r, o)                                                                          \
  asm volatile(                                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" \
      ::"r"(taddr), "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]), "r"(r[o + 5]), \
      "r"(r[o + 6]), "r"(r[o + 7]), "r"(r[o + 8]), "r"(r[o + 9]), "r"(r[o + 10]), "r"(r[o + 11]),              \
      "r"(r[o + 12]), "r"(r[o + 13]), "r"(r[o + 14]), "r"(r[o + 15])                                          \
      : "memory")

// 64 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  NVMLA_TMEM_LD16(taddr + 0, r, 0);
  NVMLA_TMEM_LD16(taddr + 16, r, 16);
  NVMLA_TMEM_LD16(taddr + 32, r, 32);
  NVMLA_TMEM_LD16(taddr + 48, r, 48);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  NVMLA_TMEM_ST16(taddr + 0, r, 0);
  NVMLA_TMEM_ST16(taddr + 16, r, 16);
  NVMLA_TMEM_ST16(taddr + 32, r, 32);
  NVMLA_TMEM_ST16(taddr + 48, r, 48);
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// named barrier among the four softmax warps (id 1), with an OR reduction
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool softmax_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void qconv_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

// swizzled byte offset of 16-byte chunk c of row r inside a 128B-swizzled
// region (rows of 128 bytes, 8-row atoms of 1 KB)
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// 16 E2M1 codes (8 bytes) times one scale -> two 16-byte fp16 chunks
__device__ __forceinline__ void unpack16(uint32_t lo, uint32_t hi, uint32_t s2, uint4& a, uint4& b) {
  uint32_t h[4];
  e2m1x8_to_f16x8(lo, h);
  a = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
  e2m1x8_to_f16x8(hi, h);
  b = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
}

// 64 latent values (32 code bytes + 4 scale bytes) of one raw row into one
// 128-byte swizzled fp16 row
__device__ __forceinline__ void unpack_row64(const uint8_t* raw_row, int code_off, int scale_off, uint8_t* dst_base,
                                             int r) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(raw_row + code_off);
  const uint4 c1 = *reinterpret_cast<const uint4*>(raw_row + code_off + 16);
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(raw_row + scale_off);
  uint4 a, b;
  unpack16(c0.x, c0.y, e4m3_to_f16x2_bcast(sc & 0xffu), a, b);
  *reinterpret_cast<uint4*>(dst_base + swz(r, 0)) = a;
  *reinterpret_cast<uint4*>(dst_base + swz(r, 1)) = b;
  unpack16(c0.z, c0.w, e4m3_to_f16x2_bcast((sc >> 8) & 0xffu), a, b);
  *reinterpret_cast<uint4*>(dst_base + swz(r, 2)) = a;
  *reinterpret_cast<uint4*>(dst_base + swz(r, 3)) = b;
  unpack16(c1.x, c1.y, e4m3_to_f16x2_bcast((sc >> 16) & 0xffu), a, b);
  *reinterpret_cast<uint4*>(dst_base + swz(r, 4)) = a;
  *reinterpret_cast<uint4*>(dst_base + swz(r, 5)) = b;
  unpack16(c1.z, c1.w, e4m3_to_f16x2_bcast(sc >> 24), a, b);
  *reinterpret_cast<uint4*>(dst_base + swz(r, 6)) = a;
  *reinterpret_cast<uint4*>(dst_base + swz(r, 7)) = b;
}

__device__ __forceinline__ void zero_row(uint8_t* dst_base, int r) {
#pragma unroll
  for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst_base + swz(r, c)) = make_uint4(0, 0, 0, 0);
}

// transposing butterfly: 64 values per lane -> lane L holds the reduction
// over the warp's 32 lanes for heads 2L and 2L+1 (in v[0], v[1])
template <bool kMax>
__device__ __forceinline__ void warp_reduce64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int n = 32 >> step;  // values kept after this step
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = upper ? v[i] : v[i + n];
      const float keep = upper ? v[i + n] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * kHeads;

  int32_t* slots = reinterpret_cast<int32_t*>(smem + kOffSlots);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
  float* m_run = reinterpret_cast<float*>(smem + kOffM);
  float* l_run = reinterpret_cast<float*>(smem + kOffL);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return sbase + kOffBar + 8 * i; };

  const int tile_lo = (split * p.tiles_total) / p.num_splits;
  const int tile_hi = ((split + 1) * p.tiles_total) / p.num_splits;
  const int kbeg = tile_lo * kTile;
  const int kend = min(tile_hi * kTile, p.topk);
  const int ntiles = max(0, (kend - kbeg + kTile - 1) / kTile);

  if (tid == 0) {
    mbar_init(bar(kBarRawFull + 0), 1);
    mbar_init(bar(kBarRawFull + 1), 1);
    mbar_init(bar(kBarRawEmpty + 0), 128);
    mbar_init(bar(kBarRawEmpty + 1), 128);
    mbar_init(bar(kBarRingFull + 0), 128);
    mbar_init(bar(kBarRingFull + 1), 128);
    mbar_init(bar(kBarRingEmpty + 0), 1);
    mbar_init(bar(kBarRingEmpty + 1), 1);
    mbar_init(bar(kBarSFull + 0), 1);
    mbar_init(bar(kBarSFull + 1), 1);
    mbar_init(bar(kBarSFree + 0), 128);
    mbar_init(bar(kBarSFree + 1), 128);
    mbar_init(bar(kBarPFull), 128);
    mbar_init(bar(kBarPFree), 1);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarQReady), 256);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kHeads) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
    alpha_s[tid] = 1.f;
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int last_issued[2] = {-1, -1};  // gather warp: last tile copied into each buffer
  if (warp == kGatherWarp) {
    // ------------------------------------------------------------ gather
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      if (i >= 2) {
        bool okw = (lane == 0) ? wait_bar(bar(kBarRawEmpty + b), ((i >> 1) - 1) & 1, abort_flag, p.err_word) : false;
        if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      }
      const int k0 = kbeg + i * kTile;
      int32_t s4[4];
      int nvalid = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        const int k = k0 + r;
        s4[j] = (k < kend) ? static_cast<int32_t>(p.sel.slot(t, k, p.err_word, blockIdx.z == 0)) : -1;
        slots[b * kTile + r] = s4[j];
        nvalid += __popc(__ballot_sync(0xffffffffu, s4[j] >= 0));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_tx(bar(kBarRawFull + b), static_cast<uint32_t>(nvalid) * kRowBytes);
      __syncwarp();
      const uint32_t dst = sbase + kOffRaw + b * kRawBytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        if (s4[j] >= 0)
          bulk_g2s(dst + r * kRowBytes, p.cache + static_cast<int64_t>(s4[j]) * kRowBytes, kRowBytes,
                   bar(kBarRawFull + b));
      }
      last_issued[b] = i;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(false, false);
      constexpr uint32_t idesc_pv = idesc_f16(true, true);
      bool ok = wait_bar(bar(kBarQReady), 0, abort_flag, p.err_word);
      tc_fence_after();
      uint32_t g = 0;  // ring position
      auto qk = [&](int i) -> bool {
        const int b = i & 1;
        if (i >= 2 && !wait_bar(bar(kBarSFree + b), ((i >> 1) - 1) & 1, abort_flag, p.err_word)) return false;
        tc_fence_after();
        const uint32_t d_s = tmem + kColS + 64 * b;
        for (int c = 0; c < kKChunks; ++c, ++g) {
          const uint32_t slot = g % kRing;
          if (!wait_bar(bar(kBarRingFull + slot), (g / kRing) & 1, abort_flag, p.err_word)) return false;
          tc_fence_after();
          const uint32_t a0 = sbase + kOffRing + slot * kChunkBytes;
          const uint32_t b0 = sbase + kOffQ + c * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16(d_s, sdesc(a0 + 32 * ks, 16, 1024), sdesc(b0 + 32 * ks, 16, 1024), idesc_qk, (c | ks) != 0);
          mma_commit(bar(kBarRingEmpty + slot));
        }
        mma_commit(bar(kBarSFull + b));
        return true;
      };
      auto pv = [&](int i) -> bool {
        if (!wait_bar(bar(kBarPFull), i & 1, abort_flag, p.err_word)) return false;
        tc_fence_after();
        const uint32_t pt = sbase + kOffPT;
        for (int v = 0; v < kVChunks; ++v, ++g) {
          const uint32_t slot = g % kRing;
          if (!wait_bar(bar(kBarRingFull + slot), (g / kRing) & 1, abort_flag, p.err_word)) return false;
          tc_fence_after();
          const int j = v >> 1, kh = v & 1;
          const uint32_t a0 = sbase + kOffRing + slot * kChunkBytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16(tmem + kColO + 64 * j, sdesc(a0 + 2048 * ks, 8192, 1024),
                    sdesc(pt + 2048 * (kh * 4 + ks), 8192, 1024), idesc_pv, !(i == 0 && kh == 0 && ks == 0));
          mma_commit(bar(kBarRingEmpty + slot));
        }
        mma_commit(bar(kBarPFree));
        mma_commit(bar(kBarODone));
        return true;
      };
      // QK of tile s+1 is issued before PV of tile s, so the tensor core
      // works while the softmax warps turn S(s) into P(s)
      if (ok && ntiles > 0) ok = qk(0);
      for (int st = 1; st <= ntiles && ok; ++st) {
        if (st < ntiles) ok = qk(st);
        if (ok) ok = pv(st - 1);
      }
      // drain: every MMA issued so far has finished once this commit lands
      mma_commit(bar(kBarDrain));
      uint32_t spins = 0;
      while (!mbar_test(bar(kBarDrain), 0) && ++spins < kSpinLimit) __nanosleep(64);
    }
    __syncwarp();
  } else if (warp < kProducerWarps) {
    // ------------------------------------------------------------ unpack
    // Q block -> fp16, K-major 128B-swizzled (shared with the softmax warps)
    for (int i = tid; i < kHeads * 72; i += 256) {
      const int h = i / 72, j = i % 72, c = j >> 3, q = j & 7;
      const int64_t qh = static_cast<int64_t>(t) * p.H + h0 + h;
      const uint4 v = c < 8 ? __ldg(reinterpret_cast<const uint4*>(p.q_latent + qh * kLatent) + j)
                            : __ldg(reinterpret_cast<const uint4*>(p.q_rope + qh * kRope) + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(bf16_bits_to_f32(w[e] & 0xffffu), bf16_bits_to_f32(w[e] >> 16));
      *reinterpret_cast<uint4*>(smem + kOffQ + c * 8192 + swz(h, q)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_async_smem();
    mbar_arrive(bar(kBarQReady));
    bool ok = true;
    uint32_t g = 0;
    const int r = tid;           // row of the K chunks produced by this thread
    const int rl = tid & 63;     // V chunks: row within the 64-row half ...
    const int hv = tid >> 6;     // ... and which 64 of the block's 128 value dims
    auto kchunks = [&](int i) -> bool {
      const int b = i & 1;
      if (!wait_bar(bar(kBarRawFull + b), (i >> 1) & 1, abort_flag, p.err_word)) return false;
      const uint8_t* raw = smem + kOffRaw + b * kRawBytes;
      const bool valid_r = slots[b * kTile + r] >= 0;
      for (int c = 0; c < kKChunks; ++c, ++g) {
        const uint32_t slot = g % kRing;
        if (!wait_bar(bar(kBarRingEmpty + slot), ((g / kRing) & 1) ^ 1, abort_flag, p.err_word)) return false;
        uint8_t* dst = smem + kOffRing + slot * kChunkBytes;
        if (!valid_r) {
          zero_row(dst, r);
        } else if (c < 8) {
          unpack_row64(raw + r * kRowBytes, 32 * c, kScaleOff + 4 * c, dst, r);
        } else {
          const uint4* rp = reinterpret_cast<const uint4*>(raw + r * kRowBytes + kRopeOff);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = rp[q];
            uint4 a, bb;
            e4m3x4_to_f16x4(v.x, a.x, a.y);
            e4m3x4_to_f16x4(v.y, a.z, a.w);
            e4m3x4_to_f16x4(v.z, bb.x, bb.y);
            e4m3x4_to_f16x4(v.w, bb.z, bb.w);
            *reinterpret_cast<uint4*>(dst + swz(r, 2 * q)) = a;
            *reinterpret_cast<uint4*>(dst + swz(r, 2 * q + 1)) = bb;
          }
        }
        fence_async_smem();
        mbar_arrive(bar(kBarRingFull + slot));
      }
      return true;
    };
    // V chunk v: value block j = v / 2 (128 dims), rows 64 * (v % 2) .. +63
    auto vchunks = [&](int i) -> bool {
      const int b = i & 1;
      const uint8_t* raw = smem + kOffRaw + b * kRawBytes;
      const int32_t* sl = slots + b * kTile;
      for (int v = 0; v < kVChunks; ++v, ++g) {
        const uint32_t slot = g % kRing;
        if (!wait_bar(bar(kBarRingEmpty + slot), ((g / kRing) & 1) ^ 1, abort_flag, p.err_word)) return false;
        const int j = v >> 1, kh = v & 1;
        const int row = 64 * kh + rl;
        uint8_t* dst = smem + kOffRing + slot * kChunkBytes + hv * 8192;
        if (sl[row] >= 0) {
          unpack_row64(raw + row * kRowBytes, 64 * j + 32 * hv, kScaleOff + 8 * j + 4 * hv, dst, rl);
        } else {
          zero_row(dst, rl);
        }
        fence_async_smem();
        mbar_arrive(bar(kBarRingFull + slot));
      }
      mbar_arrive(bar(kBarRawEmpty + b));
      return true;
    };
    if (ntiles > 0) ok = kchunks(0);
    for (int st = 1; st <= ntiles && ok; ++st) {
      if (st < ntiles) ok = kchunks(st);
      if (ok) ok = vchunks(st - 1);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int sw = warp - kSoftmaxWarp0;  // 0..3 = TMEM lane quadrant
    const int k = sw * 32 + lane;          // row of this thread
    // help with the Q conversion (threads 128..255 take the odd halves)
    for (int i = tid; i < kHeads * 72; i += 256) {
      const int h = i / 72, j = i % 72, c = j >> 3, q = j & 7;
      const int64_t qh = static_cast<int64_t>(t) * p.H + h0 + h;
      const uint4 v = c < 8 ? __ldg(reinterpret_cast<const uint4*>(p.q_latent + qh * kLatent) + j)
                            : __ldg(reinterpret_cast<const uint4*>(p.q_rope + qh * kRope) + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(bf16_bits_to_f32(w[e] & 0xffffu), bf16_bits_to_f32(w[e] >> 16));
      *reinterpret_cast<uint4*>(smem + kOffQ + c * 8192 + swz(h, q)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_async_smem();
    mbar_arrive(bar(kBarQReady));

    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int b = i & 1;
      ok = wait_bar(bar(kBarSFull + b), (i >> 1) & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(tmem + lane_base + kColS + 64 * b, sr);
      tc_fence_before();
      mbar_arrive(bar(kBarSFree + b));
      const bool valid = slots[b * kTile + k] >= 0;
      float s[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) s[h] = valid ? __uint_as_float(sr[h]) * p.sl2 : -INFINITY;
      // per-head maximum over the tile's 128 rows
      float v[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) v[h] = s[h];
      warp_reduce64<true>(v, lane);
      red[sw * 64 + 2 * lane] = v[0];
      red[sw * 64 + 2 * lane + 1] = v[1];
      softmax_sync();
      bool need = false;
      if (sw == 0 || sw == 1) {
        const int h = k;  // 0..63
        const float mt = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
        const float mo = m_run[h];
        float mn = mo, al = 1.f;
        if (mo == -INFINITY) {
          mn = mt;
        } else if (mt > mo + kTau) {
          mn = mt;
          al = exp2f(mo - mn);
          need = true;
        }
        m_run[h] = mn;
        alpha_s[h] = al;
      }
      need = softmax_sync_or(need);
      // P = exp2(s - m) for this row
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float m = m_run[h];
        s[h] = (m == -INFINITY) ? 0.f : exp2f(s[h] - m);
      }
      // P^T row -> shared memory (fp16, MN-major, 128B-swizzled)
      if (i >= 1) {
        ok = wait_bar(bar(kBarPFree), (i - 1) & 1, abort_flag, p.err_word);
        if (softmax_sync_or(!ok)) {
          ok = false;
          break;
        }
      }
      uint8_t* pt = smem + kOffPT;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 q;
        q.x = pack_f16x2(s[8 * c + 0], s[8 * c + 1]);
        q.y = pack_f16x2(s[8 * c + 2], s[8 * c + 3]);
        q.z = pack_f16x2(s[8 * c + 4], s[8 * c + 5]);
        q.w = pack_f16x2(s[8 * c + 6], s[8 * c + 7]);
        *reinterpret_cast<uint4*>(pt + swz(k, c)) = q;
      }
      fence_async_smem();
      // per-head sums over the tile
      warp_reduce64<false>(s, lane);
      red_sum[sw * 64 + 2 * lane] = s[0];
      red_sum[sw * 64 + 2 * lane + 1] = s[1];
      softmax_sync();
      if (sw == 0 || sw == 1) {
        const int h = k;
        l_run[h] = l_run[h] * alpha_s[h] +
                   ((red_sum[h] + red_sum[64 + h]) + (red_sum[128 + h] + red_sum[192 + h]));
      }
      if (need && i >= 1) {
        // rescale O^T once PV of the previous tile has finished
        ok = wait_bar(bar(kBarODone), (i - 1) & 1, abort_flag, p.err_word);
        if (softmax_sync_or(!ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t orr[64];
          tmem_ld64(tmem + lane_base + kColO + 64 * j, orr);
#pragma unroll
          for (int h = 0; h < 64; ++h) orr[h] = __float_as_uint(__uint_as_float(orr[h]) * alpha_s[h]);
          tmem_st64(tmem + lane_base + kColO + 64 * j, orr);
        }
        tc_fence_before();
      }
      mbar_arrive(bar(kBarPFull));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && ntiles > 0) ok = wait_bar(bar(kBarODone), (ntiles - 1) & 1, abort_flag, p.err_word);
    ok = !softmax_sync_or(!ok);  // uniform; l_run is final after this barrier
    if (ok) {
      tc_fence_after();
      const int64_t tok = t;
      for (int j = 0; j < 4; ++j) {
        uint32_t orr[64];
        if (ntiles > 0) {
          tmem_ld64(tmem + lane_base + kColO + 64 * j, orr);
        } else {
#pragma unroll
          for (int h = 0; h < 64; ++h) orr[h] = 0u;
        }
        const int dv = 128 * j + k;
        if (p.num_splits == 1) {
#pragma unroll 8
          for (int h = 0; h < 64; ++h) {
            const float l = l_run[h];
            const float o = l > 0.f ? __uint_as_float(orr[h]) / l : 0.f;
            p.out[(tok * p.H + h0 + h) * kLatent + dv] = __float2bfloat16_rn(o);
          }
        } else {
          const int64_t base = (tok * p.num_splits + split) * p.H + h0;
#pragma unroll 8
          for (int h = 0; h < 64; ++h) p.ws_o[(base + h) * kLatent + dv] = __uint_as_float(orr[h]);
        }
      }
      if (sw < 2) {
        const int h = k;
        const float m = m_run[h], l = l_run[h];
        if (p.num_splits == 1) {
          p.lse[tok * p.H + h0 + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        } else {
          const int64_t base = (tok * p.num_splits + split) * p.H + h0;
          p.ws_ml[(base + h) * 2] = l > 0.f ? m : -INFINITY;
          p.ws_ml[(base + h) * 2 + 1] = l;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (*abort_flag && warp == kGatherWarp && lane == 0) {
    // let bulk copies still in flight land before the CTA exits: wait for
    // the phase of the last tile issued into each buffer (bounded)
    for (int b = 0; b < 2; ++b) {
      if (last_issued[b] < 0) continue;
      const uint32_t par = (last_issued[b] >> 1) & 1;
      uint32_t spins = 0;
      while (!mbar_test(bar(kBarRawFull + b), par) && ++spins < kSpinLimit) __nanosleep(64);
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace tc

bool tc_supported(int H) { return H % tc::kHeads == 0; }
bool tc_fp8_rows_supported(int) { return false; }

int tc_default_splits(int T, int H, int topk, int num_sms) {
  const int tiles = (topk + tc::kTile - 1) / tc::kTile;
  const int ctas_per_split = T * (H / tc::kHeads);
  int s = num_sms / max(1, ctas_per_split);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  const int per = (tiles + s - 1) / s;  // tiles of the busiest CTA
  return (tiles + per - 1) / per;       // fewest splits with that load
}

size_t tc_workspace_bytes(int T, int H, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(T) * splits * H * (kLatent + 2) * sizeof(float);
}

cudaError_t launch_merge(const float* ws_o, const float* ws_ml, int T, int S, int H, __nv_bfloat16* out, float* lse,
                         cudaStream_t stream);

cudaError_t launch_decode_tc(int fmt, const void* q_latent, const void* q_rope, const uint8_t* cache,
                             const RowSelect& sel, const int32_t* row_idx, int T, int H, int topk, float sm_scale,
                             void* out, float* lse, void* workspace, int splits, int32_t* err_word,
                             cudaStream_t stream) {
  if (fmt != 0) return cudaErrorNotSupported;
  (void)row_idx;
  tc::Params p;
  p.q_latent = static_cast<const __nv_bfloat16*>(q_latent);
  p.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
  p.cache = cache;
  p.sel = sel;
  p.T = T;
  p.H = H;
  p.topk = topk;
  p.sl2 = sm_scale * kLog2e;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.num_splits = splits;
  p.tiles_total = (topk + tc::kTile - 1) / tc::kTile;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = splits > 1 ? p.ws_o + static_cast<size_t>(T) * splits * H * kLatent : nullptr;
  p.err_word = err_word;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(splits, T, H / tc::kHeads);
  tc::decode_tc_kernel<<<grid, tc::kThreads, tc::kSmemAlloc, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  return launch_merge(p.ws_o, p.ws_ml, T, splits, H, p.out, lse, stream);
}

}  // namespace nvmla
