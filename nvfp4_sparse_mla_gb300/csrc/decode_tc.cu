// Sparse MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: "Prime Inference: Fast, Reliable Serving for Frontier
// Open Models", section "A native NVFP4 sparse-MLA decode kernel" -- for each
// query token only the rows the indexer selected are loaded, unpacked on chip
// and attended to with FP16 operands and FP32 accumulation, with no FP8
// staging buffer in GPU memory; the token's selected rows are divided among a
// cluster of cooperating CTAs whose partial results are combined through
// distributed shared memory in the same launch. "Prime Intellect unveils
// Prime Inference", section "4-bit caches open the way": item 1 (one warp
// group unpacks rows while others compute scores and accumulate), item 3
// (empty slots of the 2048-slot list contribute nothing).
//
// One cluster = one query token x 64 heads; its S CTAs take contiguous
// ranges of the token's slots, in tiles of 128 rows. Roles in a CTA:
//
//   warps 0-7  unpack: thread (row r, part h) loads the parts of its cache
//              row it needs (192 of the 352 bytes) straight into registers
//              and writes fp16 operands (E2M1 x E4M3 is exact in fp16) into
//              shared memory, 128B-swizzled: latent chunk c = 2j + h (64
//              dims) for j = 0..3 and half of the RoPE chunk. Each piece of
//              the next tile's row is requested as soon as the current tile
//              no longer needs its registers.
//   MMA issue: one softmax thread issues QK as chunk pairs land and PV as
//              soon as P^T is written; M = 128 throughout:
//                S^T[128 rows, 64 heads]   = K[128 x 576] . Q^T   (9 chunks)
//                O^T[512 dims, 64 heads]  += V^T[512 x 128] . P^T (4 blocks)
//              The latent chunks are unpacked once: a K-major 128-row x
//              64-dim chunk is byte for byte the MN-major layout of V^T for
//              those 64 value dims, so block j of PV reads chunks 2j, 2j+1.
//              Block j's completion frees chunks 2j, 2j+1 for the next tile.
//   warps 8-15 softmax: warp (lane quadrant q, head half g) owns TMEM lanes
//              32q..32q+31 (= rows) and heads 32g..32g+31. The running
//              maximum of every head stays fixed while no score exceeds it by
//              more than 2^8 (P stays below 256, safe in fp16); only a tile
//              that does (always the first) pays for the exact cross-row
//              maximum and the rescale of O^T in TMEM. Row sums accumulate per
//              thread and are reduced across rows once, at the end. P^T goes
//              to shared memory in place of the RoPE chunk, which QK no
//              longer needs.
//
// Start-up issues the dependent loads first (slot list -> block table ->
// rows of the first tile; L2 prefetch of the later tiles' rows) and converts
// the query block while they are in flight.
//
// Combine: a token's only CTA writes out / lse itself. With S CTAs, each
// writes O / l (fp16) and its per-head (m, l) to the workspace (they stay in
// L2); after one cluster barrier, CTA r weights the S partials of its share
// of the 512 value dims by l_s 2^(m_s - M) / L (M, L over the cluster) and
// writes bf16 out (rank 0 also writes lse). Distributed shared memory moves
// 64 KB per CTA more slowly than this L2 round trip does on GB300.
//
// Shared memory: query block (72 KB, later the output staging buffer) +
// latent tile (128 KB) + RoPE/P^T chunk (16 KB, later the combine weights) +
// slot list. TMEM: S^T 64 columns, O^T 4 x 64 columns.
// Every mbarrier wait is bounded: on timeout the CTA sets
// NVMLA_ERRW_WAIT_TIMEOUT, drains its MMAs and still takes part in the
// cluster barrier, so that every CTA of the cluster exits.
#include "common.cuh"

namespace nvmla {

namespace tc {

// Optional timeline instrumentation: a build with -DNVMLA_TRACE records
// %globaltimer at fixed points of each CTA's schedule into nvmla_tc_trace
// (read back with nvmla_tc_trace_read). Off by default: no code is emitted.
#ifdef NVMLA_TRACE
constexpr int kTraceCtas = 1024;
constexpr int kTracePoints = 128;
__device__ unsigned long long nvmla_tc_trace[kTraceCtas][kTracePoints];
#define NVMLA_TRACE_POINT(id)                                                                        \
  do {                                                                                               \
    const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                  \
    if (cta_ < kTraceCtas) {                                                                         \
      unsigned long long t_;                                                                         \
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t_));                                          \
      nvmla_tc_trace[cta_][(id)] = t_;                                                               \
      if ((id) == 0 || (id) == 34) nvmla_tc_trace[cta_][120 + ((id) == 34)] = clock64();             \
    }                                                                                                \
  } while (0)
#else
#define NVMLA_TRACE_POINT(id) \
  do {                        \
  } while (0)
#endif

constexpr int kTile = 128;           // rows per tile (MMA M)
constexpr int kHeads = 64;           // heads per CTA (MMA N)
constexpr int kMaxTiles = 16;        // 2048 slots
constexpr int kThreads = 512;        // 16 warps: 4 per SM sub-partition
constexpr int kUnpackThreads = 256;  // warps 0-7
constexpr int kSoftmaxWarp0 = 8;     // warps 8-15; thread 256 also issues every MMA
constexpr int kAllocWarp = 9;        // allocates and frees TMEM
constexpr int kMaxCluster = 16;      // CTAs sharing one token
constexpr int kChunkBytes = 16384;   // 128 rows x 128 bytes
constexpr int kPieces = 12;          // 16-byte pieces of a row one unpack thread holds
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;        // S^T: columns [0, 64)
constexpr uint32_t kColO = 64;       // O^T block j: columns [64 + 64 j, +64)
constexpr float kTau = 8.0f;         // rescale threshold, log2 units
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// shared memory map (bytes); the base is 1 KB aligned
constexpr int kOffQ = 0;                              // 9 x 8 KB: query, K-major; later output staging
constexpr int kOffL = kOffQ + 9 * 8192;               // 8 x 16 KB: latent tile; later the fp16 partial
constexpr int kOffR = kOffL + 8 * kChunkBytes;        // 16 KB: RoPE chunk, then P^T
constexpr int kOffSlots = kOffR + kChunkBytes;        // kMaxTiles x 128 int32
constexpr int kOffRed = kOffSlots + kMaxTiles * kTile * 4;  // 4 quadrants x 64 heads fp32
constexpr int kOffM = kOffRed + 4 * kHeads * 4;       // 64 fp32 running maxima (log2 units)
constexpr int kOffAlpha = kOffM + kHeads * 4;         // 64 fp32 rescale factors, later combine weights
constexpr int kOffMl = kOffAlpha + kHeads * 4;        // 64 x (m, l) published to the cluster
constexpr int kOffBar = kOffMl + kHeads * 8;
enum Bar {
  kBarPairFull = 0,  // 4: latent chunks 2j, 2j+1 written (8 unpack warps)
  kBarRopeFull = 4,  // RoPE chunk written (8 unpack warps)
  kBarLFree = 5,     // 4: PV block j done -> chunks 2j, 2j+1 reusable (commit)
  kBarRFree = 9,     // PV done -> RoPE/P^T chunk reusable (commit)
  kBarSFull = 10,    // QK done (commit)
  kBarPFull = 11,    // P^T written and O^T rescaled (8 softmax warps)
  kBarODone = 12,    // PV done (commit)
  kBarDrain = 13,    // every MMA finished (commit)
  kNumBars = 14
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kHeads * kLatent * 2 <= 9 * 8192, "output staging fits the query region");

struct Params {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;
  RowSelect sel;
  int T, H, topk;
  float sl2;
  __nv_bfloat16* out;
  float* lse;
  __half* ws_o16;   // [T][H / 64][S][8 head pieces][512][8 heads] partials O / l
  float* ws_ml;     // [T][H / 64][S][64][2] (m in log2 units, l)
  int num_splits;  // == cluster size
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
// try_wait that lets the hardware suspend the thread until the phase
// completes or about `hint_ns` pass, so waiting warps take no issue slots
__device__ __forceinline__ bool mbar_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity: try_wait suspends in
// hardware until the phase completes or a short internal timeout; the loop
// gives up after kWaitLimitNs of wall time, raising the CTA's abort flag and
// NVMLA_ERRW_WAIT_TIMEOUT. Also returns false once another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err_word) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_wait_hint(bar, parity, 20000)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) report_error(err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  return false;
}

// Bounded wait by a whole warp: only lane 0 polls the barrier (the other
// lanes wait at the warp barrier), and every lane gets the same outcome.
// The acquire of lane 0 covers the warp through __syncwarp's ordering.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* err_word) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, err_word);
  __syncwarp();  // orders the other lanes' later accesses after lane 0's acquire
  return __shfl_sync(0xffffffffu, ok, 0);
}

// Bounded wait without abort handling (drain paths).
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_wait_hint(bar, parity, 20000) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

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

#define NVMLA_TMEM_LD16F(taddr, r, o)                                                                         \
  asm volatile(                                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
      : "=f"(r[o + 0]), "=f"(r[o + 1]), "=f"(r[o + 2]), "=f"(r[o + 3]), "=f"(r[o + 4]), "=f"(r[o + 5]),       \
        "=f"(r[o + 6]), "=f"(r[o + 7]), "=f"(r[o + 8]), "=f"(r[o + 9]), "=f"(r[o + 10]), "=f"(r[o + 11]),     \
        "=f"(r[o + 12]), "=f"(r[o + 13]), "=f"(r[o + 14]), "=f"(r[o + 15])                                    \
      : "r"(taddr))

// 64 consecutive TMEM columns of this thread's lane, as fp32
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&r)[64]) {
  NVMLA_TMEM_LD16F(taddr + 0, r, 0);
  NVMLA_TMEM_LD16F(taddr + 16, r, 16);
  NVMLA_TMEM_LD16F(taddr + 32, r, 32);
  NVMLA_TMEM_LD16F(taddr + 48, r, 48);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

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

// 32 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&r)[32]) {
  NVMLA_TMEM_LD16F(taddr + 0, r, 0);
  NVMLA_TMEM_LD16F(taddr + 16, r, 16);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  NVMLA_TMEM_LD16(taddr + 0, r, 0);
  NVMLA_TMEM_LD16(taddr + 16, r, 16);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// named barrier among the eight softmax warps (id 1); the _or form returns
// the OR of a predicate over the group (used to make the outcome of a
// bounded wait, or a data-dependent branch, uniform)
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool softmax_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// one arrival per warp once every lane is past this point
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// swizzled byte offset of 16-byte chunk c of row r inside a 128B-swizzled
// region (rows of 128 bytes, 8-row atoms of 1 KB)
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// ---- cluster: rank, and a barrier over every thread of every CTA with
// release / acquire semantics at cluster scope
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// L2-only loads (the data was written by other CTAs of the cluster)
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float2 ldg_cg_f2(const float* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}

// fire-and-forget prefetch of a row into L2 (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16 E2M1 codes (8 bytes) times one scale -> two 16-byte fp16 chunks
__device__ __forceinline__ void unpack16(uint32_t lo, uint32_t hi, uint32_t s2, uint4& a, uint4& b) {
  uint32_t h[4];
  e2m1x8_to_f16x8(lo, h);
  a = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
  e2m1x8_to_f16x8(hi, h);
  b = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
}

__device__ __forceinline__ void zero_row(uint8_t* dst_base, int r) {
#pragma unroll
  for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst_base + swz(r, c)) = make_uint4(0, 0, 0, 0);
}

// transposing butterfly: 32 values per lane -> lane L holds the reduction
// over the warp's 32 lanes of value L (in v[0])
template <bool kMax>
__device__ __forceinline__ void warp_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int n = 16 >> step;  // values kept after this step
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

// The 16-byte pieces of a 352-byte row that unpack thread part h holds:
// codes of latent chunks h, h+2, h+4, h+6 (pieces 2c, 2c+1), both scale
// pieces (16, 17) and its half of the RoPE bytes (18 + 2h, 19 + 2h).
__device__ __forceinline__ int piece_of(int n, int h) {
  return n < 8 ? 2 * (2 * (n >> 1) + h) + (n & 1) : (n < 10 ? 16 + (n - 8) : 18 + 2 * h + (n - 10));
}

// latent chunk c = 2j + h of one row (64 dims) from the held pieces
__device__ __forceinline__ void write_latent(const uint4 (&raw)[kPieces], int j, int h, uint8_t* chunk, int r) {
  const uint4 c0 = raw[2 * j], c1 = raw[2 * j + 1];
  const int c = 2 * j + h;
  const uint4 sp = raw[8 + (c >> 2)];  // scale piece: groups 16*(c>>2) .. +15
  const uint32_t sw = ((c & 3) == 0) ? sp.x : ((c & 3) == 1) ? sp.y : ((c & 3) == 2) ? sp.z : sp.w;
  uint4 a, b;
  unpack16(c0.x, c0.y, e4m3_to_f16x2_bcast(sw & 0xffu), a, b);
  *reinterpret_cast<uint4*>(chunk + swz(r, 0)) = a;
  *reinterpret_cast<uint4*>(chunk + swz(r, 1)) = b;
  unpack16(c0.z, c0.w, e4m3_to_f16x2_bcast((sw >> 8) & 0xffu), a, b);
  *reinterpret_cast<uint4*>(chunk + swz(r, 2)) = a;
  *reinterpret_cast<uint4*>(chunk + swz(r, 3)) = b;
  unpack16(c1.x, c1.y, e4m3_to_f16x2_bcast((sw >> 16) & 0xffu), a, b);
  *reinterpret_cast<uint4*>(chunk + swz(r, 4)) = a;
  *reinterpret_cast<uint4*>(chunk + swz(r, 5)) = b;
  unpack16(c1.z, c1.w, e4m3_to_f16x2_bcast(sw >> 24), a, b);
  *reinterpret_cast<uint4*>(chunk + swz(r, 6)) = a;
  *reinterpret_cast<uint4*>(chunk + swz(r, 7)) = b;
}

// RoPE values 32h .. 32h + 31 of one row
__device__ __forceinline__ void write_rope(const uint4 (&raw)[kPieces], int h, uint8_t* chunk, int r) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = raw[10 + q];
    uint4 a, b;
    e4m3x4_to_f16x4(v.x, a.x, a.y);
    e4m3x4_to_f16x4(v.y, a.z, a.w);
    e4m3x4_to_f16x4(v.z, b.x, b.y);
    e4m3x4_to_f16x4(v.w, b.z, b.w);
    *reinterpret_cast<uint4*>(chunk + swz(r, 4 * h + 2 * q)) = a;
    *reinterpret_cast<uint4*>(chunk + swz(r, 4 * h + 2 * q + 1)) = b;
  }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ int32_t ldg_nc_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Held pieces n0 .. n1-1 of the row in slot `slot` (nothing for a masked
// slot). The loads are volatile so that they are issued here, as soon as the
// registers are free, and not sunk next to their first use.
__device__ __forceinline__ void load_pieces(const uint8_t* cache, int32_t slot, int h, uint4 (&raw)[kPieces], int n0,
                                            int n1) {
  if (slot < 0) return;
  const uint8_t* row = cache + static_cast<int64_t>(slot) * kRowBytes;
#pragma unroll
  for (int n = 0; n < kPieces; ++n)
    if (n >= n0 && n < n1) raw[n] = ldg_nc_v4(row + 16 * piece_of(n, h));
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, h0 = blockIdx.z * kHeads;
  const int S = p.num_splits;
  const uint32_t rank = cluster_rank();  // the CTA's split: clusters span blockIdx.x

  int32_t* slots = reinterpret_cast<int32_t*>(smem + kOffSlots);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* m_run = reinterpret_cast<float*>(smem + kOffM);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* ml_pub = reinterpret_cast<float*>(smem + kOffMl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return sbase + kOffBar + 8 * i; };

  const int tile_lo = (static_cast<int>(rank) * p.tiles_total) / S;
  const int tile_hi = ((static_cast<int>(rank) + 1) * p.tiles_total) / S;
  const int kbeg = tile_lo * kTile;
  const int kend = min(tile_hi * kTile, p.topk);
  const int nkeys = max(0, kend - kbeg);
  const int ntiles = (nkeys + kTile - 1) / kTile;  // <= kMaxTiles (host check)

  if (tid == 0) NVMLA_TRACE_POINT(40);

  // sequence facts of this token
  const int32_t seq = p.sel.q_seq_idx ? __ldg(p.sel.q_seq_idx + t) : 0;
  const int32_t* bt_row = p.sel.block_table + static_cast<int64_t>(seq) * p.sel.max_pages;
  const int32_t* idx_row = p.sel.topk_idx + static_cast<int64_t>(t) * p.topk;
  // slot of position pos (-1 for padding or a bad entry, which is reported
  // when `report`)
  auto slot_of_pos = [&](int32_t pos, int64_t limit, bool report) -> int32_t {
    if (pos == -1) return -1;
    if (pos < 0 || pos >= limit) {
      if (report) report_error(p.err_word, NVMLA_ERRW_BAD_INDEX, 1);
      return -1;
    }
    const int64_t page = __ldg(bt_row + (pos >> 6));
    const int64_t s = page * kPage + (pos & 63);
    if (page < 0 || s >= p.sel.num_slots) {
      if (report) report_error(p.err_word, NVMLA_ERRW_BAD_SLOT, 1);
      return -1;
    }
    return static_cast<int32_t>(s);
  };

  // ---- start-up: the dependent loads first (slot list, block table, rows),
  // the query block while they are in flight
  const bool is_unpack = tid < kUnpackThreads;
  const int ur = tid & 127, uh = (tid >> 7) & 1;  // unpack threads: row, part
  const int sj = tid - kUnpackThreads;            // softmax threads: 0..255
  uint4 raw[kPieces];
  int32_t slot0 = -1;
  int32_t pos0 = -1;
  constexpr int kLaterPer = kMaxTiles / 2;  // later tiles per softmax thread
  int32_t posl[kLaterPer];
  if (is_unpack) {
    if (kbeg + ur < kend) pos0 = ldg_nc_s32(idx_row + kbeg + ur);
  } else {
    // softmax thread sj handles row sj % 128 of tiles 1 + sj / 128 + 2m
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + (sj >> 7) + 2 * m;
      const int key = kbeg + i * kTile + (sj & 127);
      posl[m] = (i < ntiles && key < kend) ? ldg_nc_s32(idx_row + key) : -1;
    }
  }
  constexpr int kQPer = kHeads * 72 / kThreads;  // 9 query pieces per thread
  uint4 qv[kQPer];
#pragma unroll
  for (int n = 0; n < kQPer; ++n) {
    const int i = tid + kThreads * n;
    const int h = i / 72, j = i % 72;
    const int64_t qh = static_cast<int64_t>(t) * p.H + h0 + h;
    qv[n] = j < 64 ? ldg_nc_v4(p.q_latent + qh * kLatent + 8 * j) : ldg_nc_v4(p.q_rope + qh * kRope + 8 * (j - 64));
  }
  int64_t limit = static_cast<int64_t>(p.sel.max_pages) * kPage;
  if (p.sel.seq_lens) {
    const int64_t L = __ldg(p.sel.seq_lens + seq);
    limit = L < limit ? L : limit;
  }
  const bool report = blockIdx.z == 0;  // one head block reports bad entries
  if (is_unpack) {
    if (ntiles > 0 && kbeg + ur < kend) slot0 = slot_of_pos(pos0, limit, report && uh == 0);
    load_pieces(p.cache, slot0, uh, raw, 0, kPieces);
    if (uh == 0) slots[ur] = slot0;
  } else {
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + (sj >> 7) + 2 * m;
      if (i < ntiles) {
        const int32_t s = slot_of_pos(posl[m], limit, report);
        slots[i * kTile + (sj & 127)] = s;
        if (s >= 0) prefetch_l2(p.cache + static_cast<int64_t>(s) * kRowBytes, kRowBytes);
      }
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(41);

  // ---- setup
  if (tid == kThreads - 1) {
    for (int j = 0; j < 4; ++j) {
      mbar_init(bar(kBarPairFull + j), 8);
      mbar_init(bar(kBarLFree + j), 1);
    }
    mbar_init(bar(kBarRopeFull), 8);
    mbar_init(bar(kBarRFree), 1);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPFull), 8);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = (sbase & 1023u) ? 1 : 0;  // swizzled operands need a 1 KB aligned base
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kHeads) m_run[tid] = -INFINITY;
  if (warp == kAllocWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // query block -> fp16, K-major 128B-swizzled (all 16 warps)
#pragma unroll
  for (int n = 0; n < kQPer; ++n) {
    const int i = tid + kThreads * n;
    const int h = i / 72, j = i % 72, c = j >> 3, q = j & 7;
    const uint32_t w[4] = {qv[n].x, qv[n].y, qv[n].z, qv[n].w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(bf16_bits_to_f32(w[e] & 0xffffu), bf16_bits_to_f32(w[e] >> 16));
    *reinterpret_cast<uint4*>(smem + kOffQ + c * 8192 + swz(h, q)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (*abort_flag && tid == 0) report_error(p.err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  if (tid == 0) NVMLA_TRACE_POINT(0);

  // roles; the softmax group's epilogue ends with the (m, l) of every head
  // published in ml_pub
  const int sw = warp - kSoftmaxWarp0;       // softmax warp 0..7
  const int quad = sw & 3, hh = sw >> 2;     // TMEM lane quadrant, head half
  const int hb = hh * 32;                    // first head of this thread
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  bool ok = true;
  if (is_unpack) {
    // ------------------------------------------------------------ unpack
    ok = *abort_flag == 0;
    int32_t cur_slot = slot0;
    for (int i = 0; i < ntiles && ok; ++i) {
      const bool valid = cur_slot >= 0;
      const int32_t nxt_slot = (i + 1 < ntiles) ? slots[(i + 1) * kTile + ur] : -1;
      if (tid == 0 && i < 2) {
        uint32_t x = raw[0].x ^ raw[11].w;  // first use: the pieces have arrived
        asm volatile("" ::"r"(x));
        NVMLA_TRACE_POINT(44 + i);
      }
      for (int j = 0; j < 4 && ok; ++j) {
        if (i >= 1) ok = wait_bar_warp(bar(kBarLFree + j), (i - 1) & 1, abort_flag, p.err_word);
        if (!ok) break;
        uint8_t* chunk = smem + kOffL + (2 * j + uh) * kChunkBytes;
        if (valid) {
          write_latent(raw, j, uh, chunk, ur);
        } else {
          zero_row(chunk, ur);
        }
        fence_async_smem();
        warp_arrive(bar(kBarPairFull + j), lane);
        // the registers of this pair (and of a scale piece once its last
        // pair is written) now take the next tile's row
        load_pieces(p.cache, nxt_slot, uh, raw, 2 * j, 2 * j + 2);
        if (j == 1) load_pieces(p.cache, nxt_slot, uh, raw, 8, 9);
        if (j == 3) load_pieces(p.cache, nxt_slot, uh, raw, 9, 10);
      }
      if (ok && i >= 1) ok = wait_bar_warp(bar(kBarRFree), (i - 1) & 1, abort_flag, p.err_word);
      if (!ok) break;
      uint8_t* rc = smem + kOffR;
      if (valid) {
        write_rope(raw, uh, rc, ur);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(rc + swz(ur, 4 * uh + c)) = make_uint4(0, 0, 0, 0);
      }
      fence_async_smem();
      warp_arrive(bar(kBarRopeFull), lane);
      load_pieces(p.cache, nxt_slot, uh, raw, 10, 12);
      cur_slot = nxt_slot;
      if (tid == 0 && i < 4) NVMLA_TRACE_POINT(14 + i);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int k = quad * 32 + lane;  // row of this thread
    const bool issuer = tid == kUnpackThreads;
    constexpr uint32_t idesc_qk = idesc_f16(false, false);
    constexpr uint32_t idesc_pv = idesc_f16(true, true);
    const uint32_t lb = sbase + kOffL, rb = sbase + kOffR, qb = sbase + kOffQ;
    // QK of one tile, issued by one thread: latent chunk pairs as they land,
    // then the RoPE chunk
    auto issue_qk = [&](int i) -> bool {
      const uint32_t par = i & 1;
      for (int j = 0; j < 4; ++j) {
        if (!wait_bar(bar(kBarPairFull + j), par, abort_flag, p.err_word)) return false;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * j + cc;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16(tmem + kColS, sdesc(lb + c * kChunkBytes + 32 * ks, 16, 1024),
                    sdesc(qb + c * 8192 + 32 * ks, 16, 1024), idesc_qk, (c | ks) != 0);
        }
      }
      if (!wait_bar(bar(kBarRopeFull), par, abort_flag, p.err_word)) return false;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_f16(tmem + kColS, sdesc(rb + 32 * ks, 16, 1024), sdesc(qb + 8 * 8192 + 32 * ks, 16, 1024), idesc_qk, 1);
      mma_commit(bar(kBarSFull));
      if (i < 4) NVMLA_TRACE_POINT(5 + 2 * i);
      return true;
    };
    // PV of one tile: block j reads latent chunks 2j, 2j+1 as V^T and P^T
    // from R; its completion frees those chunks for the next tile
    auto issue_pv = [&](int i) -> bool {
      if (!wait_bar(bar(kBarPFull), i & 1, abort_flag, p.err_word)) return false;
      tc_fence_after();
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_f16(tmem + kColO + 64 * j, sdesc(lb + 2 * j * kChunkBytes + 2048 * ks, kChunkBytes, 1024),
                  sdesc(rb + 2048 * ks, 8192, 1024), idesc_pv, !(i == 0 && ks == 0));
        mma_commit(bar(kBarLFree + j));
      }
      mma_commit(bar(kBarRFree));
      mma_commit(bar(kBarODone));
      if (i < 4) NVMLA_TRACE_POINT(6 + 2 * i);
      return true;
    };

    float lp[32];  // this row's share of its heads' sums
#pragma unroll
    for (int h = 0; h < 32; ++h) lp[h] = 0.f;
    ok = !softmax_sync_or(*abort_flag != 0);
    // the issuer's outcome is made uniform across its warp before any
    // warp-collective operation
    auto issued = [&](bool mine) -> bool { return __shfl_sync(0xffffffffu, mine, 0); };
    for (int i = 0; i < ntiles && ok; ++i) {
      // a failed PV issue of the previous tile left the abort flag raised;
      // the issuer then issues nothing more, and the OR below ends the loop
      // for the whole group at once
      bool okq = true;
      if (issuer) okq = *abort_flag == 0 && issue_qk(i);
      ok = issued(okq);
      if (ok) ok = wait_bar_warp(bar(kBarSFull), i & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(21 + 3 * i);
      const bool valid = slots[i * kTile + k] >= 0;
      float s[32];
      tmem_ld32f(tmem + lane_base + kColS + hb, s);
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
      // does any score exceed its head's running maximum by more than 2^tau?
      float excess = -INFINITY;
      if (valid) {
#pragma unroll
        for (int h = 0; h < 32; ++h) excess = fmaxf(excess, s[h] - m_run[hb + h]);
      }
      const bool slow = softmax_sync_or(excess > kTau);
      if (slow) {
        // exact per-head maximum of this tile (destroys s; reloaded below)
        warp_reduce32<true>(s, lane);
        red[quad * 64 + hb + lane] = s[0];
        softmax_sync();
        if (quad == 0) {
          const int h = hb + lane;
          const float mt = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
          const float mo = m_run[h];
          const float mn = fmaxf(mo, mt);
          alpha_s[h] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
          m_run[h] = mn;
        }
        softmax_sync();
#pragma unroll
        for (int h = 0; h < 32; ++h) lp[h] *= alpha_s[hb + h];
        if (i >= 1) {
          // O^T holds the finished PV of the earlier tiles (QK of this tile
          // could only start after the last of them); 16 columns at a time
#pragma unroll 1
          for (int jq = 0; jq < 8; ++jq) {
            const uint32_t col = kColO + 64 * (jq >> 1) + hb + 16 * (jq & 1);
            uint32_t orr[16];
            NVMLA_TMEM_LD16(tmem + lane_base + col, orr, 0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const float* al = alpha_s + hb + 16 * (jq & 1);
#pragma unroll
            for (int e = 0; e < 16; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * al[e]);
            NVMLA_TMEM_ST16(tmem + lane_base + col, orr, 0);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tmem_ld32f(tmem + lane_base + kColS + hb, s);
#pragma unroll
        for (int h = 0; h < 32; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
      }
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(22 + 3 * i);
      // P = 2^(s - m); masked rows give 0
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float pv = valid ? ex2(s[h] - m_run[hb + h]) : 0.f;
        s[h] = pv;
        lp[h] += pv;
      }
      // P^T row (this thread's 32 heads) -> the RoPE chunk's place (QK of
      // this tile is complete)
      uint8_t* pt = smem + kOffR;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint4 q;
        q.x = pack_f16x2(s[8 * cc + 0], s[8 * cc + 1]);
        q.y = pack_f16x2(s[8 * cc + 2], s[8 * cc + 3]);
        q.z = pack_f16x2(s[8 * cc + 4], s[8 * cc + 5]);
        q.w = pack_f16x2(s[8 * cc + 6], s[8 * cc + 7]);
        *reinterpret_cast<uint4*>(pt + swz(k, 4 * hh + cc)) = q;
      }
      fence_async_smem();
      tc_fence_before();
      warp_arrive(bar(kBarPFull), lane);
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(23 + 3 * i);
      if (issuer) issue_pv(i);
    }
    // ------------------------------------------------------------ row sums
    if (ok && ntiles > 0) ok = wait_bar_warp(bar(kBarODone), (ntiles - 1) & 1, abort_flag, p.err_word);
    ok = !softmax_sync_or(!ok);
    tc_fence_after();
    if (tid == 256) NVMLA_TRACE_POINT(33);
    warp_reduce32<false>(lp, lane);
    red[quad * 64 + hb + lane] = lp[0];
    softmax_sync();
    if (quad == 0) {
      const int h = hb + lane;
      const float l = (red[h] + red[64 + h]) + (red[128 + h] + red[192 + h]);
      const bool live = ok && l > 0.f;
      ml_pub[2 * h] = live ? m_run[h] : -INFINITY;
      ml_pub[2 * h + 1] = live ? l : 0.f;
      alpha_s[h] = live ? 1.f / l : 0.f;
    }
    if (issuer) {
      // every MMA issued has finished once this commit lands
      mma_commit(bar(kBarDrain));
      wait_bar_drain(bar(kBarDrain), 0);
    }
  }

  // ------------------------------------------------------------ combine
  if (S == 1) {
    // the token's only CTA: O / l as bf16 [64 heads][512 dims] staged in the
    // query block's place, then 16-byte stores of out
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + kOffQ);
    __syncthreads();  // alpha_s (1 / l) of every head is written
    if (!is_unpack) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const int dv = 128 * j + quad * 32 + lane;
        uint32_t o[32];
        if (ok && ntiles > 0) {
          tmem_ld32(tmem + lane_base + kColO + 64 * j + hb, o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
          stage[(hb + e) * kLatent + dv] = __float2bfloat16_rn(__uint_as_float(o[e]) * alpha_s[hb + e]);
      }
      tc_fence_before();
      if (quad == 0) {
        const int h = hb + lane;
        const float m = ml_pub[2 * h], l = ml_pub[2 * h + 1];
        p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      }
    }
    __syncthreads();
    if (warp == kAllocWarp) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
#pragma unroll
    for (int u = 0; u < kHeads * (kLatent / 8) / kThreads; ++u) {
      const int pc = tid + kThreads * u, h = pc >> 6, g = pc & 63;
      const uint4 v = *reinterpret_cast<const uint4*>(stage + h * kLatent + 8 * g);
      *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.H + h0 + h) * kLatent + 8 * g) = v;
    }
  } else {
    // S CTAs: each writes O / l (fp16, 8-head pieces x 512 dims) and its (m, l) to
    // the workspace; after a cluster barrier CTA `rank` combines the S
    // partials of its share [dv0, dv0 + ndv) of the value dims
    const int64_t cbase = (static_cast<int64_t>(t) * gridDim.z + blockIdx.z) * S;  // first split of this cluster
    __syncthreads();  // alpha_s (1 / l) of every head is written
    if (!is_unpack) {
      __half* wo = p.ws_o16 + (cbase + rank) * (kLatent * kHeads);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const int dv = 128 * j + quad * 32 + lane;
        uint32_t o[32];
        if (ok && ntiles > 0) {
          tmem_ld32(tmem + lane_base + kColO + 64 * j + hb, o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int hl = 8 * cc + 2 * e;
            w4[e] = pack_f16x2(__uint_as_float(o[hl]) * alpha_s[hb + hl],
                               __uint_as_float(o[hl + 1]) * alpha_s[hb + hl + 1]);
          }
          // piece-major [8 head pieces][512 dims][8 heads]: a warp's lanes
          // (consecutive dims) store 512 contiguous bytes
          *reinterpret_cast<uint4*>(wo + ((4 * hh + cc) * kLatent + dv) * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      tc_fence_before();
      if (quad == 0) {
        const int h = hb + lane;
        *reinterpret_cast<float2*>(p.ws_ml + ((cbase + rank) * kHeads + h) * 2) =
            make_float2(ml_pub[2 * h], ml_pub[2 * h + 1]);
      }
    }
    // release / acquire at cluster scope: every partial of the cluster is
    // visible to every CTA of it
    cluster_sync_all();
    if (tid == 256) NVMLA_TRACE_POINT(35);
    if (warp == kAllocWarp) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    const int dv0 = 8 * ((static_cast<int>(rank) * (kLatent / 8)) / S);
    const int ndv = 8 * (((static_cast<int>(rank) + 1) * (kLatent / 8)) / S) - dv0;
    const int nitems = ndv * 8;  // (dim, 8-head piece)
    const __half* wo0 = p.ws_o16 + cbase * (kLatent * kHeads);
    uint4 v[8];
    auto load_batch = [&](int item, int s0) {
      const int piece = item / ndv, dl = item - piece * ndv;
      const int64_t off = static_cast<int64_t>(piece * kLatent + dv0 + dl) * 8;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (s0 + u < S) v[u] = ldg_cg_v4(wo0 + static_cast<int64_t>(s0 + u) * (kLatent * kHeads) + off);
    };
    // this thread's first partials are requested before the weights are known
    if (tid < nitems) load_batch(tid, 0);
    float* coef = reinterpret_cast<float*>(smem + kOffR);  // [S][64] combine weights
    if (tid < kHeads) {
      const int h = tid;
      float2 ml[kMaxCluster];
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s)
        if (s < S) ml[s] = ldg_cg_f2(p.ws_ml + ((cbase + s) * kHeads + h) * 2);
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s)
        if (s < S) M = fmaxf(M, ml[s].x);
      float L = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) {
        if (s < S) {
          const float w = ml[s].y > 0.f ? ml[s].y * ex2(ml[s].x - M) : 0.f;
          ml[s].y = w;
          L += w;
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s)
        if (s < S) coef[s * kHeads + h] = ml[s].y * inv;
      if (rank == 0) p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    if (tid == 256) NVMLA_TRACE_POINT(36);
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + kOffQ);  // [64 heads][ndv]
    for (int it = tid; it < nitems; it += kThreads) {
      const int piece = it / ndv, dl = it - piece * ndv;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int s0 = 0; s0 < S; s0 += 8) {
        if (s0 > 0 || it != tid) load_batch(it, s0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (s0 + u < S) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            const float* c = coef + (s0 + u) * kHeads + 8 * piece;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
              acc[2 * e] += c[2 * e] * f.x;
              acc[2 * e + 1] += c[2 * e + 1] * f.y;
            }
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) stage[(8 * piece + e) * ndv + dl] = __float2bfloat16_rn(acc[e]);
    }
    __syncthreads();
    if (tid == 256) NVMLA_TRACE_POINT(38);
    const int per_head = ndv / 8;
    for (int pc = tid; pc < kHeads * per_head; pc += kThreads) {
      const int h = pc / per_head, g = pc - h * per_head;
      const uint4 w = *reinterpret_cast<const uint4*>(stage + h * ndv + 8 * g);
      *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.H + h0 + h) * kLatent + dv0 + 8 * g) = w;
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(34);
}

}  // namespace tc

bool tc_supported(int H) { return H % tc::kHeads == 0; }
bool tc_fp8_rows_supported(int) { return false; }

namespace {

// Per-device launch setup of the kernel: its shared-memory size, and for
// every cluster size S how many clusters of S CTAs can be resident at once
// (0: S cannot be launched).
struct TcDevice {
  bool ready = false;
  int max_active[tc::kMaxCluster + 1] = {0};
};
TcDevice g_tc_dev[64];

int tc_prepare() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  TcDevice& d = g_tc_dev[dev];
  if (d.ready) return dev;
  cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::kSmemBytes);
  if (e != cudaSuccess) return -1;
  const bool non_portable =
      cudaFuncSetAttribute(tc::decode_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  for (int s = 1; s <= tc::kMaxCluster; ++s) {
    d.max_active[s] = 0;
    if (s > 8 && !non_portable) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s, 1, 1);
    cfg.blockDim = dim3(tc::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tc::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = s;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc::decode_tc_kernel, &cfg) == cudaSuccess) d.max_active[s] = n;
  }
  cudaGetLastError();  // a refused cluster size leaves no sticky error
  d.ready = true;
  return dev;
}

}  // namespace

int tc_max_splits() {
  const int dev = tc_prepare();
  if (dev < 0) return 8;  // no device: the portable cluster size
  int s = tc::kMaxCluster;
  while (s > 1 && g_tc_dev[dev].max_active[s] < 1) --s;
  return s;
}

// Key splits per token: enough CTAs to fill the SMs, at most as many
// clusters as can be resident at once, then the fewest splits that give the
// busiest CTA the same number of tiles.
int tc_default_splits(int T, int H, int topk, int num_sms) {
  const int tiles = (topk + tc::kTile - 1) / tc::kTile;
  const int clusters = T * (H / tc::kHeads);
  int s = num_sms / max(1, clusters);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  const int dev = tc_prepare();
  if (dev < 0) {
    if (s > 8) s = 8;
  } else {
    while (s > 1 && g_tc_dev[dev].max_active[s] < clusters) --s;
  }
  const int per = (tiles + s - 1) / s;  // tiles of the busiest CTA
  return (tiles + per - 1) / per;       // fewest splits with that load
}

size_t tc_workspace_bytes(int T, int H, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(T) * (H / tc::kHeads) * splits *
         (tc::kHeads * kLatent * sizeof(__half) + tc::kHeads * 2 * sizeof(float));
}

cudaError_t launch_decode_tc(int fmt, const void* q_latent, const void* q_rope, const uint8_t* cache,
                             const RowSelect& sel, const int32_t* row_idx, int T, int H, int topk, float sm_scale,
                             void* out, float* lse, void* workspace, int splits, int32_t* err_word,
                             cudaStream_t stream) {
  if (fmt != 0) return cudaErrorNotSupported;
  (void)row_idx;
  if (tc_prepare() < 0) return cudaErrorInvalidDevice;
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
  p.ws_o16 = static_cast<__half*>(workspace);
  p.ws_ml = splits > 1 ? reinterpret_cast<float*>(p.ws_o16 + static_cast<size_t>(T) * (H / tc::kHeads) * splits *
                                                                 tc::kHeads * kLatent)
                       : nullptr;
  p.num_splits = splits;
  p.tiles_total = (topk + tc::kTile - 1) / tc::kTile;
  p.err_word = err_word;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, T, H / tc::kHeads);
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = splits;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc::decode_tc_kernel, p);
}

}  // namespace nvmla

#ifdef NVMLA_TRACE
extern "C" int nvmla_tc_trace_read(void* host_dst, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(host_dst, nvmla::tc::nvmla_tc_trace, bytes));
}
#endif
