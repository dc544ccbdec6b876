// Sparse MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: "Prime Inference: Fast, Reliable Serving for Frontier
// Open Models", section "A native NVFP4 sparse-MLA decode kernel" -- for each
// query token only the rows the indexer selected are loaded, unpacked on chip
// and attended to with FP16 operands and FP32 accumulation, with no FP8
// staging buffer in GPU memory; the token's selected rows are divided among a
// cluster of cooperating CTAs whose partial results are combined in the same
// launch. "Prime Intellect unveils Prime Inference", section "4-bit caches
// open the way": item 1 (one warp group unpacks rows while others compute
// scores and accumulate), item 3 (empty slots of the 2048-slot list
// contribute nothing).
//
// One cluster = one query token x 64 heads; its S CTAs take contiguous
// ranges of the token's slots, in tiles of 128 rows. Both contractions run as
// tcgen05.mma kind::f16 (M = 128, N = 64, K = 16) in swap-AB orientation, the
// 64 heads being N:
//   S^T[128 rows, 64 heads]  = K[128 x 576] . Q^T     A: K in TMEM, B: Q in shared memory
//   O^T[512 dims, 64 heads] += V^T[512 x 128] . P^T   A: V^T, B: P^T, both in shared memory
// TMEM (512 columns): S^T in columns 0-63, O^T in 64-319 (4 blocks of 128
// dims), and a ring of 6 K slots of 32 columns (64 fp16 dims x 128 rows) in
// 320-511. A tile's K is 9 chunks of 64 dims (8 latent, 1 RoPE): QK batch A
// takes chunk uses 0-5 in slots 0-5, batch B uses 6-8 in slots 0-2, once
// batch A's MMAs have read them.
//
// Roles in a CTA (18 warps, 96 registers a thread):
//
//   warps 0-7   unpack: thread (row r, half h) holds the half of its cache
//               row it converts -- the code bytes of latent dims
//               256h..256h+255 and their 16 scale bytes, half 0 also the
//               RoPE bytes -- and writes fp16 values (E2M1 x E4M3 is exact in
//               fp16) into the K ring with tcgen05.st. Each piece of the next
//               tile's row is requested as soon as the current tile no longer
//               needs its registers.
//   warps 8-15  softmax: warp (lane quadrant q, head half g) owns TMEM lanes
//               32q..32q+31 (= rows) and heads 32g..32g+31. It copies the
//               latent chunks out of the K ring into the V tile in shared
//               memory (128B-swizzled: a K-major 128-row chunk of 64 dims is
//               the MN-major layout of V^T for those dims), reads S^T and
//               writes P^T to shared memory. A head's running maximum starts,
//               on the first tile, at the largest score of rows 0, 32, 64 and
//               96, and stays fixed while no score exceeds it by more than
//               2^15 (P stays below 2^15, safe in fp16); only a tile that
//               does pays for the exact cross-row maximum and the rescale of
//               O^T in TMEM. Row sums accumulate per thread and are reduced
//               across rows once, at the end.
//   warp 16     issues the QK MMAs (one thread); allocates and frees TMEM.
//   warp 17     issues the PV MMAs (one thread). PV block j reads V chunks j
//               and j + 4 (dims 64j.. and 256 + 64j..). Blocks 0-1 commit on
//               their own, so the next tile's V copy into chunks 0, 1, 4 and
//               5 starts while blocks 2-3 run.
//
// The next tile's unpack and QK overlap the current tile's softmax and PV.
// The FP8-row variant loads 576-byte E4M3 rows and converts them without
// scales; everything from the K ring on is shared.
//
// Start-up issues the dependent loads first (slot list and sequence ->
// block table and sequence length -> rows of the first tile, three levels;
// the rows are requested before the sequence length arrives and ignored if
// they lie past it) and converts the query block (bf16 -> fp16) while they
// are in flight; the later tiles' rows are prefetched into L2 after it.
//
// Combine: a token's only CTA writes out / lse itself. With S CTAs, each
// normalises its O^T block by block as PV finishes (O / l, fp16, in the
// freed latent chunk) and stores it to the workspace with TMA bulk copies,
// plus its per-head (m, l); after one cluster barrier CTA r loads its share
// of the 512 value dims from all S partials (TMA bulk loads into the freed
// query block), weights them by l_s 2^(m_s - M) / L (M, L over the cluster)
// and writes bf16 out (rank 0 also writes lse). On GB300 this round trip
// through L2 moves a CTA's 64 KB partial faster than distributed shared
// memory does.
//
// Shared memory: query block (72 KB) + slot list (8 KB), later the combine's
// receive buffer; V tile (128 KB), later the partial staging; P^T (16 KB),
// later the combine weights.
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
    }                                                                                                \
  } while (0)
// the same, once the 32-bit value v is available
#define NVMLA_TRACE_AFTER(id, v)                                                                     \
  do {                                                                                               \
    const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                  \
    if (cta_ < kTraceCtas) {                                                                         \
      unsigned long long t_;                                                                         \
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t_) : "r"(v));                                \
      nvmla_tc_trace[cta_][(id)] = t_;                                                               \
    }                                                                                                \
  } while (0)
#else
#define NVMLA_TRACE_POINT(id) \
  do {                        \
  } while (0)
#define NVMLA_TRACE_AFTER(id, v) \
  do {                           \
  } while (0)
#endif

constexpr int kTile = 128;              // rows per tile (MMA M)
constexpr int kHeads = 64;              // heads per CTA (MMA N)
constexpr int kMaxTiles = 16;           // 2048 slots
constexpr int kUnpackThreads = 256;     // warps 0-7
constexpr int kSoftmax0 = 256;          // warps 8-15: threads 256..511
constexpr int kQkWarp = 16;             // issues the QK MMAs; allocates TMEM
constexpr int kPvWarp = 17;             // issues the PV MMAs
constexpr int kThreads = 576;           // 18 warps
constexpr int kMaxCluster = 16;         // CTAs sharing one token
constexpr int kChunkBytes = 16384;      // 128 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;           // S^T: columns [0, 64)
constexpr uint32_t kColO = 64;          // O^T block j: columns [64 + 64 j, +64)
constexpr uint32_t kColK = 320;         // K ring: kRing slots of 32 columns (64 fp16 dims x 128 rows)
constexpr int kRing = 6;                // a tile's 9 K chunks: batch A = chunk uses 0-5 in slots 0-5,
                                        // batch B = uses 6-8 in slots 0-2
static_assert(kColK + 32 * kRing <= kTmemCols, "TMEM budget");
constexpr float kTau = 15.0f;           // rescale threshold, log2 units: P < 2^15 fits fp16
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kPartBytes = kLatent * kHeads * 2;  // one CTA's fp16 partial: 64 KB
constexpr int kMlBytes = kHeads * 8;              // its per-head (m, l)

// shared memory map (bytes); the base is 1 KB aligned
constexpr int kOffQ = 0;                               // 9 x 8 KB: query, K-major
constexpr int kOffSlots = kOffQ + 9 * 8192;            // kMaxTiles x 128 int32
constexpr int kRxBytes = kOffSlots + kMaxTiles * kTile * 4;  // query + slots: combine receive buffer
constexpr int kOffL = kRxBytes;                        // 8 x 16 KB: V (latent) tile, later partial staging
constexpr int kOffR = kOffL + 8 * kChunkBytes;         // 16 KB: P^T, then the combine weights
constexpr int kOffRed = kOffR + kChunkBytes;           // 4 quadrants x 64 heads fp32
constexpr int kOffM = kOffRed + 4 * kHeads * 4;        // 64 fp32 running maxima (log2 units)
constexpr int kOffAlpha = kOffM + kHeads * 4;          // 64 fp32 rescale factors, later 1 / l
constexpr int kOffMl = kOffAlpha + kHeads * 4;         // 64 x (m, l) of this CTA
constexpr int kOffBar = kOffMl + kMlBytes;
enum Bar {
  // Few barriers on purpose: a wait or a branch between tcgen05.mma
  // instructions stalls the issuing thread for about as long as several
  // MMAs, so the issuer waits once per batch of MMAs.
  kBarKFullA = 0,    // K chunks 0-5 of a tile in the ring (8 unpack warps) and S^T of the
                     // previous tile read (8 softmax warps)
  kBarKFreeA = 1,    // QK batch A done -> ring slots 0-2 reusable (commit)
  kBarKFullB = 2,    // K chunks 6-8 in ring slots 0-2 (8 unpack warps)
  kBarQKDone = 3,    // QK done: S^T full, every ring slot reusable (commit)
  kBarPVReady = 4,   // P^T written and V copied out of the K ring (8 softmax warps)
  kBarPVDone = 5,    // PV done: V tile and P^T buffer reusable, O^T settled (commit)
  kBarDrain = 6,     // every MMA finished (commit)
  kBarRx = 7,        // combine: the S partial slices have landed (TMA)
  kBarQ = 8,         // the raw query block has landed (TMA)
  kBarLastPV = 9,    // 4: block j of the last tile's PV done (commit)
  kBarRxMl = 13,     // combine: the S (m, l) blocks have landed (TMA)
  kBarVCopyA = 14,   // ring slots 0-2 copied into the V tile (8 softmax warps)
  kBarVCopyB = 15,   // the rest of the tile's latent chunks copied (8 softmax warps)
  kBarPVHalf = 16,   // PV blocks 0-1 done: V chunks 0, 1, 4, 5 reusable (commit)
  kNumBars = 17
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffL % 1024 == 0 && kOffR % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kOffMl % 16 == 0, "bulk copy source alignment");

// value dims [dim_lo(r), dim_lo(r + 1)) are combined by CTA r of S
__host__ __device__ constexpr int dim_lo(int r, int S) { return 4 * ((r * (kLatent / 4)) / S); }
// receive buffer of the combine: S slices of D rows of 128 bytes, then S (m, l) blocks
__host__ __device__ constexpr int rx_bytes(int D, int S) { return S * (D * 128 + kMlBytes); }
constexpr bool rx_fits_every_split_count() {
  for (int S = 2; S <= kMaxCluster; ++S)
    for (int r = 0; r < S; ++r)
      if (rx_bytes(dim_lo(r + 1, S) - dim_lo(r, S), S) > kRxBytes) return false;
  return true;
}
static_assert(rx_fits_every_split_count(), "combine receive buffer");

struct Params {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;
  RowSelect sel;
  int T, H, topk;
  float sl2;
  __nv_bfloat16* out;
  float* lse;
  __half* ws_o16;  // [T][H / 64][S][512 dims][64 heads] partials O / l (16-byte units swizzled by dim)
  float* ws_ml;    // [T][H / 64][S][64][2] (m in log2 units, l)
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
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or about `hint_ns` pass, so that waiting warps neither take
// issue slots nor hammer shared memory
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

// Bounded wait for the phase with the given parity: the thread sleeps in
// try_wait until the phase completes; the loop gives up after kWaitLimitNs
// of wall time, raising the CTA's abort flag and NVMLA_ERRW_WAIT_TIMEOUT.
// Also returns false once another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err_word) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_wait_hint(bar, parity, 100000)) return true;
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
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0);
}

// Bounded wait without abort handling (drain paths).
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity) && globaltimer_ns() - t0 < kWaitLimitNs) {
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

// 32 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&r)[32]) {
  NVMLA_TMEM_LD16F(taddr + 0, r, 0);
  NVMLA_TMEM_LD16F(taddr + 16, r, 16);
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

// maximum over the warp (every lane gets it); not volatile, so that
// independent reductions can be issued back to back
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
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

// ---- cluster rank and a barrier over every thread of every CTA with
// release / acquire semantics at cluster scope
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---- TMA bulk copies (1-D): addresses 16-byte aligned, sizes multiples of 16
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// fire-and-forget prefetch of a row into L2 (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- global loads (read-only path); the loads are volatile so that they
// are issued where they stand, as soon as their registers are free, and not
// sunk next to their first use
__device__ __forceinline__ void ldg_nc_v8(const void* p, uint32_t* v) {
  asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
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

// one row of a K chunk (64 dims = 32 columns of fp16 pairs) into this
// thread's TMEM lane: column 4u + e holds dims 8u + 2e, 8u + 2e + 1
__device__ __forceinline__ void tmem_store_chunk(const uint32_t (&c)[8], uint32_t scw, bool valid, uint32_t taddr) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[16];
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
      const int g = 2 * half + g2;
      const uint32_t s2 = e4m3_to_f16x2_bcast((scw >> (8 * g)) & 0xffu);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[4];
        e2m1x8_to_f16x8(c[2 * g + q], h);
#pragma unroll
        for (int e = 0; e < 4; ++e) w[8 * g2 + 4 * q + e] = valid ? hmul2_u32(h[e], s2) : 0u;
      }
    }
    NVMLA_TMEM_ST16(taddr + 16 * half, w, 0);
  }
}

// the RoPE chunk of one row (64 E4M3 bytes -> 32 columns of fp16 pairs)
__device__ __forceinline__ void tmem_store_rope(const uint32_t (&v)[16], bool valid, uint32_t taddr) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t lo, hi;
      e4m3x4_to_f16x4(v[8 * half + q], lo, hi);
      w[2 * q] = valid ? lo : 0u;
      w[2 * q + 1] = valid ? hi : 0u;
    }
    NVMLA_TMEM_ST16(taddr + 16 * half, w, 0);
  }
}

// QK MMA with A (the K rows) in TMEM and B (Q^T) in shared memory
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
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

// The cache's row format: 352-byte NVFP4 rows, or 576-byte FP8 rows (512
// latent + 64 RoPE E4M3 values, no scales).
enum RowFmt { kFmtNvfp4 = 0, kFmtFp8 = 1 };

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const Params p) {
  constexpr int kRB = FMT == kFmtFp8 ? kFp8RowBytes : kRowBytes;  // bytes per cache row
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

  if (tid == 0) NVMLA_TRACE_POINT(0);

  // ---- the query block (bf16, 64 KB latent + 8 KB RoPE, contiguous in
  // global memory) is requested first, with two TMA bulk loads into the
  // latent tile's space; it is converted after the barrier setup below
  if (tid == 0) {
    mbar_init(bar(kBarQ), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
    mbar_arrive_expect_tx(bar(kBarQ), kHeads * kDqk * 2);
    const int64_t qh0 = static_cast<int64_t>(t) * p.H + h0;
    bulk_load(sbase + kOffL, p.q_latent + qh0 * kLatent, kHeads * kLatent * 2, bar(kBarQ));
    bulk_load(sbase + kOffL + kHeads * kLatent * 2, p.q_rope + qh0 * kRope, kHeads * kRope * 2, bar(kBarQ));
  }

  // ---- start-up, level 1: the token's sequence and slot-list entries
  const bool is_unpack = tid < kUnpackThreads;
  const bool is_softmax = tid >= kSoftmax0 && tid < kSoftmax0 + 256;
  const int ur = tid & 127, uh = (tid >> 7) & 1;  // unpack threads: row, half
  const int sj = tid - kSoftmax0;                 // softmax threads: 0..255
  const int32_t seq_raw = p.sel.q_seq_idx ? ldg_nc_s32(p.sel.q_seq_idx + t) : 0;
  int32_t pos0 = -1;
  constexpr int kLaterPer = kMaxTiles / 2;  // later tiles per softmax thread
  int32_t posl[kLaterPer];
  if (is_unpack) {
    if (kbeg + ur < kend) pos0 = ldg_nc_s32(p.sel.topk_idx + static_cast<int64_t>(t) * p.topk + kbeg + ur);
  } else if (is_softmax) {
    // softmax thread sj handles row sj % 128 of tiles 1 + sj / 128 + 2m
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + (sj >> 7) + 2 * m;
      const int key = kbeg + i * kTile + (sj & 127);
      posl[m] = (i < ntiles && key < kend) ? ldg_nc_s32(p.sel.topk_idx + static_cast<int64_t>(t) * p.topk + key) : -1;
    }
  }
  // ---- level 2: block-table entries (page index clamped into the row, so
  // the load is in bounds whatever the entry) and the sequence length
  const bool seq_ok = seq_raw >= 0 && seq_raw < p.sel.num_seqs;
  const int32_t seq = seq_ok ? seq_raw : 0;
  const int32_t* bt_row = p.sel.block_table + static_cast<int64_t>(seq) * p.sel.max_pages;
  auto page_of = [&](int32_t pos) -> int32_t {
    const int32_t pi = min(max(pos >> 6, 0), p.sel.max_pages - 1);
    return ldg_nc_s32(bt_row + pi);
  };
  const bool report = blockIdx.z == 0;  // one head block reports bad entries
  // slot of position pos given its block-table entry (-1 for padding or a
  // bad entry, which is reported when `rep`)
  auto classify = [&](int32_t pos, int32_t page, int64_t limit, bool rep) -> int32_t {
    if (pos == -1) return -1;
    if (!seq_ok || pos < 0 || pos >= limit) {
      if (rep) report_error(p.err_word, NVMLA_ERRW_BAD_INDEX, 1);
      return -1;
    }
    const int64_t s = static_cast<int64_t>(page) * kPage + (pos & 63);
    if (page < 0 || s >= p.sel.num_slots) {
      if (rep) report_error(p.err_word, NVMLA_ERRW_BAD_SLOT, 1);
      return -1;
    }
    return static_cast<int32_t>(s);
  };
  // the physical row of pos, if it has one, before the sequence length is
  // known: its bytes are requested early and ignored when the row turns out
  // to lie past the sequence's end
  auto phys_slot = [&](int32_t pos, int32_t page) -> int32_t {
    if (!seq_ok || pos < 0 || (pos >> 6) >= p.sel.max_pages || page < 0) return -1;
    const int64_t s = static_cast<int64_t>(page) * kPage + (pos & 63);
    return s < p.sel.num_slots ? static_cast<int32_t>(s) : -1;
  };
  int32_t page0 = 0;
  int32_t pagel[kLaterPer];
  if (tid == 0) NVMLA_TRACE_AFTER(3, pos0);
  if (tid == 0) NVMLA_TRACE_AFTER(4, seq_raw);
  if (is_unpack) {
    page0 = page_of(pos0);
    if (tid == 0) NVMLA_TRACE_AFTER(5, page0);
  } else if (is_softmax) {
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) pagel[m] = (1 + (sj >> 7) + 2 * m < ntiles) ? page_of(posl[m]) : 0;
  }
  int64_t limit = static_cast<int64_t>(p.sel.max_pages) * kPage;
  if (p.sel.seq_lens) {
    const int64_t L = ldg_nc_s32(p.sel.seq_lens + seq);
    limit = L < limit ? L : limit;
  }

  // ---- level 3: rows of the first tile (unpack threads, into registers);
  // the later tiles' slots (softmax threads)
  // NVFP4: code bytes of latent chunks 4uh + j (32 each) and the scale bytes
  // of groups 16uh .. 16uh + 15. FP8: the E4M3 bytes of latent chunks
  // 4uh + 0..2 (64 each; chunk 4uh + 3 is loaded with the RoPE bytes).
  uint32_t rc[4][FMT == kFmtFp8 ? 16 : 8];
  uint4 rs;           // scale bytes (NVFP4)
  uint32_t rr[16];    // the 64 RoPE bytes (half 0 only)
  int32_t slot0 = -1;
  auto row_of = [&](int32_t slot) { return p.cache + cache_row_offset(slot, p.sel.page_rows, kRB); };
  // the part of a row batch A needs
  auto load_codes = [&](int32_t slot, int j) {
    if constexpr (FMT == kFmtFp8) {
      if (slot >= 0 && j < 3) {
        ldg_nc_v8(row_of(slot) + 256 * uh + 64 * j, rc[j]);
        ldg_nc_v8(row_of(slot) + 256 * uh + 64 * j + 32, rc[j] + 8);
      }
    } else {
      if (slot >= 0) ldg_nc_v8(row_of(slot) + 128 * uh + 32 * j, rc[j]);
    }
  };
  auto load_scale = [&](int32_t slot) {
    if constexpr (FMT != kFmtFp8)
      if (slot >= 0) rs = ldg_nc_v4(row_of(slot) + kScaleOff + 16 * uh);
  };
  // the part batch B needs beyond that
  auto load_rope = [&](int32_t slot) {
    if (slot < 0) return;
    const uint8_t* row = row_of(slot);
    if constexpr (FMT == kFmtFp8) {
      ldg_nc_v8(row + 256 * uh + 192, rc[3]);
      ldg_nc_v8(row + 256 * uh + 224, rc[3] + 8);
    }
    if (uh == 0) {
      constexpr int off = FMT == kFmtFp8 ? kLatent : kRopeOff;
      ldg_nc_v8(row + off, rr);
      ldg_nc_v8(row + off + 32, rr + 8);
    }
  };
  if (is_unpack) {
    const bool mine = ntiles > 0 && kbeg + ur < kend;
    const int32_t sspec = mine ? phys_slot(pos0, page0) : -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) load_codes(sspec, j);
    load_scale(sspec);
    if (mine) slot0 = classify(pos0, page0, limit, report && uh == 0);
    if (uh == 0) slots[ur] = slot0;
  } else if (is_softmax) {
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + (sj >> 7) + 2 * m;
      if (i < ntiles) slots[i * kTile + (sj & 127)] = classify(posl[m], pagel[m], limit, report);
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(1);

  // ---- setup: barriers, TMEM, the query block
  if (tid == kThreads - 1) {
    mbar_init(bar(kBarKFullA), 16);
    mbar_init(bar(kBarKFreeA), 1);
    mbar_init(bar(kBarKFullB), 8);
    mbar_init(bar(kBarQKDone), 1);
    mbar_init(bar(kBarPVReady), 8);
    mbar_init(bar(kBarVCopyA), 8);
    mbar_init(bar(kBarVCopyB), 8);
    mbar_init(bar(kBarPVDone), 1);
    mbar_init(bar(kBarPVHalf), 1);
    mbar_init(bar(kBarDrain), 2);
    mbar_init(bar(kBarRx), 1);
    mbar_init(bar(kBarRxMl), 1);
    for (int j = 0; j < 4; ++j) mbar_init(bar(kBarLastPV + j), 1);
    *abort_flag = (sbase & 1023u) ? 1 : 0;  // swizzled operands need a 1 KB aligned base
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kHeads) m_run[tid] = -INFINITY;
  if (warp == kQkWarp) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // query block -> fp16, K-major 128B-swizzled (4608 pieces of 16 bytes);
  // then the latent tile's space is free for the unpack
  if (wait_bar_warp(bar(kBarQ), 0, abort_flag, p.err_word)) {
    if (tid == 0) NVMLA_TRACE_POINT(6);
    const uint8_t* qraw = smem + kOffL;
    for (int i = tid; i < kHeads * 72; i += kThreads) {
      const int h = i / 72, j = i % 72, c = j >> 3, q = j & 7;
      const uint4 v = *reinterpret_cast<const uint4*>(
          qraw + (j < 64 ? h * (kLatent * 2) + 16 * j : kHeads * kLatent * 2 + h * (kRope * 2) + 16 * (j - 64)));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(bf16_bits_to_f32(w[e] & 0xffffu), bf16_bits_to_f32(w[e] >> 16));
      *reinterpret_cast<uint4*>(smem + kOffQ + c * 8192 + swz(h, q)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(7);
  fence_async_smem();
  __syncthreads();
  if (*abort_flag && tid == 0) report_error(p.err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  if (tid == 0) NVMLA_TRACE_POINT(2);

  const int sw = warp - 8;                    // softmax warp 0..7
  const int quad = sw & 3, hh = sw >> 2;      // TMEM lane quadrant, head half
  const int hb = hh * 32;                     // first head of this thread
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  const int64_t cbase = (static_cast<int64_t>(t) * gridDim.z + blockIdx.z) * S;  // first split of this cluster
  bool ok = true;
  if (is_unpack) {
    // ------------------------------------------------------------ unpack
    // Chunk use u of a tile (u = 0..8): latent chunk 4 (u & 1) + u / 2 for
    // u < 8, the RoPE chunk for u = 8; half uh writes the uses of parity uh
    // (and half 0 the RoPE chunk). Uses 0-5 sit in ring slots 0-5 (batch A),
    // uses 6-8 in slots 0-2 (batch B).
    ok = *abort_flag == 0;
    int32_t cur_slot = slot0;
    const uint32_t krow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kColK;  // this row's lane
    if (tid == 0) NVMLA_TRACE_AFTER(8, rc[0][0]);
    for (int i = 0; i < ntiles && ok; ++i) {
      const bool valid = cur_slot >= 0;
      const int32_t nxt_slot = (i + 1 < ntiles) ? slots[(i + 1) * kTile + ur] : -1;
      const uint32_t sc[4] = {rs.x, rs.y, rs.z, rs.w};
      // K batch A: latent chunks 4uh + 0..2 -> slots uh, 2 + uh, 4 + uh, once
      // QK of the previous tile is done and its V has been copied out
      if (i >= 1) {
        ok = wait_bar_warp(bar(kBarQKDone), (i - 1) & 1, abort_flag, p.err_word);
        if (ok) ok = wait_bar_warp(bar(kBarVCopyB), (i - 1) & 1, abort_flag, p.err_word);
      }
      if (!ok) break;
      if (tid == 0 && i < 2) NVMLA_TRACE_POINT(70 + 10 * i);
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        if constexpr (FMT == kFmtFp8) {
          tmem_store_rope(rc[j], valid, krow + 32 * (2 * j + uh));
        } else {
          tmem_store_chunk(rc[j], sc[j], valid, krow + 32 * (2 * j + uh));
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      warp_arrive(bar(kBarKFullA), lane);
      if (tid == 0 && i < 2) NVMLA_TRACE_POINT(10 + 4 * i);
      // K batch B: latent chunk 4uh + 3 -> slot uh; the RoPE chunk (half 0)
      // -> slot 2; once batch A's MMAs are done and slots 0-2 copied to V.
      // The RoPE bytes are requested first, their latency hidden by the waits.
      load_rope(cur_slot);
      ok = wait_bar_warp(bar(kBarKFreeA), i & 1, abort_flag, p.err_word);
      if (ok) ok = wait_bar_warp(bar(kBarVCopyA), i & 1, abort_flag, p.err_word);
      if (!ok) break;
      if (tid == 0 && i < 2) NVMLA_TRACE_POINT(72 + 10 * i);
      tc_fence_after();
      if constexpr (FMT == kFmtFp8) {
        tmem_store_rope(rc[3], valid, krow + 32 * uh);
      } else {
        tmem_store_chunk(rc[3], sc[3], valid, krow + 32 * uh);
      }
      if (uh == 0) tmem_store_rope(rr, valid, krow + 64);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      warp_arrive(bar(kBarKFullB), lane);
      if (tid == 0 && i < 2) NVMLA_TRACE_POINT(11 + 4 * i);
      // these registers now take the next tile's row
#pragma unroll
      for (int j = 0; j < 4; ++j) load_codes(nxt_slot, j);
      load_scale(nxt_slot);
      cur_slot = nxt_slot;
      if (tid == 0 && i < 2) NVMLA_TRACE_POINT(12 + 4 * i);
    }
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads on different SM sub-partitions: one issues QK
    // (batch A, 24 MMAs, and batch B, 12, per tile), the other PV (32 per
    // tile). A thread issuing tcgen05.mma competes for issue with the other
    // warps of its sub-partition, so one issuer alone cannot keep the tensor
    // core busy; the two streams touch different accumulators and are
    // ordered only through the barriers. One wait before each batch, one
    // commit after it, fully unrolled straight-line MMA sequences in between
    // (a loop branch between MMAs costs issue time).
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(false, false);
      constexpr uint32_t idesc_pv = idesc_f16(true, true);
      const uint32_t lb = sbase + kOffL, rb = sbase + kOffR, qb = sbase + kOffQ;
      const uint32_t ring = tmem + kColK;
      bool mok = *abort_flag == 0;
      if (warp == kPvWarp) {
        // Block j reads V chunks j and j + 4: after blocks 0-1 the next
        // tile's V copy may start on chunks 0, 1, 4, 5. The last tile's PV
        // reports each block instead, so that the epilogue can start on it
        // (a separate copy of the sequence: a conditional branch between
        // MMAs costs issue time).
        auto issue_pv = [&](int i) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16(tmem + kColO + 64 * j, sdesc(lb + j * kChunkBytes + 2048 * ks, 4 * kChunkBytes, 1024),
                      sdesc(rb + 2048 * ks, 8192, 1024), idesc_pv, (i | ks) != 0);
          }
          mma_commit(bar(kBarPVHalf));
#pragma unroll
          for (int j = 2; j < 4; ++j) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16(tmem + kColO + 64 * j, sdesc(lb + j * kChunkBytes + 2048 * ks, 4 * kChunkBytes, 1024),
                      sdesc(rb + 2048 * ks, 8192, 1024), idesc_pv, (i | ks) != 0);
          }
          mma_commit(bar(kBarPVDone));
        };
        auto issue_pv_last = [&](int i) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16(tmem + kColO + 64 * j, sdesc(lb + j * kChunkBytes + 2048 * ks, 4 * kChunkBytes, 1024),
                      sdesc(rb + 2048 * ks, 8192, 1024), idesc_pv, (i | ks) != 0);
            mma_commit(bar(kBarLastPV + j));
          }
          mma_commit(bar(kBarPVDone));
        };
        for (int i = 0; i < ntiles && mok; ++i) {
          mok = wait_bar(bar(kBarPVReady), i & 1, abort_flag, p.err_word);
          if (!mok) break;
          tc_fence_after();
          if (i < 2) NVMLA_TRACE_POINT(60 + 6 * i);
          if (i + 1 < ntiles) {
            issue_pv(i);
          } else {
            issue_pv_last(i);
          }
          if (i < 2) NVMLA_TRACE_POINT(61 + 6 * i);
        }
      } else {
        for (int i = 0; i < ntiles && mok; ++i) {
          mok = wait_bar(bar(kBarKFullA), i & 1, abort_flag, p.err_word);
          if (!mok) break;
          tc_fence_after();
          if (i < 2) NVMLA_TRACE_POINT(50 + 8 * i);
          // batch A: uses 0..5 (slot u, query chunk 4 (u & 1) + u / 2)
#pragma unroll
          for (int u = 0; u < 6; ++u) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f16_ts(tmem + kColS, ring + 32 * u + 8 * ks,
                         sdesc(qb + (4 * (u & 1) + (u >> 1)) * 8192 + 32 * ks, 16, 1024), idesc_qk, (u | ks) != 0);
          }
          mma_commit(bar(kBarKFreeA));
          if (i < 2) NVMLA_TRACE_POINT(51 + 8 * i);
          mok = wait_bar(bar(kBarKFullB), i & 1, abort_flag, p.err_word);
          if (!mok) break;
          tc_fence_after();
          if (i < 2) NVMLA_TRACE_POINT(54 + 8 * i);
          // batch B: uses 6, 7 (latent chunks 3, 7) in slots 0, 1; use 8 (RoPE) in slot 2
#pragma unroll
          for (int u = 0; u < 3; ++u) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f16_ts(tmem + kColS, ring + 32 * u + 8 * ks,
                         sdesc(qb + (u == 2 ? 8 : 3 + 4 * u) * 8192 + 32 * ks, 16, 1024), idesc_qk, 1);
          }
          mma_commit(bar(kBarQKDone));
          if (i < 2) NVMLA_TRACE_POINT(55 + 8 * i);
        }
      }
      // every MMA this thread issued has finished once both issuers' commits land
      mma_commit(bar(kBarDrain));
      wait_bar_drain(bar(kBarDrain), 0);
    }
    __syncwarp();
  } else if (is_softmax) {
    // ------------------------------------------------------------ softmax
    const int k = quad * 32 + lane;  // row of this thread
    float lp[32];  // this row's share of its heads' sums
#pragma unroll
    for (int h = 0; h < 32; ++h) lp[h] = 0.f;
    // the later tiles' rows to L2, now that the first tile's are in flight
    // (requested together with them, they delay them)
    for (int i = 1 + (sj >> 7); i < ntiles; i += 2) {
      const int32_t sl = slots[i * kTile + (sj & 127)];
      if (sl >= 0) prefetch_l2(p.cache + cache_row_offset(sl, p.sel.page_rows, kRB), kRB);
    }
    // S^T is free for the first tile
    warp_arrive(bar(kBarKFullA), lane);
    ok = !softmax_sync_or(*abort_flag != 0);
    // V tile i from the K ring (its latent chunks are the V operand's rows):
    // this warp copies columns 16hh..16hh+15 of each ring slot, row k
    uint8_t* vrow = smem + kOffL;
    auto copy_slot = [&](int slot, int chunk) {
      uint8_t* dst = vrow + chunk * kChunkBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t w[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                     : "r"(tmem + lane_base + kColK + 32 * slot + 16 * hh + 8 * half));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int q = 0; q < 2; ++q)
          *reinterpret_cast<uint4*>(dst + swz(quad * 32 + lane, 4 * hh + 2 * half + q)) =
              make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
    };
    for (int i = 0; i < ntiles && ok; ++i) {
      // part A: slots 0-2 hold latent chunks 0, 4, 1 until batch B reuses
      // them; their V chunks are free once PV blocks 0-1 of the previous
      // tile are done
      ok = wait_bar_warp(bar(kBarKFullA), i & 1, abort_flag, p.err_word);
      if (ok && i >= 1) ok = wait_bar_warp(bar(kBarPVHalf), (i - 1) & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      copy_slot(0, 0);
      copy_slot(1, 4);
      copy_slot(2, 1);
      tc_fence_before();
      warp_arrive(bar(kBarVCopyA), lane);
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(104 + 10 * i);
      // chunks 5, 2, 6 (slots 3-5, which batch B leaves alone) while the
      // unpack fills batch B; chunks 2 and 6 once the whole PV is done
      copy_slot(3, 5);
      if (i >= 1) ok = wait_bar_warp(bar(kBarPVDone), (i - 1) & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      copy_slot(4, 2);
      copy_slot(5, 6);
      // part B: chunks 3, 7 (slots 0, 1, batch B)
      ok = wait_bar_warp(bar(kBarKFullB), i & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      copy_slot(0, 3);
      copy_slot(1, 7);
      fence_async_smem();
      tc_fence_before();
      warp_arrive(bar(kBarVCopyB), lane);
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(105 + 10 * i);
      ok = wait_bar_warp(bar(kBarQKDone), i & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(30 + 3 * i);
      const bool valid = slots[i * kTile + k] >= 0;
      float s[32];
      tmem_ld32f(tmem + lane_base + kColS + hb, s);
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(100 + 10 * i);
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
      // does any score exceed its head's running maximum by more than 2^tau?
      float excess = -INFINITY;
      if (i == 0) {
        // The running maximum starts at the largest of rows 0, 32, 64 and 96
        // (-inf where all four are masked): any value that some score
        // reaches is a valid reference, and the exact reduction below runs
        // only if a score of the tile lies more than 2^tau above it.
        if (lane == 0) {
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4)
            *reinterpret_cast<float4*>(red + quad * 64 + hb + 4 * h4) =
                make_float4(s[4 * h4], s[4 * h4 + 1], s[4 * h4 + 2], s[4 * h4 + 3]);
        }
        softmax_sync();
        if (quad == 0) {
          const int h = hb + lane;
          m_run[h] = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
        }
        softmax_sync();
      }
      if (valid) {
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 m4 = *reinterpret_cast<const float4*>(m_run + hb + 4 * h4);
          excess = fmaxf(excess, fmaxf(fmaxf(s[4 * h4] - m4.x, s[4 * h4 + 1] - m4.y),
                                       fmaxf(s[4 * h4 + 2] - m4.z, s[4 * h4 + 3] - m4.w)));
        }
      }
      // (the barrier below also publishes the first tile's m_run)
      const bool slow = softmax_sync_or(excess > kTau);
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(101 + 10 * i);
      // (PV of the previous tile has finished: waited for before the V copy)
      // S^T is in registers: QK of the next tile may overwrite it
      tc_fence_before();
      warp_arrive(bar(kBarKFullA), lane);
      if (slow) {
        // exact per-head maximum of this tile: warp reductions that leave s
        // intact, then across the four lane quadrants
        float mine = -INFINITY;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float mh = warp_max(s[h]);
          mine = lane == h ? mh : mine;
        }
        red[quad * 64 + hb + lane] = mine;
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
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + hb + 4 * h4);
          lp[4 * h4] *= a4.x;
          lp[4 * h4 + 1] *= a4.y;
          lp[4 * h4 + 2] *= a4.z;
          lp[4 * h4 + 3] *= a4.w;
        }
        if (i >= 1) {
          // O^T holds the finished PV of every earlier tile
          tc_fence_after();
          if (ok) {
            // 16 columns at a time
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
        }
      }
      // P = 2^(s - m); masked rows give 0
#pragma unroll
      for (int h4 = 0; h4 < 8; ++h4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_run + hb + 4 * h4);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 4 * h4 + e;
          const float pv = valid ? ex2(s[h] - mm[e]) : 0.f;
          s[h] = pv;
          lp[h] += pv;
        }
      }
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(102 + 10 * i);
      // P^T row (this thread's 32 heads) -> R, once PV of the previous tile
      // has read it
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
      warp_arrive(bar(kBarPVReady), lane);
      if (tid == kSoftmax0 && i < 2) NVMLA_TRACE_POINT(31 + 3 * i);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
    }
    // ------------------------------------------------------------ row sums
    ok = !softmax_sync_or(!ok);
    warp_reduce32<false>(lp, lane);
    red[quad * 64 + hb + lane] = lp[0];
    softmax_sync();
    if (quad == 0) {
      const int h = hb + lane;
      const float l = (red[h] + red[64 + h]) + (red[128 + h] + red[192 + h]);
      const bool live = ok && ntiles > 0 && l > 0.f;
      ml_pub[2 * h] = live ? m_run[h] : -INFINITY;
      ml_pub[2 * h + 1] = live ? l : 0.f;
      alpha_s[h] = live ? 1.f / l : 0.f;
      if (S == 1) p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = live ? (m_run[h] + log2f(l)) * kLn2 : -INFINITY;
    }
    fence_async_smem();  // ml_pub is read by a bulk copy below
    softmax_sync();
    if (tid == kSoftmax0) NVMLA_TRACE_POINT(40);
    // ------------------------------------------------------------ O^T, block by block as PV finishes
    __half* wo = p.ws_o16 + (cbase + rank) * (kLatent * kHeads);
    bool have = ok && ntiles > 0;
    for (int j = 0; j < 4; ++j) {
      if (have) have = wait_bar_warp(bar(kBarLastPV + j), 0, abort_flag, p.err_word);
      tc_fence_after();
      float o[32];
      if (have) {
        tmem_ld32f(tmem + lane_base + kColO + 64 * j + hb, o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
      // TMEM lane k of block j: dim 64j + k (k < 64) or 256 + 64j + k - 64
      const int d = (k < 64) ? 64 * j + k : 256 + 64 * j + (k - 64);
      if (S == 1) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          p.out[(static_cast<int64_t>(t) * p.H + h0 + hb + e) * kLatent + d] =
              __float2bfloat16_rn(o[e] * alpha_s[hb + e]);
      } else {
        // normalised partial (fp16, [row k][64 heads], unit u of row k at
        // u ^ (k & 7)) staged in latent chunk j, which PV no longer reads
        uint8_t* stg = smem + kOffL + j * kChunkBytes + k * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int hl = 8 * cc + 2 * e;
            w4[e] = pack_f16x2(o[hl] * alpha_s[hb + hl], o[hl + 1] * alpha_s[hb + hl + 1]);
          }
          *reinterpret_cast<uint4*>(stg + (((4 * hh + cc) ^ (k & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        fence_async_smem();
        softmax_sync();
        if (tid == kSoftmax0) {
          const uint32_t src = sbase + kOffL + j * kChunkBytes;
          bulk_store(wo + (64 * j) * kHeads, src, 64 * 128);
          bulk_store(wo + (256 + 64 * j) * kHeads, src + 64 * 128, 64 * 128);
          if (j == 3) bulk_store(p.ws_ml + (cbase + rank) * (kHeads * 2), sbase + kOffMl, kMlBytes);
          bulk_commit();
          if (j == 0) NVMLA_TRACE_POINT(47);
        }
      }
    }
    tc_fence_before();
    if (S > 1 && tid == kSoftmax0) {
      // the partial is complete in global memory before the cluster barrier
      bulk_wait_all();
      fence_async_global();
    }
    if (tid == kSoftmax0) NVMLA_TRACE_POINT(41);
  }

  // ------------------------------------------------------------ combine
  __syncthreads();  // every role is done with TMEM
  if (warp == kQkWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (S > 1) {
    // release / acquire at cluster scope: every partial of the cluster is
    // visible to every CTA of it
    cluster_sync_all();
    if (tid == 0) NVMLA_TRACE_POINT(42);
    const int d0 = dim_lo(static_cast<int>(rank), S);
    const int D = dim_lo(static_cast<int>(rank) + 1, S) - d0;
    const uint32_t rx = sbase + kOffQ;
    const uint32_t rx_ml = rx + S * D * 128;
    if (tid == 0) {
      // the small (m, l) blocks first: the weights are computed while the
      // partial slices are still on their way
      fence_async_global();
      mbar_arrive_expect_tx(bar(kBarRxMl), static_cast<uint32_t>(S * kMlBytes));
      for (int s = 0; s < S; ++s)
        bulk_load(rx_ml + s * kMlBytes, p.ws_ml + (cbase + s) * (kHeads * 2), kMlBytes, bar(kBarRxMl));
      mbar_arrive_expect_tx(bar(kBarRx), static_cast<uint32_t>(S * D * 128));
      for (int s = 0; s < S; ++s)
        bulk_load(rx + s * D * 128, p.ws_o16 + (cbase + s) * (kLatent * kHeads) + d0 * kHeads, D * 128, bar(kBarRx));
    }
    // combine weights l_s 2^(m_s - M) / L per head, [S][64] in R: eight
    // consecutive lanes per head, splits s = q, q + 8
    float* coef = reinterpret_cast<float*>(smem + kOffR);
    const float* rml = reinterpret_cast<const float*>(smem + kOffQ + S * D * 128);
    if (tid < 8 * kHeads && wait_bar_warp(bar(kBarRxMl), 0, abort_flag, p.err_word)) {
      const int h = tid >> 3, q = tid & 7;
      float m2[2], l2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int s = q + 8 * e;
        l2[e] = s < S ? rml[s * 128 + 2 * h + 1] : 0.f;
        m2[e] = l2[e] > 0.f ? rml[s * 128 + 2 * h] : -INFINITY;
      }
      float M = fmaxf(m2[0], m2[1]);
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float w2[2], L = 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        w2[e] = l2[e] > 0.f ? l2[e] * ex2(m2[e] - M) : 0.f;
        L += w2[e];
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (q + 8 * e < S) coef[(q + 8 * e) * kHeads + h] = w2[e] * inv;
      if (rank == 0 && q == 0)
        p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    if (tid == 0) NVMLA_TRACE_POINT(45);
    wait_bar_warp(bar(kBarRx), 0, abort_flag, p.err_word);
    __syncthreads();
    if (tid == 0) NVMLA_TRACE_POINT(43);
    // item = (head group u, dim row dl): lanes take consecutive dims
    const uint8_t* rxp = smem + kOffQ;
    for (int it = tid; it < D * 8; it += kThreads) {
      const int u = it / D, dl = it - u * D, d = d0 + dl;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int s = 0; s < S; ++s) {
        const uint4 v = *reinterpret_cast<const uint4*>(rxp + s * D * 128 + dl * 128 + ((u ^ (d & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const float4 c0 = *reinterpret_cast<const float4*>(coef + s * kHeads + 8 * u);
        const float4 c1 = *reinterpret_cast<const float4*>(coef + s * kHeads + 8 * u + 4);
        const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          acc[2 * e] += c[2 * e] * f.x;
          acc[2 * e + 1] += c[2 * e + 1] * f.y;
        }
      }
      // straight to out: the lanes of a warp write consecutive dims of a head
      __nv_bfloat16* o = p.out + (static_cast<int64_t>(t) * p.H + h0 + 8 * u) * kLatent + d;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e * kLatent] = __float2bfloat16_rn(acc[e]);
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(44);
}

}  // namespace tc

bool tc_supported(int H) { return H % tc::kHeads == 0; }
bool tc_fp8_rows_supported(int) { return false; }

namespace {

// Per-device launch setup of the kernel: its shared-memory size, and for
// every cluster size S how many clusters of S CTAs can be resident at once
// (0: S cannot be launched).
// Per-device launch set-up, filled on the first call on each device. Two host
// threads making their first call on one device at once may both fill it,
// with the same values; one that sees `ready` before the occupancy table
// (the flag is a plain bool) reads zeros there and takes one split for that
// call, which is slower but gives the same results.
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
  // both row formats: the same launch shape and resources
  bool non_portable = true;
  for (auto* k : {tc::decode_tc_kernel<tc::kFmtNvfp4>, tc::decode_tc_kernel<tc::kFmtFp8>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
    if (e != cudaSuccess) return -1;
    non_portable = non_portable &&
                   cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  }
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
    if (cudaOccupancyMaxActiveClusters(&n, tc::decode_tc_kernel<tc::kFmtNvfp4>, &cfg) == cudaSuccess) d.max_active[s] = n;
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

// Key splits per token. Each candidate split count S is costed as the waves
// of clusters it needs (the clusters of S CTAs the device holds at once, from
// the occupancy query) times the time of one wave, modelled from measurements
// at 64 heads and top-2048 on a GB300: a fixed part (start-up and the split
// combine) plus a per-tile part for the busiest CTA. The cheapest S wins (the
// smaller on a tie), then the fewest splits that give the busiest CTA the
// same number of tiles. Up to one wave of clusters this is the largest S
// that still fits; beyond it, fewer, longer waves can win.
int tc_default_splits(int T, int H, int topk, int num_sms) {
  constexpr double kWaveFixedUs = 19.0;  // per wave: start-up, tail, combine
  constexpr double kTileUs = 5.0;        // per 128-row tile of the busiest CTA
  const int tiles = (topk + tc::kTile - 1) / tc::kTile;
  const int clusters = max(1, T * (H / tc::kHeads));
  const int dev = tc_prepare();
  int best = 1;
  double best_cost = -1.0;
  for (int s = 1; s <= min(tiles, tc::kMaxCluster); ++s) {
    // clusters of s CTAs resident at once (no device: the portable sizes,
    // one CTA per SM)
    const int resident = dev < 0 ? (s <= 8 ? num_sms / s : 0) : g_tc_dev[dev].max_active[s];
    if (resident < 1) continue;
    const int waves = (clusters + resident - 1) / resident;
    const int per = (tiles + s - 1) / s;
    const double cost = waves * (kWaveFixedUs + kTileUs * per);
    if (best_cost < 0.0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  const int per = (tiles + best - 1) / best;  // tiles of the busiest CTA
  return (tiles + per - 1) / per;             // fewest splits with that load
}

size_t tc_workspace_bytes(int T, int H, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(T) * (H / tc::kHeads) * splits * (tc::kPartBytes + tc::kMlBytes);
}

cudaError_t launch_decode_tc(int fmt, const void* q_latent, const void* q_rope, const uint8_t* cache,
                             const RowSelect& sel, const int32_t* row_idx, int T, int H, int topk, float sm_scale,
                             void* out, float* lse, void* workspace, int splits, int32_t* err_word,
                             cudaStream_t stream) {
  // fmt: 0 = NVFP4 rows, 2 = FP8 rows in a paged cache
  if (fmt != 0 && fmt != 2) return cudaErrorNotSupported;
  (void)row_idx;
  if (tc_prepare() < 0) return cudaErrorInvalidDevice;
  if (splits < 1 || splits > tc::kMaxCluster) return cudaErrorInvalidValue;
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
  if (fmt == 2) return cudaLaunchKernelEx(&cfg, tc::decode_tc_kernel<tc::kFmtFp8>, p);
  return cudaLaunchKernelEx(&cfg, tc::decode_tc_kernel<tc::kFmtNvfp4>, p);
}

}  // namespace nvmla

#ifdef NVMLA_TRACE
extern "C" int nvmla_tc_trace_read(void* host_dst, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(host_dst, nvmla::tc::nvmla_tc_trace, bytes));
}
#endif
