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
// One CTA = one query token x 64 heads x a range of the token's slots, taken
// in tiles of 128 rows. Roles:
//
//   warps 0-7  unpack: thread (row r, part h) loads the parts of its cache
//              row it needs (192 of the 352 bytes) straight into registers,
//              one tile ahead, and writes fp16 operands (E2M1 x E4M3 is exact
//              in fp16) into shared memory, 128B-swizzled: latent chunk
//              c = 2j + h (64 dims) for j = 0..3 and half of the RoPE chunk.
//   MMA issue: one softmax thread issues QK as chunk pairs land and PV as
//              soon as P^T is written; M = 128 throughout:
//                S^T[128 rows, 64 heads]   = K[128 x 576] . Q^T   (9 chunks)
//                O^T[512 dims, 64 heads]  += V^T[512 x 128] . P^T (4 blocks)
//              The latent chunks are unpacked once: a K-major 128-row x
//              64-dim chunk is byte for byte the MN-major layout of V^T for
//              those 64 value dims, so block j of PV reads chunks 2j, 2j+1.
//              Block j's completion frees chunks 2j, 2j+1 for the next tile.
//   warps 8-11 softmax: thread = row (TMEM lane). The running maximum of
//              every head stays fixed while no score exceeds it by more than
//              2^8 (P stays below 256, safe in fp16); only a tile that does
//              (always the first) pays for the exact cross-row maximum and
//              the rescale of O^T in TMEM. Row sums accumulate per thread and
//              are reduced across rows once, at the end. P^T goes to shared
//              memory in place of the RoPE chunk, which QK no longer needs.
//
// Shared memory: query block (72 KB) + latent tile (128 KB) + RoPE/P^T chunk
// (16 KB) + slot list. TMEM: S^T 64 columns, O^T 4 x 64 columns.
//
// Key splits: several CTAs may share a token; each then writes its
// normalised partial output (fp16) with (m, l) and a merge kernel combines
// them; a single CTA writes out/lse directly.
// Every wait is bounded: on timeout the CTA sets NVMLA_ERRW_WAIT_TIMEOUT,
// drains its MMAs, frees TMEM and exits.
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

constexpr int kTile = 128;          // rows per tile (MMA M)
constexpr int kHeads = 64;          // heads per CTA (MMA N)
constexpr int kMaxTiles = 16;       // 2048 slots
constexpr int kThreads = 384;         // 12 warps: 3 per SM sub-partition
constexpr int kUnpackThreads = 256;  // warps 0-7
constexpr int kSoftmaxWarp0 = 8;     // warps 8-11; thread 256 also issues every MMA
constexpr int kAllocWarp = 8;        // allocates and frees TMEM
constexpr int kChunkBytes = 16384;   // 128 rows x 128 bytes
constexpr int kPieces = 12;          // 16-byte pieces of a row one unpack thread holds
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;        // S^T: columns [0, 64)
constexpr uint32_t kColO = 64;       // O^T block j: columns [64 + 64 j, +64)
constexpr float kTau = 8.0f;         // rescale threshold, log2 units
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// shared memory map (bytes); the base is 1 KB aligned
constexpr int kOffQ = 0;                              // 9 x 8 KB: query, K-major
constexpr int kOffL = kOffQ + 9 * 8192;               // 8 x 16 KB: latent tile
constexpr int kOffR = kOffL + 8 * kChunkBytes;        // 16 KB: RoPE chunk, then P^T
constexpr int kOffSlots = kOffR + kChunkBytes;        // kMaxTiles x 128 int32
constexpr int kOffRed = kOffSlots + kMaxTiles * kTile * 4;  // 4 x 64 fp32
constexpr int kOffM = kOffRed + 4 * kHeads * 4;       // 64 fp32 running maxima
constexpr int kOffAlpha = kOffM + kHeads * 4;         // 64 fp32 rescale factors
constexpr int kOffLsum = kOffAlpha + kHeads * 4;      // 64 fp32 final row sums
constexpr int kOffBar = kOffLsum + kHeads * 4;
enum Bar {
  kBarQReady = 0,    // query block converted (12 warps)
  kBarPairFull = 1,  // 4: latent chunks 2j, 2j+1 written (8 unpack warps)
  kBarRopeFull = 5,  // RoPE chunk written (8 unpack warps)
  kBarLFree = 6,     // 4: PV block j done -> chunks 2j, 2j+1 reusable (commit)
  kBarRFree = 10,    // PV done -> RoPE/P^T chunk reusable (commit)
  kBarSFull = 11,    // QK done (commit)
  kBarPFull = 12,    // P^T written and O^T rescaled (4 softmax warps)
  kBarODone = 13,    // PV done (commit)
  kBarDrain = 14,    // every MMA finished (commit)
  kBarSlots = 15,    // slot list of tiles 1.. written (4 softmax warps)
  kNumBars = 16
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;
  RowSelect sel;
  int T, H, topk;
  float sl2;
  __nv_bfloat16* out;
  float* lse;
  __half* ws_o16;  // [T][S][512][H] normalised partials
  float* ws_ml;    // [T][S][H][2] (m in log2 units, l)
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

// named barrier among the four softmax warps (id 1); the _or form returns
// the OR of a predicate over the group (used to make the outcome of a
// bounded wait, or a data-dependent branch, uniform)
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

// The query block (64 heads x 576 dims, bf16 in global memory) as fp16 in
// the K-major 128B-swizzled layout of the QK B operand. The 384 threads of
// the unpack and softmax warps each convert 12 of the 4608 16-byte pieces;
// all loads are issued before the first conversion so their latencies overlap.
__device__ __forceinline__ void convert_query(const __nv_bfloat16* q_latent, const __nv_bfloat16* q_rope,
                                              int64_t head0, uint8_t* qsmem, int tid) {
  constexpr int kPer = kHeads * 72 / 384;  // 12
  uint4 v[kPer];
#pragma unroll
  for (int n = 0; n < kPer; ++n) {
    const int i = tid + 384 * n;
    const int h = i / 72, j = i % 72;
    const int64_t qh = head0 + h;
    v[n] = j < 64 ? __ldg(reinterpret_cast<const uint4*>(q_latent + qh * kLatent) + j)
                  : __ldg(reinterpret_cast<const uint4*>(q_rope + qh * kRope) + (j - 64));
  }
#pragma unroll
  for (int n = 0; n < kPer; ++n) {
    const int i = tid + 384 * n;
    const int h = i / 72, j = i % 72, c = j >> 3, q = j & 7;
    const uint32_t w[4] = {v[n].x, v[n].y, v[n].z, v[n].w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(bf16_bits_to_f32(w[e] & 0xffffu), bf16_bits_to_f32(w[e] >> 16));
    *reinterpret_cast<uint4*>(qsmem + c * 8192 + swz(h, q)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
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

// The 16-byte pieces of a 352-byte row that unpack thread part h holds:
// codes of latent chunks h, h+2, h+4, h+6 (pieces 2c, 2c+1), both scale
// pieces (16, 17) and its half of the RoPE bytes (18 + 2h, 19 + 2h).
__device__ __forceinline__ int piece_of(int n, int h) {
  return n < 8 ? 2 * (2 * (n >> 1) + h) + (n & 1) : (n < 10 ? 16 + (n - 8) : 18 + 2 * h + (n - 10));
}

__device__ __forceinline__ void load_row(const uint8_t* cache, int32_t slot, int h, uint4 (&raw)[kPieces]) {
  if (slot < 0) return;
  const uint4* row = reinterpret_cast<const uint4*>(cache + static_cast<int64_t>(slot) * kRowBytes);
#pragma unroll
  for (int n = 0; n < kPieces; ++n) raw[n] = __ldg(row + piece_of(n, h));
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

// row pieces of one unpack thread; the loads are volatile so that they are
// issued here (one tile ahead) and not sunk next to their first use
__device__ __forceinline__ void load_row_now(const uint8_t* cache, int32_t slot, int h, uint4 (&raw)[kPieces]) {
  if (slot < 0) return;
  const uint8_t* row = cache + static_cast<int64_t>(slot) * kRowBytes;
#pragma unroll
  for (int n = 0; n < kPieces; ++n) raw[n] = ldg_nc_v4(row + 16 * piece_of(n, h));
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * kHeads;

  int32_t* slots = reinterpret_cast<int32_t*>(smem + kOffSlots);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* m_run = reinterpret_cast<float*>(smem + kOffM);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return sbase + kOffBar + 8 * i; };

  const int tile_lo = (split * p.tiles_total) / p.num_splits;
  const int tile_hi = ((split + 1) * p.tiles_total) / p.num_splits;
  const int kbeg = tile_lo * kTile;
  const int kend = min(tile_hi * kTile, p.topk);
  const int nkeys = max(0, kend - kbeg);
  const int ntiles = (nkeys + kTile - 1) / kTile;  // <= kMaxTiles (host check)

  if (tid == 0) NVMLA_TRACE_POINT(40);

  // sequence facts of this token
  const int32_t seq = p.sel.q_seq_idx ? __ldg(p.sel.q_seq_idx + t) : 0;
  const int32_t* bt_row = p.sel.block_table + static_cast<int64_t>(seq) * p.sel.max_pages;
  const int32_t* idx_row = p.sel.topk_idx + static_cast<int64_t>(t) * p.topk;
  auto limit_of = [&]() -> int64_t {
    int64_t lim = static_cast<int64_t>(p.sel.max_pages) * kPage;
    if (p.sel.seq_lens) {
      const int64_t L = __ldg(p.sel.seq_lens + seq);
      lim = L < lim ? L : lim;
    }
    return lim;
  };
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

  // ---- loads that do not depend on shared memory start before setup
  const int ur = tid & 127, uh = (tid >> 7) & 1;  // unpack threads: row, part
  uint4 rawA[kPieces], rawB[kPieces];
  int32_t slotA = -1, slotB = -1;
  int32_t pos0 = -1;
  if (tid < kUnpackThreads && kbeg + ur < kend) pos0 = ldg_nc_s32(idx_row + kbeg + ur);
  constexpr int kQPer = kHeads * 72 / kThreads;  // 12 query pieces per thread
  uint4 qv[kQPer];
#pragma unroll
  for (int n = 0; n < kQPer; ++n) {
    const int i = tid + kThreads * n;
    const int h = i / 72, j = i % 72;
    const int64_t qh = static_cast<int64_t>(t) * p.H + h0 + h;
    qv[n] = j < 64 ? ldg_nc_v4(p.q_latent + qh * kLatent + 8 * j) : ldg_nc_v4(p.q_rope + qh * kRope + 8 * (j - 64));
  }

  // ---- setup
  if (tid == kThreads - 1) {
    mbar_init(bar(kBarQReady), 12);
    for (int j = 0; j < 4; ++j) {
      mbar_init(bar(kBarPairFull + j), 8);
      mbar_init(bar(kBarLFree + j), 1);
    }
    mbar_init(bar(kBarRopeFull), 8);
    mbar_init(bar(kBarRFree), 1);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarSlots), 4);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (*abort_flag && tid == 0) report_error(p.err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  if (tid == 0) NVMLA_TRACE_POINT(0);

  // query block -> fp16, K-major 128B-swizzled (all 12 warps)
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
  warp_arrive(bar(kBarQReady), lane);

  if (tid < kUnpackThreads) {
    // ------------------------------------------------------------ unpack
    // tile 0: page of the row, then its pieces (errors reported by part 0;
    // the softmax warps build the slot list of the later tiles)
    if (ntiles > 0) {
      slotA = (kbeg + ur < kend) ? slot_of_pos(pos0, limit_of(), uh == 0 && blockIdx.z == 0) : -1;
      if (tid == 0) NVMLA_TRACE_POINT(41);
      load_row_now(p.cache, slotA, uh, rawA);
      if (uh == 0) slots[ur] = slotA;
    }
    if (tid == 0) NVMLA_TRACE_POINT(13);
    bool ok = *abort_flag == 0;
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      return wait_bar_warp(b, parity, abort_flag, p.err_word);
    };
    // one tile: chunks are written as the previous tile's PV frees them; the
    // next tile's rows are requested after the first pair
    auto tile = [&](int i, const uint4 (&cur)[kPieces], int32_t cur_slot, uint4 (&nxt)[kPieces],
                    int32_t& nxt_slot) -> bool {
      const bool valid = cur_slot >= 0;
      if (tid == 0 && i < 2) {
        uint32_t x = cur[0].x ^ cur[11].w;  // first use: the pieces have arrived
        asm volatile("" ::"r"(x));
        NVMLA_TRACE_POINT(44 + i);
      }
      for (int j = 0; j < 4; ++j) {
        if (i >= 1 && !wait_warp(bar(kBarLFree + j), (i - 1) & 1)) return false;
        uint8_t* chunk = smem + kOffL + (2 * j + uh) * kChunkBytes;
        if (valid) {
          write_latent(cur, j, uh, chunk, ur);
        } else {
          zero_row(chunk, ur);
        }
        fence_async_smem();
        warp_arrive(bar(kBarPairFull + j), lane);
        if (j == 0 && i + 1 < ntiles) {
          if (i == 0 && !wait_warp(bar(kBarSlots), 0)) return false;
          nxt_slot = slots[(i + 1) * kTile + ur];
          load_row_now(p.cache, nxt_slot, uh, nxt);
        }
      }
      if (i >= 1 && !wait_warp(bar(kBarRFree), (i - 1) & 1)) return false;
      uint8_t* rc = smem + kOffR;
      if (valid) {
        write_rope(cur, uh, rc, ur);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(rc + swz(ur, 4 * uh + c)) = make_uint4(0, 0, 0, 0);
      }
      fence_async_smem();
      warp_arrive(bar(kBarRopeFull), lane);
      return true;
    };
    // tiles alternate between the two register sets
    for (int i = 0; i < ntiles && ok; i += 2) {
      ok = tile(i, rawA, slotA, rawB, slotB);
      if (tid == 0 && i < 4) NVMLA_TRACE_POINT(14 + i);
      if (ok && i + 1 < ntiles) ok = tile(i + 1, rawB, slotB, rawA, slotA);
      if (tid == 0 && i + 1 < 4) NVMLA_TRACE_POINT(15 + i);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int sw = warp - kSoftmaxWarp0;  // 0..3 = TMEM lane quadrant
    const int k = sw * 32 + lane;          // row of this thread
    const bool issuer = tid == kUnpackThreads;
    // slot list of this thread's row in the later tiles
    {
      const int64_t limit = limit_of();
      int32_t pos[kMaxTiles];
#pragma unroll
      for (int i = 1; i < kMaxTiles; ++i) {
        const int key = kbeg + i * kTile + k;
        pos[i] = (i < ntiles && key < kend) ? ldg_nc_s32(idx_row + key) : -1;
      }
#pragma unroll
      for (int i = 1; i < kMaxTiles; ++i)
        if (i < ntiles) slots[i * kTile + k] = slot_of_pos(pos[i], limit, blockIdx.z == 0);
      warp_arrive(bar(kBarSlots), lane);
    }
    constexpr uint32_t idesc_qk = idesc_f16(false, false);
    constexpr uint32_t idesc_pv = idesc_f16(true, true);
    const uint32_t lb = sbase + kOffL, rb = sbase + kOffR, qb = sbase + kOffQ;
    // QK of one tile, issued by one thread: latent chunk pairs as they land,
    // then the RoPE chunk
    auto issue_qk = [&](int i) -> bool {
      const uint32_t par = i & 1;
      if (i == 0 && !wait_bar(bar(kBarQReady), 0, abort_flag, p.err_word)) return false;
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

    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    float lp[64];  // this row's share of every head's sum
#pragma unroll
    for (int h = 0; h < 64; ++h) lp[h] = 0.f;
    bool ok = !softmax_sync_or(*abort_flag != 0);
    // the issuer's outcome is made uniform across its warp before any
    // warp-collective operation
    auto issued = [&](bool mine) -> bool { return __shfl_sync(0xffffffffu, mine, 0); };
    for (int i = 0; i < ntiles && ok; ++i) {
      bool okq = true;
      if (issuer) okq = issue_qk(i);
      ok = issued(okq);
      if (ok) ok = wait_bar_warp(bar(kBarSFull), i & 1, abort_flag, p.err_word);
      if (softmax_sync_or(!ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(21 + 3 * i);
      const bool valid = slots[i * kTile + k] >= 0;
      float s[64];
      tmem_ld64f(tmem + lane_base + kColS, s);
      if (tid == 256 && i < 2) NVMLA_TRACE_POINT(50 + 8 * i);
#pragma unroll
      for (int h = 0; h < 64; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
      // does any score exceed its head's running maximum by more than 2^tau?
      float excess = -INFINITY;
      if (valid) {
#pragma unroll
        for (int h = 0; h < 64; ++h) excess = fmaxf(excess, s[h] - m_run[h]);
      }
      const bool slow = softmax_sync_or(excess > kTau);
      if (tid == 256 && i < 2) NVMLA_TRACE_POINT(51 + 8 * i);
      if (slow) {
        // exact per-head maximum of this tile (destroys s; reloaded below)
        warp_reduce64<true>(s, lane);
        if (tid == 256 && i < 2) NVMLA_TRACE_POINT(52 + 8 * i);
        red[sw * 64 + 2 * lane] = s[0];
        red[sw * 64 + 2 * lane + 1] = s[1];
        softmax_sync();
        if (tid == 256 && i < 2) NVMLA_TRACE_POINT(53 + 8 * i);
        if (sw < 2) {
          const int h = k;
          const float mt = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
          const float mo = m_run[h];
          const float mn = fmaxf(mo, mt);
          alpha_s[h] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
          m_run[h] = mn;
        }
        softmax_sync();
        if (tid == 256 && i < 2) NVMLA_TRACE_POINT(54 + 8 * i);
#pragma unroll
        for (int h = 0; h < 64; ++h) lp[h] *= alpha_s[h];
        if (i >= 1) {
          // O^T holds the finished PV of the earlier tiles (QK of this tile
          // could only start after the last of them); 16 columns at a time
#pragma unroll 1
          for (int jq = 0; jq < 16; ++jq) {
            const uint32_t ta = tmem + lane_base + kColO + 16 * jq;
            uint32_t orr[16];
            NVMLA_TMEM_LD16(ta, orr, 0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const float* al = alpha_s + 16 * (jq & 3);
#pragma unroll
            for (int e = 0; e < 16; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * al[e]);
            NVMLA_TMEM_ST16(ta, orr, 0);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        if (tid == 256 && i < 2) NVMLA_TRACE_POINT(55 + 8 * i);
        tmem_ld64f(tmem + lane_base + kColS, s);
#pragma unroll
        for (int h = 0; h < 64; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
        if (tid == 256 && i < 2) NVMLA_TRACE_POINT(56 + 8 * i);
      }
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(22 + 3 * i);
      // P = 2^(s - m); masked rows give 0
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float pv = valid ? ex2(s[h] - m_run[h]) : 0.f;
        s[h] = pv;
        lp[h] += pv;
      }
      // P^T row -> the RoPE chunk's place (QK of this tile is complete)
      uint8_t* pt = smem + kOffR;
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
      tc_fence_before();
      warp_arrive(bar(kBarPFull), lane);
      if (tid == 256 && i < 4) NVMLA_TRACE_POINT(23 + 3 * i);
      bool okp = true;
      if (issuer) okp = issue_pv(i);
      ok = issued(okp);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && ntiles > 0) ok = wait_bar_warp(bar(kBarODone), (ntiles - 1) & 1, abort_flag, p.err_word);
    ok = !softmax_sync_or(!ok);
    if (tid == 256) NVMLA_TRACE_POINT(33);
    if (ok) {
      // row sums of every head, reduced across the 128 rows
      warp_reduce64<false>(lp, lane);
      red[sw * 64 + 2 * lane] = lp[0];
      red[sw * 64 + 2 * lane + 1] = lp[1];
      softmax_sync();
      if (sw < 2) {
        const float l = (red[k] + red[64 + k]) + (red[128 + k] + red[192 + k]);
        lsum[k] = l;
        alpha_s[k] = l > 0.f ? 1.f / l : 0.f;  // reused: 1 / l of every head
      }
      softmax_sync();
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
#pragma unroll
          for (int h = 0; h < 64; ++h)
            p.out[(tok * p.H + h0 + h) * kLatent + dv] = __float2bfloat16_rn(__uint_as_float(orr[h]) * alpha_s[h]);
        } else {
          // normalised partial o = O / l as fp16, 64 heads of one value dim
          // contiguous: eight 16-byte stores
          __half* dst = p.ws_o16 + ((tok * p.num_splits + split) * kLatent + dv) * p.H + h0;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int h = 8 * c + 2 * e;
              w4[e] = pack_f16x2(__uint_as_float(orr[h]) * alpha_s[h], __uint_as_float(orr[h + 1]) * alpha_s[h + 1]);
            }
            reinterpret_cast<uint4*>(dst)[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (sw < 2) {
        const int h = k;
        const float m = m_run[h], l = lsum[h];
        if (p.num_splits == 1) {
          p.lse[tok * p.H + h0 + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        } else {
          const int64_t base = (tok * p.num_splits + split) * p.H + h0;
          p.ws_ml[(base + h) * 2] = l > 0.f ? m : -INFINITY;
          p.ws_ml[(base + h) * 2 + 1] = l;
        }
      }
    }
    if (tid == 256) NVMLA_TRACE_POINT(35);
    if (issuer) {
      // every MMA issued has finished once this commit lands
      mma_commit(bar(kBarDrain));
      wait_bar_drain(bar(kBarDrain), 0);
    }
    tc_fence_before();
  }

  __syncthreads();
  if (tid == 0) NVMLA_TRACE_POINT(34);
  if (warp == kAllocWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Merge of the fp16 partials of S key splits for one (token, 64-head block,
// 32 value dims): with M = max_s m_s, L = sum_s l_s 2^(m_s - M) and
// w_s = l_s 2^(m_s - M) / L, out[h][d] = sum_s w_s o_s[d][h] (bf16) and
// lse = (M + log2 L) ln 2 (written by the first dim block).
constexpr int kMergeDims = 32;
__global__ void __launch_bounds__(256) merge_tc_kernel(const __half* __restrict__ ws_o16,
                                                       const float* __restrict__ ws_ml, int S, int H,
                                                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  __shared__ float wgt[kMaxTiles][kHeads];
  __shared__ float tileo[kMergeDims][kHeads + 1];
  const int t = blockIdx.x, h0 = blockIdx.y * kHeads, d0 = blockIdx.z * kMergeDims, tid = threadIdx.x;
  if (tid < kHeads) {
    const int h = h0 + tid;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ws_ml[((static_cast<int64_t>(t) * S + s) * H + h) * 2]);
    float L = 0.f;
    for (int s = 0; s < S; ++s) {
      const float2 ml = *reinterpret_cast<const float2*>(ws_ml + ((static_cast<int64_t>(t) * S + s) * H + h) * 2);
      const float w = (ml.x == -INFINITY) ? 0.f : ml.y * exp2f(ml.x - M);
      wgt[s][tid] = w;
      L += w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = 0; s < S; ++s) wgt[s][tid] *= inv;
    if (blockIdx.z == 0) lse[static_cast<int64_t>(t) * H + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  // thread (d = tid / 8, heads 8 (tid % 8) .. +7)
  const int dl = tid >> 3, hq = (tid & 7) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < S; ++s) {
    const uint4 v = *reinterpret_cast<const uint4*>(ws_o16 + ((static_cast<int64_t>(t) * S + s) * kLatent + d0 + dl) * H +
                                                    h0 + hq);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h2 = *reinterpret_cast<const __half2*>(&w[e]);
      const float2 f = __half22float2(h2);
      acc[2 * e] += wgt[s][hq + 2 * e] * f.x;
      acc[2 * e + 1] += wgt[s][hq + 2 * e + 1] * f.y;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) tileo[dl][hq + e] = acc[e];
  __syncthreads();
  // transposed write: thread (head h = tid / 4, dims 8 (tid % 4) .. +7)
  const int h = tid >> 2, dq = (tid & 3) * 8;
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(tileo[dq + 2 * e][h], tileo[dq + 2 * e + 1][h]);
    o[e] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(out + (static_cast<int64_t>(t) * H + h0 + h) * kLatent + d0 + dq) =
      make_uint4(o[0], o[1], o[2], o[3]);
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
  return static_cast<size_t>(T) * splits * H * (kLatent * sizeof(__half) + 2 * sizeof(float));
}

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
  p.ws_o16 = static_cast<__half*>(workspace);
  p.ws_ml = splits > 1 ? reinterpret_cast<float*>(p.ws_o16 + static_cast<size_t>(T) * splits * H * kLatent) : nullptr;
  p.err_word = err_word;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc::decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(splits, T, H / tc::kHeads);
  tc::decode_tc_kernel<<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  tc::merge_tc_kernel<<<dim3(T, H / tc::kHeads, kLatent / tc::kMergeDims), 256, 0, stream>>>(p.ws_o16, p.ws_ml, splits,
                                                                                              H, p.out, lse);
  return cudaGetLastError();
}

}  // namespace nvmla

#ifdef NVMLA_TRACE
extern "C" int nvmla_tc_trace_read(void* host_dst, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(host_dst, nvmla::tc::nvmla_tc_trace, bytes));
}
#endif
