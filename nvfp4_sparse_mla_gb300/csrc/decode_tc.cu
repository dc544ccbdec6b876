// Sparse MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: "Prime Inference: Fast, Reliable Serving for Frontier
// Open Models", section "A native NVFP4 sparse-MLA decode kernel" -- for each
// query token only the rows the indexer selected are loaded, unpacked on chip
// and attended to with FP16 operands and FP32 accumulation, with no FP8
// staging buffer in GPU memory; the token's selected rows are divided among a
// cluster of cooperating CTAs whose partial results are combined through
// distributed shared memory in the same launch. "Prime Intellect unveils
// Prime Inference", section "4-bit caches open the way": item 1 (one group of
// warps unpacks rows while the tensor core computes scores and accumulates),
// item 3 (empty slots of the 2048-slot list contribute nothing).
//
// One cluster = one query token x 64 heads; its S CTAs take contiguous
// ranges of the token's slots, in tiles of 128 rows. Both contractions run as
// tcgen05.mma kind::f16 (M = 128, N = 64, K = 16) in swap-AB orientation, the
// 64 heads being N (an M = 64 instruction takes as long as an M = 128 one):
//   S^T[128 rows, 64 heads]  = K[128 x 576] . Q^T    A: latent K in shared memory,
//                                                    RoPE K in TMEM; B: Q^T
//   O^T[512 dims, 64 heads] += V^T[512 x 128] . P^T  A: V^T (the same latent
//                                                    tile, read MN-major); B: P^T
// The latent part of a row is unpacked once, into a 128B-swizzled K-major
// tile in shared memory: read K-major it is QK's A operand, read MN-major it
// is V^T for PV. TMEM (512 columns): S^T in 0-63, O^T in 64-319 (block j =
// dims 128j..128j+127), the tile's RoPE K in 320-351.
//
// Roles (16 warps, 128 registers a thread; a 17th warp would put five warps
// on one SM sub-partition and cap every thread at 96 registers):
//   every warp  warp w owns TMEM lane quadrant w & 3 and quarter u = w >> 2:
//               thread (row r = 32 (w & 3) + lane, quarter u) holds a quarter
//               of cache row r -- latent dims 128u..128u+127 (the code bytes
//               and their 8 scales) and RoPE dims 16u..16u+15 -- and writes
//               them as fp16 (E2M1 x E4M3 is exact in fp16): the latent into
//               chunks 2u, 2u+1 of the tile, the RoPE values into TMEM. The
//               same thread then runs the softmax of row r for heads
//               16u..16u+15: S^T from TMEM, P^T to shared memory.
//   warp 15     also allocates TMEM, and its lane 0 issues every MMA between
//               its own steps: a tile's 36 QK MMAs right after the warp's
//               part of the tile is written, the 32 PV MMAs (four blocks of
//               128 value dims, each committed on its own so that the next
//               tile's unpack refills that block's two chunks while the later
//               blocks run) right after its share of P^T. The warp unpacks
//               quarter 3, which waits for the last PV block in any case.
//
// Start-up: the slot-list entries, then the query block straight into
// registers (converted to fp16 Q^T while the rows are on their way), then
// the block-table entries; the first tile's rows come by one TMA bulk copy
// each into the latent tile's space, the next tiles' rows are prefetched
// into L2. Per tile the order is unpack -> QK -> softmax -> PV; a later
// tile's rows are requested into registers after a softmax (NVFP4: two tiles
// ahead), and a tile's unpack overlaps the previous PV block by block.
//
// Softmax: the running maximum of a head starts, on the first tile, at the
// largest score of rows 0, 32, 64 and 96 and stays fixed while no score
// exceeds it by more than 2^15 (P below 2^15 is safe in fp16); a tile that
// does pays for the exact maximum and rescales O^T in TMEM. Row sums
// accumulate per thread and are reduced once, at the end.
//
// Combine: a token's only CTA writes out / lse itself. With S CTAs each
// stages its normalised partial O / l (fp16, [512 dims][64 heads]) and its
// per-head (m, l) in its own shared memory; after one cluster barrier CTA r
// reads its share of the value dims from every CTA of the cluster with
// distributed-shared-memory loads, weights them by l_s 2^(m_s - M) / L and
// writes bf16 out (rank 0 also writes lse). No global workspace is used.
//
// Every mbarrier wait is bounded: on timeout the CTA sets
// NVMLA_ERRW_WAIT_TIMEOUT, the MMA issuer drains its MMAs, and every thread
// still takes part in the same cluster barriers, so that every CTA exits.
#include "common.cuh"
#include "decode_tc_layout.h"

// A build with -DNVMLA_DEBUG_BOUNDS checks every data-dependent index of the
// kernel (cache rows, block-table and slot-list entries, output positions,
// tile and split counts) against its buffer and records a failure as
// NVMLA_ERRW_BOUNDS in err_word; the shared-memory and TMEM offsets come
// from decode_tc_layout.h, which a host-compiled test checks exhaustively.
// The default build compiles the checks away.
#ifdef NVMLA_DEBUG_BOUNDS
#define NVMLA_CHECK(cond)                                                \
  do {                                                                   \
    if (!(cond)) report_error(p.err_word, NVMLA_ERRW_BOUNDS, 1);          \
  } while (0)
#else
#define NVMLA_CHECK(cond) \
  do {                    \
  } while (0)
#endif

#include <atomic>
#include <mutex>

namespace nvmla {

namespace tc {

// Optional timeline instrumentation: a build with -DNVMLA_TRACE records
// %globaltimer at fixed points of each CTA's schedule into nvmla_tc_trace
// (read back with nvmla_tc_trace_read). Off by default: no code is emitted.
#ifdef NVMLA_TRACE
constexpr int kTraceCtas = 2048;
constexpr int kTracePoints = 64;
__device__ unsigned long long nvmla_tc_trace[kTraceCtas][kTracePoints];
#define NVMLA_TRACE_POINT(id)                                                                       \
  do {                                                                                              \
    const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                 \
    if (cta_ < kTraceCtas) {                                                                        \
      unsigned long long t_;                                                                        \
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t_));                                         \
      nvmla_tc_trace[cta_][(id)] = t_;                                                              \
    }                                                                                               \
  } while (0)
// the same, once the 32-bit value v is available
#define NVMLA_TRACE_AFTER(id, v)                                                                    \
  do {                                                                                              \
    const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                 \
    if (cta_ < kTraceCtas) {                                                                        \
      unsigned long long t_;                                                                        \
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t_) : "r"(v));                               \
      nvmla_tc_trace[cta_][(id)] = t_;                                                              \
    }                                                                                               \
  } while (0)
// a value instead of the time
#define NVMLA_TRACE_VALUE(id, v)                                                                    \
  do {                                                                                              \
    const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                 \
    if (cta_ < kTraceCtas) nvmla_tc_trace[cta_][(id)] = (v);                                        \
  } while (0)
// tiles whose schedule is recorded: the first and NVMLA_TRACE_TILE (1 unless
// the build sets it)
#ifndef NVMLA_TRACE_TILE
#define NVMLA_TRACE_TILE 1
#endif
#define NVMLA_TRACED_TILE(i) ((i) == 0 || (i) == NVMLA_TRACE_TILE)
#define NVMLA_TRACE_SLOT(i) ((i) == 0 ? 0 : 1)
#else
#define NVMLA_TRACE_TILE (-1)
#define NVMLA_TRACED_TILE(i) false
#define NVMLA_TRACE_SLOT(i) 0
#define NVMLA_TRACE_POINT(id) \
  do {                        \
  } while (0)
#define NVMLA_TRACE_AFTER(id, v) \
  do {                           \
  } while (0)
#define NVMLA_TRACE_VALUE(id, v) \
  do {                           \
  } while (0)
#endif

constexpr int kPrefetchAhead = 3;       // tiles whose rows are prefetched into L2 ahead of use
constexpr float kTau = 15.0f;           // rescale threshold, log2 units: P < 2^15 fits fp16
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
// (the shared-memory and TMEM layout, and every offset into them, are in
// decode_tc_layout.h)

struct Params {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_rope;
  const uint8_t* cache;
  RowSelect sel;
  int T, H, topk;
  float sl2;
  __nv_bfloat16* out;
  float* lse;
  int num_splits;     // == cluster size
  int tiles_total;
  int32_t* err_word;
  uint32_t p_wait_ns;  // limit of the MMA issuer's wait for P^T; 0 = the default
  int force_p_timeout; // test hook: that wait gives up at once
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
// try_wait until the phase completes; the loop gives up after `limit_ns` of
// wall time, raising the CTA's abort flag and NVMLA_ERRW_WAIT_TIMEOUT.
// Also returns false once another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err_word,
                                         uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint32_t hint = limit_ns < 100000u ? static_cast<uint32_t>(limit_ns) : 100000u;
  while (true) {
    if (mbar_wait_hint(bar, parity, hint)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
  if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) report_error(err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  return false;
}

// A wait that gives up at once (the test hook for the abort path).
__device__ __forceinline__ bool give_up(volatile int* abort_flag, int32_t* err_word) {
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

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Runs of MMAs along K in one asm statement, so that the compiler keeps only
// the two base descriptors live instead of one pair per MMA: the descriptors
// of step k are the bases plus kOffA / kOffB (16-byte units) plus k times the
// per-step advance (the start-address field sits in the low bits and no run
// crosses 256 KB, so the adds never carry out of it). The first MMA
// overwrites D when acc0 is 0; the others accumulate.
// QK over one 64-dim chunk: 4 steps of 32 bytes in A (K-major) and B.
template <int kOffA, int kOffB>
__device__ __forceinline__ void mma_chunk_qk(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a0, a1, a2, a3, b0, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 q, %3, %3;\n\t"
      "add.s64 a0, %1, %5;\n\tadd.s64 a1, a0, 2;\n\tadd.s64 a2, a0, 4;\n\tadd.s64 a3, a0, 6;\n\t"
      "add.s64 b0, %2, %6;\n\tadd.s64 b1, b0, 2;\n\tadd.s64 b2, b0, 4;\n\tadd.s64 b3, b0, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a0, b0, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc0), "n"(kOffA), "n"(kOffB)
      : "memory");
}
// QK over the RoPE chunk with A in TMEM: 4 steps of 8 columns in A, 32
// bytes in B; always accumulates.
template <int kOffB>
__device__ __forceinline__ void mma_chunk_qk_tmem(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b0, b1, b2, b3;\n\t"
      "setp.eq.b32 q, %3, %3;\n\t"
      "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
      "add.s64 b0, %2, %4;\n\tadd.s64 b1, b0, 2;\n\tadd.s64 b2, b0, 4;\n\tadd.s64 b3, b0, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b0, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "n"(kOffB)
      : "memory");
}
// PV over one block of 128 value dims: 8 steps of 16 rows = 2048 bytes
// (128 units) in A (MN-major V^T) and B (MN-major P^T).
template <int kOffA>
__device__ __forceinline__ void mma_block_pv(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a0, a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 q, %3, %3;\n\t"
      "add.s64 a0, %1, %5;\n\tadd.s64 a1, a0, 128;\n\tadd.s64 a2, a0, 256;\n\tadd.s64 a3, a0, 384;\n\t"
      "add.s64 a4, a0, 512;\n\tadd.s64 a5, a0, 640;\n\tadd.s64 a6, a0, 768;\n\tadd.s64 a7, a0, 896;\n\t"
      "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
      "add.s64 b4, %2, 512;\n\tadd.s64 b5, %2, 640;\n\tadd.s64 b6, %2, 768;\n\tadd.s64 b7, %2, 896;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a0, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, q;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc0), "n"(kOffA)
      : "memory");
}

#define NVMLA_TMEM_LD16F(taddr, r, o)                                                                         \
  asm volatile(                                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
      : "=f"(r[o + 0]), "=f"(r[o + 1]), "=f"(r[o + 2]), "=f"(r[o + 3]), "=f"(r[o + 4]), "=f"(r[o + 5]),       \
        "=f"(r[o + 6]), "=f"(r[o + 7]), "=f"(r[o + 8]), "=f"(r[o + 9]), "=f"(r[o + 10]), "=f"(r[o + 11]),     \
        "=f"(r[o + 12]), "=f"(r[o + 13]), "=f"(r[o + 14]), "=f"(r[o + 15])                                    \
      : "r"(taddr))

#define NVMLA_TMEM_ST16F(taddr, r, o)                                                                         \
  asm volatile(                                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" \
      ::"r"(taddr), "f"(r[o + 0]), "f"(r[o + 1]), "f"(r[o + 2]), "f"(r[o + 3]), "f"(r[o + 4]), "f"(r[o + 5]), \
      "f"(r[o + 6]), "f"(r[o + 7]), "f"(r[o + 8]), "f"(r[o + 9]), "f"(r[o + 10]), "f"(r[o + 11]),              \
      "f"(r[o + 12]), "f"(r[o + 13]), "f"(r[o + 14]), "f"(r[o + 15])                                          \
      : "memory")

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&w)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 16 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&r)[16]) {
  NVMLA_TMEM_LD16F(taddr, r, 0);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// named barrier among the 512 worker threads (id 1); the _or form returns
// the OR of a predicate over the group (used to make the outcome of a
// bounded wait, or a data-dependent branch, uniform)
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ bool workers_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 512, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// maximum over the warp (every lane gets it)
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


// ---- cluster rank, a barrier over every thread of every CTA with release /
// acquire semantics at cluster scope, and distributed-shared-memory loads
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// ---- TMA bulk copy (1-D): addresses 16-byte aligned, sizes multiples of 16
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(bar)
               : "memory");
}

// fire-and-forget prefetch of a row into L2 (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- global loads (read-only path); volatile so that they are issued where
// they stand, as soon as their registers are free
__device__ __forceinline__ void ldg_nc_v8(const void* p, uint32_t* v) {
  asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}
__device__ __forceinline__ void ldg_nc_v4(const void* p, uint32_t* v) {
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "l"(p));
}
__device__ __forceinline__ void ldg_nc_v2(const void* p, uint32_t* v) {
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "l"(p));
}
__device__ __forceinline__ int32_t ldg_nc_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// The cache's row format: 352-byte NVFP4 rows, or 576-byte FP8 rows (512
// latent + 64 RoPE E4M3 values, no scales).
enum RowFmt { kFmtNvfp4 = 0, kFmtFp8 = 1 };

// A worker's quarter of one cache row, as loaded: latent dims 128u..128u+127
// and RoPE dims 16u..16u+15.
template <int FMT>
struct Quarter;
template <>
struct Quarter<kFmtNvfp4> {
  uint32_t c[16];  // 64 code bytes: words 0-7 = dims 128u..+63, words 8-15 = +64..+127
  uint32_t sc[2];  // 8 scale bytes: groups 8u..8u+7
  uint32_t rr[4];  // 16 RoPE bytes
};
template <>
struct Quarter<kFmtFp8> {
  uint32_t c[32];  // 128 E4M3 bytes: words 0-15 = dims 128u..+63, 16-31 = +64..+127
  uint32_t rr[4];  // 16 RoPE bytes
};

template <int FMT>
__device__ __forceinline__ void load_quarter(Quarter<FMT>& q, const uint8_t* row, int u) {
  if constexpr (FMT == kFmtFp8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) ldg_nc_v8(row + 128 * u + 32 * j, q.c + 8 * j);
    ldg_nc_v4(row + kLatent + 16 * u, q.rr);
  } else {
    ldg_nc_v8(row + 64 * u, q.c);
    ldg_nc_v8(row + 64 * u + 32, q.c + 8);
    ldg_nc_v2(row + kScaleOff + 8 * u, q.sc);
    ldg_nc_v4(row + kRopeOff + 16 * u, q.rr);
  }
}

// Latent chunk 2u + h2 of row r (64 dims) as fp16 into the tile, zeros for a
// masked row. Piece p (16 bytes) of the row holds dims 8p..8p+7.
template <int FMT>
__device__ __forceinline__ void store_chunk(const Quarter<FMT>& q, int h2, bool valid, uint8_t* chunk, int r) {
  if constexpr (FMT == kFmtFp8) {
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) {
      uint32_t w[4];
      e4m3x4_to_f16x4(q.c[16 * h2 + 2 * pc], w[0], w[1]);
      e4m3x4_to_f16x4(q.c[16 * h2 + 2 * pc + 1], w[2], w[3]);
      const uint4 v = valid ? make_uint4(w[0], w[1], w[2], w[3]) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(chunk + swz(r, pc)) = v;
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t s2 = e4m3_to_f16x2_bcast((q.sc[h2] >> (8 * g)) & 0xffu);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        uint32_t h[4];
        e2m1x8_to_f16x8(q.c[8 * h2 + 2 * g + e], h);
        const uint4 v = valid ? make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2),
                                           hmul2_u32(h[3], s2))
                              : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(chunk + swz(r, 2 * g + e)) = v;
      }
    }
  }
}

// RoPE dims 16u..16u+15 of the row as fp16 into TMEM columns kColR + 8u..+7
// of this thread's lane (zeros for a masked row)
template <int FMT>
__device__ __forceinline__ void store_rope(const Quarter<FMT>& q, bool valid, uint32_t taddr) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t lo, hi;
    e4m3x4_to_f16x4(q.rr[j], lo, hi);
    w[2 * j] = valid ? lo : 0u;
    w[2 * j + 1] = valid ? hi : 0u;
  }
  tmem_st8(taddr, w);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const Params p) {
  constexpr int kRB = FMT == kFmtFp8 ? kFp8RowBytes : kRowBytes;  // bytes per cache row
  constexpr int kRawPitch = FMT == kFmtFp8 ? kRawPitchFp8 : kRawPitchNvfp4;  // first-tile rows in shared memory
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

  const int kbeg = tile_lo(static_cast<int>(rank), S, p.tiles_total) * kTile;
  const int kend = min(tile_lo(static_cast<int>(rank) + 1, S, p.tiles_total) * kTile, p.topk);
  const int nkeys = max(0, kend - kbeg);
  const int ntiles = (nkeys + kTile - 1) / kTile;  // <= kMaxTiles (host check)

  if (tid == 0) NVMLA_TRACE_POINT(0);

  const int quad = warp & 3, qu = warp >> 2;  // TMEM lane quadrant, row quarter
  const int r = quad * 32 + lane;             // row of the tile
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  const bool report = blockIdx.z == 0;               // one head block reports bad entries

  // ---- start-up, level 1: the token's sequence and slot-list entries
  const int32_t seq_raw = p.sel.q_seq_idx ? ldg_nc_s32(p.sel.q_seq_idx + t) : 0;
  const int32_t* tk_row = p.sel.topk_idx + static_cast<int64_t>(t) * p.topk;
  int32_t pos0 = -1;
  constexpr int kLaterPer = kMaxTiles / 4;  // later tiles per worker thread
  int32_t posl[kLaterPer];
  {
    NVMLA_CHECK(S >= 1 && S <= kMaxCluster && ntiles >= 0 && ntiles <= kMaxTiles && kbeg >= 0 && kend <= p.topk);
    if (kbeg + r < kend) pos0 = ldg_nc_s32(tk_row + kbeg + r);
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + qu + 4 * m;
      const int key = kbeg + i * kTile + r;
      if (i < ntiles && key < kend) NVMLA_CHECK(key >= 0 && key < p.topk && i < kMaxTiles);
      posl[m] = (i < ntiles && key < kend) ? ldg_nc_s32(tk_row + key) : -1;
    }
  }
  // ---- the query block (bf16, 64 KB latent + 8 KB RoPE for the CTA's 64
  // heads, each part contiguous in global memory), requested right after the
  // slot-list entries, straight into registers: 16-byte unit u = tid + 512 m
  // (m < 8) of the latent part, unit tid of the RoPE part. It is converted
  // to fp16 Q^T while the first tile's rows are on their way; the TMA unit
  // is left to those rows.
  uint32_t qv[9][4];
  {
    const int64_t qh0 = static_cast<int64_t>(t) * p.H + h0;
    const uint8_t* ql = reinterpret_cast<const uint8_t*>(p.q_latent + qh0 * kLatent);
    const uint8_t* qr = reinterpret_cast<const uint8_t*>(p.q_rope + qh0 * kRope);
#pragma unroll
    for (int m = 0; m < 8; ++m) ldg_nc_v4(ql + q_src_off(tid, m), qv[m]);
    ldg_nc_v4(qr + q_src_off(tid, 8), qv[8]);
  }
  static_assert(kQBytes == 9 * kThreads * 16, "nine 16-byte units of the query block per thread");
  if (tid == 0) {
    mbar_init(bar(kBarRows0), kTile);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the first tile's row barrier is initialised before any thread arrives on it
  __syncthreads();
  // ---- level 2: block-table entries (page index clamped into the row, so
  // the load is in bounds whatever the entry) and the sequence length
  const bool seq_ok = seq_raw >= 0 && seq_raw < p.sel.num_seqs;
  const int32_t seq = seq_ok ? seq_raw : 0;
  const int32_t* bt_row = p.sel.block_table + static_cast<int64_t>(seq) * p.sel.max_pages;
  auto page_of = [&](int32_t pos) -> int32_t {
    const int32_t pi = min(max(pos >> 6, 0), p.sel.max_pages - 1);
    NVMLA_CHECK(pi >= 0 && pi < p.sel.max_pages && seq >= 0 && seq < p.sel.num_seqs);
    return ldg_nc_s32(bt_row + pi);
  };
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
  auto row_of = [&](int32_t slot) {
    NVMLA_CHECK(slot >= 0 && slot < p.sel.num_slots);
    return p.cache + cache_row_offset(slot, p.sel.page_rows, kRB);
  };
  int32_t page0 = 0;
  int32_t pagel[kLaterPer];
  if (tid == 0) NVMLA_TRACE_AFTER(25, pos0);
  {
    page0 = page_of(pos0);
    if (tid == 0) NVMLA_TRACE_AFTER(26, page0);
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) pagel[m] = (1 + qu + 4 * m < ntiles) ? page_of(posl[m]) : 0;
  }
  int64_t limit = static_cast<int64_t>(p.sel.max_pages) * kPage;
  if (p.sel.seq_lens) {
    const int64_t L = ldg_nc_s32(p.sel.seq_lens + seq);
    limit = L < limit ? L : limit;
  }
  if (tid == 0) NVMLA_TRACE_AFTER(27, static_cast<int32_t>(limit));

  // ---- level 3: the first tile's rows, one TMA bulk copy per row into
  // shared memory, issued by the row's quarter-0 thread; the later tiles'
  // slots into shared memory, their rows prefetched into L2
  Quarter<FMT> raw;   // the row quarter of the tile unpacked next
  Quarter<FMT> rawn;  // NVFP4: the one after it, requested a tile ahead
  int32_t slot0 = -1;
  {
    const bool mine = ntiles > 0 && kbeg + r < kend;
    const int32_t sspec = mine ? phys_slot(pos0, page0) : -1;
    if (qu == 0) {
      // the barrier must see this thread's arrival before the copy's bytes
      if (sspec >= 0) {
        mbar_arrive_expect_tx(bar(kBarRows0), kRB);
        bulk_load(sbase + raw_row_off(r, kRawPitch), row_of(sspec), kRB, bar(kBarRows0));
      } else {
        mbar_arrive(bar(kBarRows0));
      }
    }
    if (tid == 0) NVMLA_TRACE_POINT(28);
    if (mine) slot0 = classify(pos0, page0, limit, report && qu == 0);
    if (qu == 0) slots[slot_index(0, r)] = slot0;
#pragma unroll
    for (int m = 0; m < kLaterPer; ++m) {
      const int i = 1 + qu + 4 * m;
      if (i < ntiles) {
        const int32_t sl = classify(posl[m], pagel[m], limit, report);
        slots[slot_index(i, r)] = sl;
        // the rows of the next three tiles into L2 now, the later ones three
        // tiles ahead of their use (all at once, they would flood the memory
        // system at start-up when a CTA has many tiles)
        if (sl >= 0 && i <= kPrefetchAhead) prefetch_l2(row_of(sl), kRB);
      }
    }
  }
  if (tid == 0) NVMLA_TRACE_POINT(1);

  // ---- setup: barriers, TMEM
  if (tid == kThreads - 1) {
    mbar_init(bar(kBarKV), 16);
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarP), 16);
    for (int j = 0; j < 4; ++j) mbar_init(bar(kBarPV + j), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = (sbase & 1023u) ? 1 : 0;  // swizzled operands need a 1 KB aligned base
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kHeads) m_run[tid] = -INFINITY;
  if (warp == kMmaWarp) {
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
  if (*abort_flag && tid == 0) report_error(p.err_word, NVMLA_ERRW_WAIT_TIMEOUT, 1);
  bool ok = *abort_flag == 0;

  {
    // ------------------------------------------------------------ workers
    // ---- the query block -> fp16 Q^T, K-major 128B-swizzled: latent unit
    // u holds head u / 64, dims 8 (u % 64)..+7 (query chunk (u % 64) / 8);
    // RoPE unit u holds head u / 8, RoPE dims 8 (u % 8)..+7 (query chunk 8)
#pragma unroll
    for (int m = 0; m < 9; ++m) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[e] = pack_f16x2(bf16_bits_to_f32(qv[m][e] & 0xffffu), bf16_bits_to_f32(qv[m][e] >> 16));
      *reinterpret_cast<uint4*>(smem + q_dst_off(tid, m)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid == 0) NVMLA_TRACE_POINT(3);
    {
      // this thread's quarter of its first-tile row, out of shared memory
      ok = ok && wait_bar_warp(bar(kBarRows0), 0, abort_flag, p.err_word);
      const uint8_t* row = smem + raw_row_off(r, kRawPitch);
      if constexpr (FMT == kFmtFp8) {
        if (ok) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + 128 * qu + 16 * k);
            raw.c[4 * k] = v.x;
            raw.c[4 * k + 1] = v.y;
            raw.c[4 * k + 2] = v.z;
            raw.c[4 * k + 3] = v.w;
          }
          const uint4 rr = *reinterpret_cast<const uint4*>(row + kLatent + 16 * qu);
          raw.rr[0] = rr.x;
          raw.rr[1] = rr.y;
          raw.rr[2] = rr.z;
          raw.rr[3] = rr.w;
        }
      } else if (ok) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(row + 64 * qu);
        const uint4 c1 = *reinterpret_cast<const uint4*>(row + 64 * qu + 16);
        const uint4 c2 = *reinterpret_cast<const uint4*>(row + 64 * qu + 32);
        const uint4 c3 = *reinterpret_cast<const uint4*>(row + 64 * qu + 48);
        const uint2 sc = *reinterpret_cast<const uint2*>(row + kScaleOff + 8 * qu);
        const uint4 rr = *reinterpret_cast<const uint4*>(row + kRopeOff + 16 * qu);
        const uint32_t cw[16] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w,
                                 c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
#pragma unroll
        for (int k = 0; k < 16; ++k) raw.c[k] = cw[k];
        raw.sc[0] = sc.x;
        raw.sc[1] = sc.y;
        raw.rr[0] = rr.x;
        raw.rr[1] = rr.y;
        raw.rr[2] = rr.z;
        raw.rr[3] = rr.w;
      }
    }
    if (tid == 0) NVMLA_TRACE_POINT(29);
    // every worker holds its first-tile row before the tile's space is written
    ok = !workers_sync_or(!ok);
    if (tid == 0) NVMLA_TRACE_POINT(39);

    float lp[16];  // this row's share of its heads' sums
#pragma unroll
    for (int h = 0; h < 16; ++h) lp[h] = 0.f;
    const uint32_t rope_col = tmem + lane_base + r_col(qu);
    const int hb = 16 * qu;  // first head of this thread's softmax share
    // this thread's part of a tile: latent chunks 2qu, 2qu + 1 of row r into
    // the latent tile, its RoPE dims into TMEM
    auto unpack = [&](bool valid) {
      store_chunk<FMT>(raw, 0, valid, smem + latent_chunk_off(2 * qu), r);
      store_chunk<FMT>(raw, 1, valid, smem + latent_chunk_off(2 * qu + 1), r);
      tc_fence_after();
      store_rope<FMT>(raw, valid, rope_col);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    };
    // ---- the first tile
    if (ok && ntiles > 0) unpack(slots[slot_index(0, r)] >= 0);
    if (tid == 0) NVMLA_TRACE_POINT(30);
    if (ok && ntiles > 0) {
      fence_async_smem();
      tc_fence_before();
      warp_arrive(bar(kBarKV), lane);
    }
    // ---- MMA issue, by lane 0 of warp kMmaWarp between its own worker
    // steps: a tile's QK right after the warp's arrival on kBarKV, its PV
    // right after the warp's arrival on kBarP. The warp unpacks quarter 3,
    // which waits for the last PV block of the previous tile in any case.
    // Each run is unrolled straight-line code: a wait or a branch between two
    // tcgen05.mma instructions stalls the issuer for about as long as an MMA.
    const bool issuer = warp == kMmaWarp && lane == 0;
    bool mok = true;  // issuer: no wait of its own has failed
    auto issue_qk = [&](int i) {
      mok = mok && wait_bar(bar(kBarKV), i & 1, abort_flag, p.err_word);
      if (!mok) return;
      tc_fence_after();
      if (NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(7 + 8 * NVMLA_TRACE_SLOT(i));
      // latent chunks c = 0..7 (A: the tile, K-major), then the RoPE K (A:
      // TMEM); query chunk c is the B operand
      constexpr uint32_t idesc_qk = idesc_f16(false, false);
      const uint64_t a_kv = sdesc(sbase + kOffKV, 16, 1024);
      const uint64_t b_q = sdesc(sbase + kOffQ, 16, 1024);
      mma_chunk_qk<0 * 1024, 0 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 0);
      mma_chunk_qk<1 * 1024, 1 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<2 * 1024, 2 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<3 * 1024, 3 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<4 * 1024, 4 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<5 * 1024, 5 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<6 * 1024, 6 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk<7 * 1024, 7 * 512>(tmem + kColS, a_kv, b_q, idesc_qk, 1);
      mma_chunk_qk_tmem<8 * 512>(tmem + kColS, tmem + kColR, b_q, idesc_qk);
      mma_commit(bar(kBarS));
      if (NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(9 + 8 * NVMLA_TRACE_SLOT(i));
    };
    auto issue_pv = [&](int i) {
      const uint64_t p_limit = p.p_wait_ns ? p.p_wait_ns : kWaitLimitNs;
      mok = mok && (p.force_p_timeout ? give_up(abort_flag, p.err_word)
                                      : wait_bar(bar(kBarP), i & 1, abort_flag, p.err_word, p_limit));
      if (!mok) return;
      tc_fence_after();
      if (NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(8 + 8 * NVMLA_TRACE_SLOT(i));
      // block j: value dims 128j..128j+127 = latent chunks 2j, 2j+1 (A: V^T,
      // MN-major, the two 64-dim halves one chunk apart; B: P^T), 8 steps of
      // 16 rows, committed on its own
      constexpr uint32_t idesc_pv = idesc_f16(true, true);
      const uint64_t a_v = sdesc(sbase + kOffKV, kChunkBytes, 1024);
      const uint64_t b_p = sdesc(sbase + kOffP, 8192, 1024);
      const uint32_t acc = i != 0;
      mma_block_pv<0 * 2048>(tmem + kColO + 0 * 64, a_v, b_p, idesc_pv, acc);
      mma_commit(bar(kBarPV + 0));
      mma_block_pv<1 * 2048>(tmem + kColO + 1 * 64, a_v, b_p, idesc_pv, acc);
      mma_commit(bar(kBarPV + 1));
      mma_block_pv<2 * 2048>(tmem + kColO + 2 * 64, a_v, b_p, idesc_pv, acc);
      mma_commit(bar(kBarPV + 2));
      mma_block_pv<3 * 2048>(tmem + kColO + 3 * 64, a_v, b_p, idesc_pv, acc);
      mma_commit(bar(kBarPV + 3));
      if (NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(10 + 8 * NVMLA_TRACE_SLOT(i));
    };
    for (int i = 0; i < ntiles && ok; ++i) {
      const bool valid = slots[slot_index(i, r)] >= 0;
      // ---- unpack tile i: chunks 2qu, 2qu + 1 once PV block qu of the
      // previous tile is done; the RoPE K once QK of the previous tile is
      // done (waited for below, in its softmax)
      bool okw = true;
      if (i >= 1) {
        okw = wait_bar_warp(bar(kBarPV + qu), (i - 1) & 1, abort_flag, p.err_word);
        if (tid == 0 && i == NVMLA_TRACE_TILE) NVMLA_TRACE_POINT(36);
        if (okw) {
          unpack(valid);
          if (tid == 0 && i == NVMLA_TRACE_TILE) NVMLA_TRACE_POINT(37);
          fence_async_smem();
          tc_fence_before();
          warp_arrive(bar(kBarKV), lane);
          if constexpr (FMT == kFmtNvfp4) {
            if (i + 1 < ntiles) raw = rawn;
          }
        }
      }
      if (tid == 0 && NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(4 + 8 * NVMLA_TRACE_SLOT(i));
      // ---- QK of tile i (the other lanes of the issuer's warp wait for it
      // in the warp barrier of the next wait)
      if (issuer && okw) issue_qk(i);
      // ---- softmax of tile i
      if (okw) okw = wait_bar_warp(bar(kBarS), i & 1, abort_flag, p.err_word);
      if (tid == 0 && NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(11 + 8 * NVMLA_TRACE_SLOT(i));
      if (workers_sync_or(!okw)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (tid == 0 && NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(5 + 8 * NVMLA_TRACE_SLOT(i));
      float s[16];
      tmem_ld16f(tmem + lane_base + s_col(hb), s);
#pragma unroll
      for (int h = 0; h < 16; ++h) s[h] = valid ? s[h] * p.sl2 : -INFINITY;
      if (i == 0) {
        // The running maximum starts at the largest of rows 0, 32, 64 and 96
        // (-inf where all four are masked): any value that some score
        // reaches is a valid reference, and the exact reduction below runs
        // only if a score of the tile lies more than 2^tau above it.
        if (lane == 0) {
#pragma unroll
          for (int h4 = 0; h4 < 4; ++h4)
            *reinterpret_cast<float4*>(red + quad * 64 + hb + 4 * h4) =
                make_float4(s[4 * h4], s[4 * h4 + 1], s[4 * h4 + 2], s[4 * h4 + 3]);
        }
        workers_sync();
        if (tid < kHeads) m_run[tid] = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
        workers_sync();
      }
      // does any score exceed its head's running maximum by more than 2^tau?
      float excess = -INFINITY;
      if (valid) {
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4) {
          const float4 m4 = *reinterpret_cast<const float4*>(m_run + hb + 4 * h4);
          excess = fmaxf(excess, fmaxf(fmaxf(s[4 * h4] - m4.x, s[4 * h4 + 1] - m4.y),
                                       fmaxf(s[4 * h4 + 2] - m4.z, s[4 * h4 + 3] - m4.w)));
        }
      }
      const bool slow = workers_sync_or(excess > kTau);
      if (slow) {
        // exact per-head maximum of this tile: warp reductions over the
        // rows, then across the four lane quadrants
        float mine = -INFINITY;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float mh = warp_max(s[h]);
          mine = (lane & 15) == h ? mh : mine;
        }
        if (lane < 16) red[quad * 64 + hb + lane] = mine;
        workers_sync();
        if (tid < kHeads) {
          const float mt = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
          const float mo = m_run[tid];
          const float mn = fmaxf(mo, mt);
          alpha_s[tid] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
          m_run[tid] = mn;
        }
        workers_sync();
#pragma unroll
        for (int h = 0; h < 16; ++h) lp[h] *= alpha_s[hb + h];
      }
      // P = 2^(s - m); masked rows give 0
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
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
      // P^T row r, heads hb..hb+15 (pieces 2qu, 2qu + 1); PV of the previous
      // tile has finished reading the buffer (it precedes this tile's QK)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint4 q4;
        q4.x = pack_f16x2(s[8 * cc + 0], s[8 * cc + 1]);
        q4.y = pack_f16x2(s[8 * cc + 2], s[8 * cc + 3]);
        q4.z = pack_f16x2(s[8 * cc + 4], s[8 * cc + 5]);
        q4.w = pack_f16x2(s[8 * cc + 6], s[8 * cc + 7]);
        *reinterpret_cast<uint4*>(smem + pt_off(r, 2 * qu + cc)) = q4;
      }
      if (slow && i >= 1) {
        // O^T to the new maximum: it holds the finished PV of every earlier
        // tile (QK of this tile was issued after it, and its commit has been
        // waited for); PV of this tile starts only after kBarP
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const uint32_t col = tmem + lane_base + o_col(j, hb);
          float o[16];
          tmem_ld16f(col, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= alpha_s[hb + e];
          NVMLA_TMEM_ST16F(col, o, 0);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      fence_async_smem();
      tc_fence_before();
      warp_arrive(bar(kBarP), lane);
      // ---- a later tile's rows into L2, kPrefetchAhead tiles ahead
      if (qu == 0 && i + 1 + kPrefetchAhead < ntiles) {
        const int32_t ps = slots[slot_index(i + 1 + kPrefetchAhead, r)];
        if (ps >= 0) prefetch_l2(row_of(ps), kRB);
      }
      // ---- rows of later tiles, requested after the softmax so that they do
      // not land during this tile's QK (the MMAs read their operands from
      // shared memory, and returning loads slow them). NVFP4 keeps two tiles
      // in flight: after the first softmax the next two tiles' rows, then
      // each time the one two tiles ahead (the next is already in raw); the
      // wider FP8 rows keep one.
      if constexpr (FMT == kFmtNvfp4) {
        if (i == 0 && 1 < ntiles) {
          const int32_t ns = slots[slot_index(1, r)];
          if (ns >= 0) load_quarter<FMT>(raw, row_of(ns), qu);
        }
        if (i + 2 < ntiles) {
          const int32_t ns = slots[slot_index(i + 2, r)];
          if (ns >= 0) load_quarter<FMT>(rawn, row_of(ns), qu);
        }
      } else {
        if (i + 1 < ntiles) {
          const int32_t ns = slots[slot_index(i + 1, r)];
          if (ns >= 0) load_quarter<FMT>(raw, row_of(ns), qu);
        }
      }
      if (tid == 0 && NVMLA_TRACED_TILE(i)) NVMLA_TRACE_POINT(6 + 8 * NVMLA_TRACE_SLOT(i));
      // ---- PV of tile i
      if (warp == kMmaWarp) {
        if (issuer) issue_pv(i);
        __syncwarp();
      }
    }
    // ------------------------------------------------------------ row sums
    ok = !workers_sync_or(!ok);
    // lanes l and l ^ 16 hold the same rows' halves: fold them, then a
    // transposing butterfly leaves head hb + (lane & 15)'s warp sum in v[0]
#pragma unroll
    for (int h = 0; h < 16; ++h) lp[h] += __shfl_xor_sync(0xffffffffu, lp[h], 16);
#pragma unroll
    for (int step = 0; step < 4; ++step) {
      const int o = 8 >> step;
      const int n = 8 >> step;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < n; ++k) {
        const float send = upper ? lp[k] : lp[k + n];
        const float keep = upper ? lp[k + n] : lp[k];
        lp[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    if (lane < 16) red[quad * 64 + hb + lane] = lp[0];
    workers_sync();
    if (tid < kHeads) {
      const int h = tid;
      const float l = (red[h] + red[64 + h]) + (red[128 + h] + red[192 + h]);
      const bool live = ok && ntiles > 0 && l > 0.f;
      ml_pub[2 * h] = live ? m_run[h] : -INFINITY;
      ml_pub[2 * h + 1] = live ? l : 0.f;
      alpha_s[h] = live ? 1.f / l : 0.f;
      NVMLA_CHECK(t < p.T && h0 + h < p.H);
      if (S == 1) p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = live ? (m_run[h] + log2f(l)) * kLn2 : -INFINITY;
    }
    workers_sync();
    if (tid == 0) NVMLA_TRACE_POINT(20);
    // ------------------------------------------------------------ O^T
    // The last PV's block 3 commit lands after blocks 0-2 (a commit covers
    // every MMA issued before it): one wait, then the four blocks' TMEM
    // loads two at a time.
    bool have = ok && ntiles > 0;
    if (have) have = wait_bar_warp(bar(kBarPV + 3), (ntiles - 1) & 1, abort_flag, p.err_word);
    tc_fence_after();
    float inv_l[16];  // 1 / l of this thread's heads (0 for an empty head)
#pragma unroll
    for (int h4 = 0; h4 < 4; ++h4) {
      const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + hb + 4 * h4);
      inv_l[4 * h4] = a4.x;
      inv_l[4 * h4 + 1] = a4.y;
      inv_l[4 * h4 + 2] = a4.z;
      inv_l[4 * h4 + 3] = a4.w;
    }
#pragma unroll
    for (int j2 = 0; j2 < 4; j2 += 2) {
      float o2[2][16];
      if (have) {
        NVMLA_TMEM_LD16F(tmem + lane_base + o_col(j2, hb), o2[0], 0);
        NVMLA_TMEM_LD16F(tmem + lane_base + o_col(j2 + 1, hb), o2[1], 0);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) o2[0][e] = o2[1][e] = 0.f;
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = j2 + jj;
        const float* o = o2[jj];
        const int d = 128 * j + r;  // TMEM lane r of block j: value dim 128 j + r
        NVMLA_CHECK(t < p.T && h0 + hb + 15 < p.H && d < kLatent);
        if (S == 1) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            p.out[(static_cast<int64_t>(t) * p.H + h0 + hb + e) * kLatent + d] = __float2bfloat16_rn(o[e] * inv_l[e]);
        } else {
          // normalised partial (fp16, [dim d][64 heads], 16-byte unit v of
          // dim row d at v ^ (d & 7)) in the latent tile, which the PV no
          // longer reads
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int hl = 8 * cc + 2 * e;
              w4[e] = pack_f16x2(o[hl] * inv_l[hl], o[hl + 1] * inv_l[hl + 1]);
            }
            *reinterpret_cast<uint4*>(smem + stage_off(d, 2 * qu + cc)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    }
    tc_fence_before();
    if (tid == 0) NVMLA_TRACE_POINT(21);
    // every MMA the issuer issued has finished once this commit lands (the
    // epilogue has waited for the last PV; after an abort, anything issued)
    if (warp == kMmaWarp) {
      if (issuer) {
        mma_commit(bar(kBarDrain));
        wait_bar_drain(bar(kBarDrain), 0);
      }
      __syncwarp();
    }
  }

  // ------------------------------------------------------------ combine
  __syncthreads();  // every role is done with TMEM; the staged partial is written
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  // the first tile's copies have landed before this CTA's shared memory can go
  if (tid == 0) wait_bar_drain(bar(kBarRows0), 0);
  if (S > 1) {
    // release / acquire at cluster scope: every CTA's staged partial and
    // (m, l) are visible to every CTA of the cluster
    cluster_sync_all();
    if (tid == 0) NVMLA_TRACE_POINT(22);
    const int d0 = dim_lo(static_cast<int>(rank), S);
    const int D = dim_lo(static_cast<int>(rank) + 1, S) - d0;
    // combine weights l_s 2^(m_s - M) / L per head, [S][64] in the P^T
    // buffer: eight consecutive lanes per head, splits s = q, q + 8
    if (tid < 8 * kHeads) {
      const int h = tid >> 3, q = tid & 7;
      float m2[2], l2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int s = q + 8 * e;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (s < S) ml = ld_cluster_f2(map_rank(sbase + kOffMl + 8 * h, static_cast<uint32_t>(s)));
        l2[e] = ml.y;
        m2[e] = ml.y > 0.f ? ml.x : -INFINITY;
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
        if (q + 8 * e < S) *reinterpret_cast<float*>(smem + coef_off(q + 8 * e, h)) = w2[e] * inv;
      if (rank == 0 && q == 0)
        p.lse[static_cast<int64_t>(t) * p.H + h0 + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    if (tid == 0) NVMLA_TRACE_POINT(23);
    // item = (dim d, 16-byte unit u of its staged row): eight consecutive
    // lanes read one dim row, so a warp reads 512 contiguous bytes of a
    // peer's shared memory at a time; unit u holds heads 8 (u ^ (d & 7))..+7.
    // The sums go, transposed, to a [64 heads][D dims] bf16 buffer in the
    // query block's space (free since the last QK): 8-dim unit c of head h
    // at unit c ^ (h >> 3) of its row, so that the eight head groups a warp
    // writes at once fall into different banks.
    const int pitch = tb_pitch(D);  // bf16 elements per head row of the buffer
    __nv_bfloat16* tb = reinterpret_cast<__nv_bfloat16*>(smem + kOffQ);
    for (int it = tid; it < D * 8; it += kThreads) {
      const int dd = it >> 3, u = it & 7, d = d0 + dd, v = u ^ (d & 7);
      const uint32_t off = sbase + stage_phys_off(d, u);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int s0 = 0; s0 < S; s0 += 8) {
        uint4 part[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          part[k] = (s0 + k < S) ? ld_cluster_v4(map_rank(off, static_cast<uint32_t>(s0 + k))) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (s0 + k >= S) break;
          const uint32_t w[4] = {part[k].x, part[k].y, part[k].z, part[k].w};
          const float4 c0 = *reinterpret_cast<const float4*>(smem + coef_off(s0 + k, 8 * v));
          const float4 c1 = *reinterpret_cast<const float4*>(smem + coef_off(s0 + k, 8 * v + 4));
          const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
            acc[2 * e] += c[2 * e] * f.x;
            acc[2 * e + 1] += c[2 * e + 1] * f.y;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) tb[tb_index(8 * v + e, dd, pitch)] = __float2bfloat16_rn(acc[e]);
    }
    if (tid == 0) NVMLA_TRACE_POINT(33);
    __syncthreads();
    if (tid == 0) NVMLA_TRACE_POINT(34);
    // out rows of this CTA's dims, 16 bytes a thread: a warp writes whole
    // 128-byte runs of a head row
    const int upr = D / 8;  // 16-byte units per head row
    for (int it = tid; it < kHeads * upr; it += kThreads) {
      const int h = it / upr, c = it - h * upr;
      NVMLA_CHECK(t < p.T && h0 + h < p.H && d0 + 8 * c + 8 <= kLatent);
      *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.H + h0 + h) * kLatent + d0 + 8 * c) =
          *reinterpret_cast<const uint4*>(tb + tb_index(h, 8 * c, pitch));
    }
    if (tid == 0) NVMLA_TRACE_POINT(35);
    // no CTA leaves while another may still read its shared memory
    cluster_sync_all();
  }
  if (tid == 0) NVMLA_TRACE_POINT(24);
}

}  // namespace tc

bool tc_supported(int H) { return H % tc::kHeads == 0; }
bool tc_fp8_rows_supported(int) { return false; }

namespace {

// Per-device launch set-up of the kernel: its shared-memory size, and for
// every cluster size S how many clusters of S CTAs can be resident at once
// (0: S cannot be launched). Filled once per device under a mutex into a
// local table and published with a release store; readers acquire the flag,
// so a caller either sees the whole table or fills it itself.
struct TcDevice {
  std::atomic<bool> ready{false};
  int max_active[tc::kMaxCluster + 1] = {0};
};
constexpr int kMaxDevices = 64;
TcDevice g_tc_dev[kMaxDevices];
std::mutex g_tc_mu;

int tc_prepare() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  TcDevice& d = g_tc_dev[dev];
  if (d.ready.load(std::memory_order_acquire)) return dev;
  std::lock_guard<std::mutex> lock(g_tc_mu);
  if (d.ready.load(std::memory_order_relaxed)) return dev;
  // both row formats: the same launch shape and resources
  bool non_portable = true;
  for (auto* k : {tc::decode_tc_kernel<tc::kFmtNvfp4>, tc::decode_tc_kernel<tc::kFmtFp8>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
    if (e != cudaSuccess) return -1;
    non_portable = non_portable &&
                   cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  }
  int table[tc::kMaxCluster + 1] = {0};
  for (int s = 1; s <= tc::kMaxCluster; ++s) {
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
    if (cudaOccupancyMaxActiveClusters(&n, tc::decode_tc_kernel<tc::kFmtNvfp4>, &cfg) == cudaSuccess) table[s] = n;
  }
  cudaGetLastError();  // a refused cluster size leaves no sticky error
  for (int s = 0; s <= tc::kMaxCluster; ++s) d.max_active[s] = table[s];
  d.ready.store(true, std::memory_order_release);
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

// The split partials travel through distributed shared memory: no workspace.
size_t tc_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_decode_tc(int fmt, const void* q_latent, const void* q_rope, const uint8_t* cache,
                             const RowSelect& sel, const int32_t* row_idx, int T, int H, int topk, float sm_scale,
                             void* out, float* lse, void* workspace, int splits, int32_t* err_word,
                             cudaStream_t stream, uint32_t p_wait_ns, int force_p_timeout) {
  // fmt: 0 = NVFP4 rows, 2 = FP8 rows in a paged cache
  if (fmt != 0 && fmt != 2) return cudaErrorNotSupported;
  (void)row_idx;
  (void)workspace;
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
  p.num_splits = splits;
  p.tiles_total = (topk + tc::kTile - 1) / tc::kTile;
  p.err_word = err_word;
  p.p_wait_ns = p_wait_ns;
  p.force_p_timeout = force_p_timeout;
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
