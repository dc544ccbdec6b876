// Shared-memory and TMEM layout of the tcgen05 decode kernel, and every
// offset the kernel computes into them, as functions of the thread, row,
// tile and split. Plain C++ (host and device): the kernel calls these, and a
// host-compiled test enumerates every argument the kernel can pass and
// checks bounds, alignment and that each store pattern covers its region
// exactly once.
#pragma once

#include <stdint.h>

#include "format.h"

#ifdef __CUDACC__
#define NVMLA_HD __host__ __device__ __forceinline__
#else
#define NVMLA_HD inline
#endif

namespace nvmla {
namespace tc {

constexpr int kTile = 128;          // rows per tile (MMA M)
constexpr int kHeads = 64;          // heads per CTA (MMA N)
constexpr int kMaxTiles = 16;       // 2048 slots
constexpr int kThreads = 512;       // 16 warps, all workers
constexpr int kMmaWarp = 15;        // allocates TMEM; its lane 0 also issues the MMAs
constexpr int kMaxCluster = 16;     // CTAs sharing one token
constexpr int kChunkBytes = 16384;  // 128 rows x 64 fp16 dims, 128B-swizzled
constexpr int kQBytes = kHeads * kDqk * 2;  // bf16 query block of one CTA: 72 KB

// TMEM (columns of 32 bits, 128 lanes)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S^T: columns [0, 64)
constexpr uint32_t kColO = 64;   // O^T block j: columns [64 + 64 j, +64)
constexpr uint32_t kColR = 320;  // RoPE K: 32 columns (64 fp16 dims x 128 rows)

// shared memory map (bytes); the base is 1 KB aligned
constexpr int kOffQ = 0;                  // Q^T: 9 chunks x 8 KB, K-major, swizzled
constexpr int kOffKV = kOffQ + 9 * 8192;  // latent tile: 8 chunks x 16 KB; first the
                                          // first tile's raw rows, last the staged partial
constexpr int kOffP = kOffKV + 8 * kChunkBytes;             // P^T 16 KB, later the combine weights
constexpr int kOffSlots = kOffP + kChunkBytes;              // kMaxTiles x 128 int32
constexpr int kOffRed = kOffSlots + kMaxTiles * kTile * 4;  // 4 quadrants x 64 heads fp32
constexpr int kOffM = kOffRed + 4 * kHeads * 4;             // 64 fp32 running maxima (log2 units)
constexpr int kOffAlpha = kOffM + kHeads * 4;               // 64 fp32 rescale factors, later 1 / l
constexpr int kOffMl = kOffAlpha + kHeads * 4;              // 64 x (m, l) of this CTA
constexpr int kOffBar = kOffMl + kHeads * 8;
enum Bar {
  kBarKV = 0,     // the tile's latent chunks and RoPE K are written (16 warps)
  kBarS = 1,      // QK done: S^T full; also every earlier MMA done (commit)
  kBarP = 2,      // P^T written, O^T rescaled if needed (16 warps)
  kBarPV = 3,     // 4: PV block j done, its two latent chunks reusable (commit)
  kBarDrain = 7,  // every MMA finished (commit)
  kBarRows0 = 8,  // the first tile's rows have landed (TMA; one arrival per row)
  kNumBars = 9
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffKV % 1024 == 0 && kOffP % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kQBytes == 9 * 8192, "Q^T is nine 8 KB chunks");
static_assert(kOffMl % 16 == 0, "(m, l) block alignment");

// The first tile's 128 rows land by TMA in the latent tile's space, an odd
// number of 16-byte units apart (NVFP4 23, FP8 37), so that the rows of
// eight consecutive lanes fall into distinct banks
constexpr int kRawPitchNvfp4 = 368;  // 352-byte rows
constexpr int kRawPitchFp8 = 592;    // 576-byte rows
constexpr int kOffRaw0 = kOffKV;
static_assert(kOffRaw0 + kTile * kRawPitchFp8 <= kOffKV + 8 * kChunkBytes, "first-tile rows fit the latent tile");

// byte offset of 16-byte piece c of row r inside a 128B-swizzled region
// (rows of 128 bytes, 8-row atoms of 1 KB)
NVMLA_HD uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// value dims [dim_lo(r), dim_lo(r + 1)) are combined by CTA r of S: whole
// groups of 8 dims, so that each CTA's share of a head row is 16-byte units
NVMLA_HD constexpr int dim_lo(int r, int S) { return 8 * ((r * (kLatent / 8)) / S); }

// tiles [lo, hi) of CTA `rank` of S, out of `total`
NVMLA_HD int tile_lo(int rank, int S, int total) { return (rank * total) / S; }

// ---- the query block: thread tid's unit m (16 bytes = 8 bf16 values;
// m < 8: latent unit tid + 512 m of the 64 x 64-unit latent part, m = 8:
// RoPE unit tid of the 64 x 8-unit RoPE part), converted to fp16, goes to
// Q^T chunk c (64 dims) at piece q of head row h
NVMLA_HD int q_src_off(int tid, int m) {  // byte offset in the part the unit comes from
  return 16 * (m < 8 ? tid + kThreads * m : tid);
}
NVMLA_HD int q_dst_off(int tid, int m) {
  const int u = tid + kThreads * m;
  const int h = m < 8 ? u >> 6 : tid >> 3;
  const int c = m < 8 ? (u & 63) >> 3 : 8;
  const int q = m < 8 ? u & 7 : tid & 7;
  return kOffQ + c * 8192 + static_cast<int>(swz(h, q));
}

// ---- the first tile's raw row r
NVMLA_HD int raw_row_off(int r, int pitch) { return kOffRaw0 + r * pitch; }

// ---- the latent tile: 16-byte piece (8 dims) `piece` of row r in chunk
// `chunk` (64 dims)
NVMLA_HD int latent_chunk_off(int chunk) { return kOffKV + chunk * kChunkBytes; }
NVMLA_HD int latent_off(int chunk, int r, int piece) { return latent_chunk_off(chunk) + static_cast<int>(swz(r, piece)); }

// ---- P^T: row r, 16-byte piece (8 heads)
NVMLA_HD int pt_off(int r, int piece) { return kOffP + static_cast<int>(swz(r, piece)); }

// ---- the tiles' slots: int32 index into the slot list at kOffSlots
NVMLA_HD int slot_index(int tile, int r) { return tile * kTile + r; }

// ---- the staged partial: dim d, unit u (heads 8u..8u+7) at unit u ^ (d & 7)
// of dim row d
NVMLA_HD int stage_off(int d, int u) { return kOffKV + d * 128 + ((u ^ (d & 7)) << 4); }
NVMLA_HD int stage_phys_off(int d, int unit) { return kOffKV + d * 128 + 16 * unit; }

// ---- the combine: weight of split s for head h (fp32)
NVMLA_HD int coef_off(int s, int h) { return kOffP + 4 * (s * kHeads + h); }
// bf16 index, in the query block's space, of (head h, dim dd of this CTA's
// share): 8-dim unit c of head h at unit c ^ (h >> 3) of its row
NVMLA_HD int tb_pitch(int D) { return (D + 63) / 64 * 64; }
NVMLA_HD int tb_index(int h, int dd, int pitch) { return h * pitch + 8 * ((dd >> 3) ^ (h >> 3)) + (dd & 7); }

// ---- TMEM: first column of a thread's 16 S^T columns (heads hb..hb+15),
// of its 16 O^T columns of block j, of its 8 RoPE columns (quarter u)
NVMLA_HD uint32_t s_col(int hb) { return kColS + static_cast<uint32_t>(hb); }
NVMLA_HD uint32_t o_col(int j, int hb) { return kColO + 64u * static_cast<uint32_t>(j) + static_cast<uint32_t>(hb); }
NVMLA_HD uint32_t r_col(int u) { return kColR + 8u * static_cast<uint32_t>(u); }

}  // namespace tc
}  // namespace nvmla
