// Host-compiled check of the tcgen05 decode kernel's shared-memory and TMEM
// index arithmetic (nvfp4_sparse_mla_gb300/csrc/decode_tc_layout.h: the
// functions the kernel itself calls). Every argument the kernel can pass is
// enumerated; each store pattern must stay inside its region, be 16-byte
// aligned where the kernel moves 16 bytes, and cover its region exactly once
// where the kernel relies on that. Prints one line per failure and exits 1
// if there is any.
#include <cstdio>
#include <set>
#include <vector>

#include "decode_tc_layout.h"

using namespace nvmla;
using namespace nvmla::tc;

static int failures = 0;
#define CHECK(cond, ...)                              \
  do {                                                \
    if (!(cond)) {                                    \
      if (failures < 50) {                            \
        std::printf("FAIL %s: ", #cond);              \
        std::printf(__VA_ARGS__);                     \
        std::printf("\n");                            \
      }                                               \
      ++failures;                                     \
    }                                                 \
  } while (0)

// a set of 16-byte units [lo, lo + n) that must be hit exactly once each
struct Cover {
  int lo, n;
  std::vector<int> hits;
  Cover(int lo_, int bytes) : lo(lo_), n(bytes / 16), hits(bytes / 16, 0) {}
  void hit(int off, const char* what) {
    CHECK(off % 16 == 0, "%s: offset %d not 16-byte aligned", what, off);
    const int u = (off - lo) / 16;
    CHECK(off >= lo && u < n, "%s: offset %d outside [%d, %d)", what, off, lo, lo + 16 * n);
    if (off >= lo && u < n) ++hits[u];
  }
  void exactly_once(const char* what) {
    int bad = 0;
    for (int u = 0; u < n; ++u) bad += hits[u] != 1;
    CHECK(bad == 0, "%s: %d of %d units not written exactly once", what, bad, n);
  }
};

int main() {
  // ---- the map: regions in order, disjoint, within the budget
  CHECK(kOffQ + kQBytes <= kOffKV, "Q^T");
  CHECK(kOffKV + 8 * kChunkBytes <= kOffP, "latent tile");
  CHECK(kOffP + kChunkBytes <= kOffSlots, "P^T");
  CHECK(kOffSlots + 4 * kMaxTiles * kTile <= kOffRed, "slots");
  CHECK(kOffRed + 4 * 4 * kHeads <= kOffM && kOffM + 4 * kHeads <= kOffAlpha && kOffAlpha + 4 * kHeads <= kOffMl &&
            kOffMl + 8 * kHeads <= kOffBar,
        "small arrays");
  CHECK(kOffBar % 8 == 0 && kOffBar + 8 * kNumBars <= kOffMisc && kOffMisc + 16 <= kSmemBytes, "barriers");
  CHECK(kSmemBytes <= 232448, "budget %d", kSmemBytes);

  // ---- the query block: 512 threads x 9 units, a bijection onto Q^T, each
  // unit landing at the chunk and piece of its dims
  {
    Cover q(kOffQ, kQBytes);
    std::set<int> lat_src, rope_src;
    for (int tid = 0; tid < kThreads; ++tid)
      for (int m = 0; m < 9; ++m) {
        const int dst = q_dst_off(tid, m), src = q_src_off(tid, m);
        q.hit(dst, "query block -> Q^T");
        if (m < 8) {
          const int u = tid + kThreads * m;  // latent unit: head u / 64, dims 8 (u % 64)
          CHECK(src == 16 * u && src + 16 <= kHeads * kLatent * 2, "latent source of unit %d", u);
          lat_src.insert(src);
          CHECK(dst == kOffQ + ((u & 63) >> 3) * 8192 + static_cast<int>(swz(u >> 6, u & 7)), "latent unit %d", u);
        } else {
          CHECK(src == 16 * tid && src + 16 <= kHeads * kRope * 2, "RoPE source of thread %d", tid);
          rope_src.insert(src);
          CHECK(dst == kOffQ + 8 * 8192 + static_cast<int>(swz(tid >> 3, tid & 7)), "RoPE unit %d", tid);
        }
      }
    q.exactly_once("Q^T");
    CHECK(static_cast<int>(lat_src.size()) == kHeads * kLatent * 2 / 16, "latent sources read once");
    CHECK(static_cast<int>(rope_src.size()) == kHeads * kRope * 2 / 16, "RoPE sources read once");
  }

  // ---- the first tile's raw rows (TMA destinations) and each thread's
  // quarter reads from them
  for (int fmt = 0; fmt < 2; ++fmt) {
    const int pitch = fmt ? kRawPitchFp8 : kRawPitchNvfp4, bytes = fmt ? kFp8RowBytes : kRowBytes;
    CHECK(pitch % 16 == 0 && (pitch / 16) % 2 == 1 && pitch >= bytes, "pitch %d", pitch);
    for (int r = 0; r < kTile; ++r) {
      const int a = raw_row_off(r, pitch);
      CHECK(a % 16 == 0 && a >= kOffKV && a + bytes <= kOffKV + 8 * kChunkBytes, "raw row %d (format %d)", r, fmt);
      if (r > 0) CHECK(a >= raw_row_off(r - 1, pitch) + bytes, "raw rows %d, %d overlap", r - 1, r);
      for (int u = 0; u < 4; ++u) {
        if (fmt == 0) {
          CHECK(64 * u + 64 <= kCodeBytes && kScaleOff + 8 * u + 8 <= kRopeOff && kRopeOff + 16 * u + 16 <= kRowBytes,
                "NVFP4 quarter %d", u);
        } else {
          CHECK(128 * u + 128 <= kLatent && kLatent + 16 * u + 16 <= kFp8RowBytes, "FP8 quarter %d", u);
        }
      }
    }
  }

  // ---- the latent tile: chunk x row x piece, a bijection onto 128 KB
  {
    Cover kv(kOffKV, 8 * kChunkBytes);
    for (int c = 0; c < 8; ++c)
      for (int r = 0; r < kTile; ++r)
        for (int pc = 0; pc < 8; ++pc) {
          const int a = latent_off(c, r, pc);
          CHECK(a == latent_chunk_off(c) + static_cast<int>(swz(r, pc)), "latent chunk base");
          CHECK(a >= latent_chunk_off(c) && a < latent_chunk_off(c) + kChunkBytes, "chunk %d row %d piece %d", c, r, pc);
          kv.hit(a, "latent tile");
        }
    kv.exactly_once("latent tile");
  }

  // ---- P^T: row x piece, a bijection onto 16 KB
  {
    Cover pt(kOffP, kChunkBytes);
    for (int r = 0; r < kTile; ++r)
      for (int pc = 0; pc < 8; ++pc) pt.hit(pt_off(r, pc), "P^T");
    pt.exactly_once("P^T");
  }

  // ---- slot list: tile x row, a bijection onto kMaxTiles x 128 int32
  {
    std::vector<int> seen(kMaxTiles * kTile, 0);
    for (int i = 0; i < kMaxTiles; ++i)
      for (int r = 0; r < kTile; ++r) {
        const int k = slot_index(i, r);
        CHECK(k >= 0 && k < kMaxTiles * kTile, "slot index %d", k);
        if (k >= 0 && k < kMaxTiles * kTile) ++seen[k];
      }
    int bad = 0;
    for (int v : seen) bad += v != 1;
    CHECK(bad == 0, "slot list: %d entries not exactly once", bad);
  }

  // ---- the staged partial: dim x unit, a bijection onto the first 64 KB of
  // the latent tile; the physical unit read back is the logical one
  {
    Cover st(kOffKV, kLatent * 128);
    for (int d = 0; d < kLatent; ++d)
      for (int u = 0; u < 8; ++u) {
        st.hit(stage_off(d, u), "staged partial");
        CHECK(stage_phys_off(d, u ^ (d & 7)) == stage_off(d, u), "staging swizzle inverse d %d u %d", d, u);
      }
    st.exactly_once("staged partial");
  }

  // ---- split ranges and the combine, for every cluster size
  for (int S = 1; S <= kMaxCluster; ++S) {
    for (int total = 1; total <= kMaxTiles; ++total) {
      int prev = 0;
      for (int r = 0; r < S; ++r) {
        const int lo = tile_lo(r, S, total), hi = tile_lo(r + 1, S, total);
        CHECK(lo == prev && hi >= lo && hi - lo <= kMaxTiles, "tiles of rank %d of %d (%d tiles)", r, S, total);
        prev = hi;
      }
      CHECK(prev == total, "tiles of %d splits cover %d", S, total);
    }
    if (S == 1) continue;
    CHECK(dim_lo(0, S) == 0 && dim_lo(S, S) == kLatent, "dims of %d splits", S);
    for (int s = 0; s < S; ++s)
      for (int h = 0; h < kHeads; h += 4) {
        const int a = coef_off(s, h);
        CHECK(a >= kOffP && a + 16 <= kOffP + kChunkBytes && (h % 8 != 0 || a % 16 == 0), "weights s %d h %d", s, h);
      }
    for (int rank = 0; rank < S; ++rank) {
      const int d0 = dim_lo(rank, S), D = dim_lo(rank + 1, S) - d0;
      CHECK(D > 0 && D % 8 == 0 && D <= 8 * ((64 + S - 1) / S), "share of rank %d of %d: %d dims", rank, S, D);
      const int pitch = tb_pitch(D);
      CHECK(kHeads * pitch * 2 <= kQBytes, "output buffer of %d dims", D);
      std::vector<int> seen(kHeads * pitch, 0);
      for (int it = 0; it < D * 8; ++it) {  // the pulls and the transposed writes
        const int dd = it >> 3, u = it & 7, d = d0 + dd, v = u ^ (d & 7);
        const int a = stage_phys_off(d, u);
        CHECK(a >= kOffKV && a + 16 <= kOffKV + kLatent * 128 && a % 16 == 0, "pull d %d u %d", d, u);
        for (int e = 0; e < 8; ++e) {
          const int k = tb_index(8 * v + e, dd, pitch);
          CHECK(k >= 0 && k < kHeads * pitch, "output buffer index %d", k);
          if (k >= 0 && k < kHeads * pitch) ++seen[k];
        }
      }
      for (int h = 0; h < kHeads; ++h)  // the 16-byte reads of the output stores
        for (int c = 0; c < D / 8; ++c) {
          const int k = tb_index(h, 8 * c, pitch);
          CHECK(k % 8 == 0 && k + 8 <= kHeads * pitch, "output read h %d c %d", h, c);
          for (int e = 0; e < 8; ++e)
            if (k + e < kHeads * pitch) CHECK(seen[k + e] == 1, "output element h %d dim %d written once", h, 8 * c + e);
        }
    }
  }

  // ---- TMEM: S^T, the four O^T blocks and the RoPE K, disjoint, inside
  // the allocation
  for (int hb = 0; hb < kHeads; hb += 16) {
    CHECK(s_col(hb) + 16 <= kColO, "S^T columns of heads %d", hb);
    for (int j = 0; j < 4; ++j) CHECK(o_col(j, hb) >= kColO && o_col(j, hb) + 16 <= kColR, "O^T block %d", j);
  }
  for (int u = 0; u < 4; ++u) CHECK(r_col(u) >= kColR && r_col(u) + 8 <= kColR + 32 && kColR + 32 <= kTmemCols, "RoPE %d", u);

  std::printf("%s: %d failures\n", failures ? "FAILED" : "ok", failures);
  return failures ? 1 : 0;
}
