/*
 * nvmla.h -- C ABI of the NVFP4 sparse-MLA library for GB300 (sm_103a).
 *
 * Two product calls:
 *
 *   nvfp4_mla_pack      quantises new tokens' MLA latent (512 values) and
 *                       RoPE part (64 values) into 352-byte rows of a paged
 *                       KV cache.
 *   sparse_mla_decode   for every query token, attends only to the cache
 *                       positions an indexer selected (up to 2048 slots,
 *                       empty slots = -1) and writes the bf16 output and the
 *                       fp32 log-sum-exp.
 *
 * and the comparison baseline built in-house:
 *
 *   nvfp4_stage_dequant_fp8 + sparse_mla_decode_fp8rows
 *                       unpack the selected rows into a temporary 576-byte
 *                       FP8 buffer in GPU memory, then attend over it.
 *
 * Sources (web pages, cited by title and section):
 *   [Serving]  "Prime Inference: Fast, Reliable Serving for Frontier Open
 *              Models", sections "Making room for low-latency decode" and
 *              "A native NVFP4 sparse-MLA decode kernel".
 *   [KV]       "Prime Inference open-model serving" (mo.ai.kr), section
 *              "KV 캐시와 데이터 전송" (KV cache and data transfer).
 *   [4-bit]    "Prime Intellect unveils Prime Inference" (wireai.ir),
 *              section "4-bit caches open the way", items 1-3.
 *
 * Conventions for every call:
 *   - Pointers marked (device) are caller-owned GPU memory on the current
 *     device; the library never frees them and keeps no reference after the
 *     call returns. Pointers marked (host) are read during the call only.
 *   - All work is enqueued asynchronously on `stream` (NULL = the legacy
 *     default stream). The call returns once the work is enqueued.
 *   - Arguments are validated on the host before anything is launched; a
 *     call that returns an error status has launched nothing.
 *   - Data-dependent problems found on the device (an index outside its
 *     sequence, a slot outside the cache) never fault: the offending entry
 *     is skipped and reported through the optional `err_word` (device,
 *     2 x int32, caller-zeroed): err_word[0] |= NVMLA_ERRW_* flags,
 *     err_word[1] += number of offending entries.
 *   - Inputs must be finite. Queries must lie within the fp16 range
 *     (|q| < 65504): the attention runs on FP16 operands [Serving, "A native
 *     NVFP4 sparse-MLA decode kernel"].
 *   - nvmla_last_error() describes the most recent failing call of the
 *     calling thread.
 *
 * Cache layout (device, uint8 [num_pages][64][352], 32-byte aligned):
 *   row = 256 code bytes | 32 scale bytes | 64 RoPE bytes  [Serving, "Making
 *   room for low-latency decode": 512 values at 4 bits with one FP8 scale per
 *   16 values, 64 RoPE values kept in FP8, 352 bytes per row].
 *   Code byte j holds latent value 2j in bits 0-3 and 2j+1 in bits 4-7 (E2M1,
 *   sign in bit 3). Scale byte g (E4M3) scales values 16g..16g+15. RoPE byte j
 *   is value j in E4M3. Position p of sequence b lives in slot
 *   block_table[b][p / 64] * 64 + p % 64, i.e. page slot / 64, row slot % 64.
 */
#ifndef NVMLA_H_
#define NVMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st* nvmla_stream_t;

typedef enum {
  NVMLA_OK = 0,
  NVMLA_ERR_INVALID_ARG = 1, /* a pointer, size, stride or alignment is wrong */
  NVMLA_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle     */
  NVMLA_ERR_CUDA = 3,        /* a CUDA runtime call failed (see last_error)   */
  NVMLA_ERR_WORKSPACE = 4    /* workspace too small for the requested split   */
} nvmla_status;

/* err_word[0] flag bits */
#define NVMLA_ERRW_BAD_INDEX 0x1   /* topk entry not -1 and outside [0, seq_len) */
#define NVMLA_ERRW_BAD_SLOT 0x2    /* block-table slot outside the cache         */
#define NVMLA_ERRW_PACK_SLOT 0x4   /* pack slot >= num_pages * 64                */
#define NVMLA_ERRW_WAIT_TIMEOUT 0x8 /* a bounded pipeline wait gave up            */
#define NVMLA_ERRW_BOUNDS 0x10      /* a library built with NVMLA_DEBUG_BOUNDS found
                                       an index outside its buffer (never set by the
                                       default build, which does not check)        */

#define NVMLA_ROW_BYTES 352
#define NVMLA_FP8_ROW_BYTES 576
#define NVMLA_PAGE_TOKENS 64
#define NVMLA_LATENT_DIM 512
#define NVMLA_ROPE_DIM 64
#define NVMLA_MAX_TOPK 2048
#define NVMLA_MAX_HEADS 128
#define NVMLA_MAX_TOKENS 65535          /* query tokens per call (T) */
#define NVMLA_MAX_TOPK_COLS (1 << 29)   /* candidates per row of nvmla_topk_select */

/*
 * nvfp4_mla_pack -- write n_tokens rows into the paged cache.
 * [Serving, "Making room for low-latency decode"]; the group scale rule
 * (E4M3 of amax/6, 6 the largest E2M1 magnitude) and the byte order are
 * this library's reading of a format the page fixes only in size.
 *
 *   latent_bf16   (device) bf16 [n_tokens][latent_stride], first 512 used;
 *                 16-byte aligned, latent_stride a multiple of 8 elements.
 *   rope_bf16     (device) bf16 [n_tokens][rope_stride], first 64 used;
 *                 4-byte aligned, rope_stride even.
 *   slot_mapping  (device) int32 [n_tokens] physical slot of each token;
 *                 a negative slot skips the token; a slot >= num_pages*64 is
 *                 skipped and flagged NVMLA_ERRW_PACK_SLOT.
 *   cache         (device) uint8 [num_pages][64][352], 32-byte aligned.
 *   err_word      (device, nullable) see above.
 *
 * Per group of 16 values: amax = max |v|; scale byte = E4M3(amax / 6), round
 * to nearest even, saturating at 448; code = E2M1(|v| / S) with S the stored
 * scale, nearest even, saturating at 6, sign bit copied from v (S = 0 gives
 * magnitude 0). RoPE: E4M3(v), nearest even, saturating, no scale.
 * n_tokens == 0 is a no-op. Returns NVMLA_OK or an error status.
 */
nvmla_status nvfp4_mla_pack(const void* latent_bf16, int64_t latent_stride,
                            const void* rope_bf16, int64_t rope_stride,
                            const int32_t* slot_mapping, int64_t n_tokens,
                            uint8_t* cache, int64_t num_pages,
                            int32_t* err_word, nvmla_stream_t stream);

/*
 * sparse_mla_decode -- sparse MLA decode attention straight from the NVFP4
 * cache, with no FP8 staging buffer in GPU memory.
 * [Serving, "A native NVFP4 sparse-MLA decode kernel": consume the indexer's
 * positions, load only the compressed rows, unpack on chip, FP16 operands
 * with FP32 accumulation; 4-bit, item 3: 2048-slot lists, empty slots padded
 * and contributing nothing].
 *
 *   q_latent     (device) bf16 [T][H][512] contiguous, 16-byte aligned.
 *   q_rope       (device) bf16 [T][H][64] contiguous, 16-byte aligned.
 *   cache        (device) uint8 [num_pages][64][352], 32-byte aligned.
 *   block_table  (device) int32 [num_seqs][max_pages_per_seq].
 *   topk_idx     (device) int32 [T][topk] logical positions; -1 = empty slot.
 *   q_seq_idx    (device, nullable) int32 [T] sequence of each token (NULL:
 *                every token belongs to sequence 0).
 *   seq_lens     (device, nullable) int32 [num_seqs] context lengths (NULL:
 *                positions are only checked against the block-table width).
 *   T, H         query tokens (0 .. NVMLA_MAX_TOKENS) and heads (multiple of
 *                16, <= 128).
 *   topk         slots per token, 1..2048.
 *   sm_scale     softmax scale applied to q.k.
 *   out          (device) bf16 [T][H][512]: sum_k softmax_k * V_k.
 *   lse          (device) fp32 [T][H]: natural-log log-sum-exp of the scaled
 *                scores. A token with no valid slot gets out = 0,
 *                lse = -inf.
 *   workspace    (device, nullable) scratch for the split-key partials of
 *                the kernels that need it; sparse_mla_decode_workspace_size()
 *                gives the size for the default configuration. With a smaller
 *                workspace the call uses fewer key splits (never fails for
 *                lack of workspace).
 *   err_word     (device, nullable) see above.
 *
 * Duplicate positions count once per slot. T == 0 is a no-op.
 */
nvmla_status sparse_mla_decode(const void* q_latent, const void* q_rope,
                               const uint8_t* cache, int64_t num_pages,
                               const int32_t* block_table, int32_t num_seqs,
                               int32_t max_pages_per_seq,
                               const int32_t* topk_idx, int32_t topk,
                               const int32_t* q_seq_idx, const int32_t* seq_lens,
                               int32_t T, int32_t H, float sm_scale,
                               void* out, float* lse,
                               void* workspace, size_t workspace_bytes,
                               int32_t* err_word, nvmla_stream_t stream);

/* Bytes of workspace sparse_mla_decode uses by default for (T, H, topk) on
 * the current device (0 when the chosen kernel needs none). */
size_t sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t topk);

/* Kernel selection for tests and benchmarks (not needed in normal use). */
typedef enum {
  NVMLA_IMPL_AUTO = 0,   /* tcgen05 kernel where it applies, else the SIMT one */
  NVMLA_IMPL_MMA = 1,    /* warp-level mma.sync kernel with split-key partials */
  NVMLA_IMPL_TCGEN05 = 2 /* tcgen05 + TMEM kernel (H a multiple of 64)         */
} nvmla_impl;

typedef struct {
  int32_t impl;        /* nvmla_impl                                       */
  int32_t num_splits;  /* key splits per token; 0 = heuristic              */
  int32_t debug_flags; /* NVMLA_DEBUG_* test hooks; 0 in normal use        */
} nvmla_decode_options;

/* Test hook of the tcgen05 kernel: its wait for the softmax's P^T gives up
 * at once, as a bounded wait that ran out would. The call then returns
 * NVMLA_OK, sets NVMLA_ERRW_WAIT_TIMEOUT in err_word, leaves out and lse
 * undefined, and every CTA exits normally (its issued MMAs drained, TMEM
 * freed, every cluster barrier met). Other kernels ignore it. */
#define NVMLA_DEBUG_FORCE_WAIT_TIMEOUT 0x1

/* sparse_mla_decode with explicit options (NULL options = defaults). */
nvmla_status sparse_mla_decode_ex(const void* q_latent, const void* q_rope,
                                  const uint8_t* cache, int64_t num_pages,
                                  const int32_t* block_table, int32_t num_seqs,
                                  int32_t max_pages_per_seq,
                                  const int32_t* topk_idx, int32_t topk,
                                  const int32_t* q_seq_idx, const int32_t* seq_lens,
                                  int32_t T, int32_t H, float sm_scale,
                                  void* out, float* lse,
                                  void* workspace, size_t workspace_bytes,
                                  int32_t* err_word, const nvmla_decode_options* opts,
                                  nvmla_stream_t stream);

/* Workspace for sparse_mla_decode_ex with the given options. */
size_t sparse_mla_decode_workspace_size_ex(int32_t T, int32_t H, int32_t topk,
                                           const nvmla_decode_options* opts);

/* Key splits per token sparse_mla_decode_ex takes for (T, H, topk) with the
 * given options (NULL = defaults) on the current device, given enough
 * workspace: the CTAs that share one token's slots [Serving, "A native
 * NVFP4 sparse-MLA decode kernel": a cluster of cooperating SMs per query
 * token]. 0 for a shape the call rejects. Host-only. */
int32_t sparse_mla_decode_splits(int32_t T, int32_t H, int32_t topk,
                                 const nvmla_decode_options* opts);

/*
 * Block-major multi-layer caches.
 * [Serving, "Changing the layout to reduce fragmentation": a block-major
 * layout keeps one block's data for several layers together, so that moving
 * KV between workers takes fewer, larger copies; "KV cache and data
 * transfer" on the [KV] page: 64-token blocks]. The layout the pages name
 * (block, layer, head, token, channel) is read here, for the single latent
 * "head" of MLA, as
 *
 *   cache  (device) uint8 [num_blocks][num_layers][64][352], 32-byte aligned:
 *          row (b, l, i) at byte ((b * num_layers + l) * 64 + i) * 352.
 *
 * The calls below read or write one layer of such a cache. Slots and block
 * tables mean what they mean for a one-layer cache (slot = block * 64 + i),
 * so one block table serves every layer; num_blocks takes num_pages' place
 * in every check. A one-layer cache is num_layers = 1, layer = 0, and then
 * these calls are nvfp4_mla_pack and sparse_mla_decode_ex. Arguments,
 * errors and results otherwise as there; in addition
 * NVMLA_ERR_INVALID_ARG unless 1 <= num_layers <= 4096 and
 * 0 <= layer < num_layers.
 */
nvmla_status nvfp4_mla_pack_layered(const void* latent_bf16, int64_t latent_stride,
                                    const void* rope_bf16, int64_t rope_stride,
                                    const int32_t* slot_mapping, int64_t n_tokens,
                                    uint8_t* cache, int64_t num_blocks,
                                    int32_t num_layers, int32_t layer,
                                    int32_t* err_word, nvmla_stream_t stream);

nvmla_status sparse_mla_decode_layered(const void* q_latent, const void* q_rope,
                                       const uint8_t* cache, int64_t num_blocks,
                                       int32_t num_layers, int32_t layer,
                                       const int32_t* block_table, int32_t num_seqs,
                                       int32_t max_pages_per_seq,
                                       const int32_t* topk_idx, int32_t topk,
                                       const int32_t* q_seq_idx, const int32_t* seq_lens,
                                       int32_t T, int32_t H, float sm_scale,
                                       void* out, float* lse,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* err_word, const nvmla_decode_options* opts,
                                       nvmla_stream_t stream);

/*
 * sparse_mla_decode_noalloc -- sparse_mla_decode without a workspace
 * argument. The pages describe no such call: it exists for callers that
 * cannot allocate GPU memory (an engine whose memory pool owns the whole
 * GPU, a replayed fixed launch sequence, a C caller with no allocator). The
 * call allocates nothing: split partials that need global memory go to a
 * scratch array of sparse_mla_decode_noalloc_max_scratch() bytes (16 MiB) in
 * device memory owned by the library, reserved on each device where the
 * library's code loads and held until the process exits.
 *
 *   Arguments, results and err_word: as sparse_mla_decode.
 *   Same kernels and split count as sparse_mla_decode given a workspace of
 *   sparse_mla_decode_workspace_size(T, H, topk) bytes, hence the same output
 *   bits.
 *   Scratch needed: none when H is a multiple of 64 (the tcgen05 kernel
 *   combines its splits in shared memory). Otherwise the mma.sync kernel's
 *   T * S * H * (512 + 2) * 4 bytes, S its split count, and T * S <=
 *   floor(SMs / ceil(H / 64)): at most 15.0 MB for every H but 112 on a
 *   152-SM GB300 (17.5 MB for H = 112). Returns NVMLA_ERR_WORKSPACE,
 *   launching nothing, when the need exceeds the scratch.
 *   The first call on each device looks up the scratch's address
 *   (cudaGetSymbolAddress) and keeps it; make that call before any stream
 *   capture on the device. The address is that of the device's current
 *   context: after cudaDeviceReset (or any destruction of the primary
 *   context) the process must not call this function on that device again.
 *   The scratch is shared: calls whose work overlaps on the GPU (different
 *   streams, threads or processes sharing one context) race on it and give
 *   wrong results. Order such calls on one stream or by events.
 *   Nothing needs zeroing beforehand; the scratch is not cleared afterwards.
 */
nvmla_status sparse_mla_decode_noalloc(const void* q_latent, const void* q_rope,
                                       const uint8_t* cache, int64_t num_pages,
                                       const int32_t* block_table, int32_t num_seqs,
                                       int32_t max_pages_per_seq,
                                       const int32_t* topk_idx, int32_t topk,
                                       const int32_t* q_seq_idx, const int32_t* seq_lens,
                                       int32_t T, int32_t H, float sm_scale,
                                       void* out, float* lse,
                                       int32_t* err_word, nvmla_stream_t stream);

/* Bytes of scratch sparse_mla_decode_noalloc holds per device. */
size_t sparse_mla_decode_noalloc_max_scratch(void);

/*
 * nvfp4_stage_dequant_fp8 -- stage 1 of the staged baseline [KV, "KV 캐시와
 * 데이터 전송": the compressed rows were first unpacked into a temporary FP8
 * buffer in GPU memory; 4-bit, section text before items 1-3].
 * For every valid slot (t, k) the selected NVFP4 row is written as one
 * 576-byte FP8 row fp8_rows[t][k] = E4M3(E2M1(code_d) * scale) for the 512
 * latent values (nearest even, saturating at 448) followed by the 64 RoPE
 * bytes unchanged; row_idx[t][k] = k for a valid slot and -1 otherwise.
 * Rows of invalid slots are not written.
 *
 *   cache, block_table, topk_idx, q_seq_idx, seq_lens: as sparse_mla_decode.
 *   fp8_rows  (device) uint8 [T][topk][576], 16-byte aligned.
 *   row_idx   (device) int32 [T][topk].
 */
nvmla_status nvfp4_stage_dequant_fp8(const uint8_t* cache, int64_t num_pages,
                                     const int32_t* block_table, int32_t num_seqs,
                                     int32_t max_pages_per_seq,
                                     const int32_t* topk_idx, int32_t topk,
                                     const int32_t* q_seq_idx, const int32_t* seq_lens,
                                     int32_t T, uint8_t* fp8_rows, int32_t* row_idx,
                                     int32_t* err_word, nvmla_stream_t stream);

/*
 * sparse_mla_decode_fp8rows -- stage 2 of the staged baseline: the same
 * attention as sparse_mla_decode over 576-byte FP8 rows, key k of token t
 * being fp8_rows[t][row_idx[t][k]] when row_idx[t][k] >= 0. Also serves an
 * FP8 (576-byte row) cache laid out per token [Serving, "Making room for
 * low-latency decode": 576-byte FP8 rows].
 *
 *   fp8_rows  (device) uint8 [T][topk][576], 16-byte aligned.
 *   row_idx   (device) int32 [T][topk], entries in [-1, topk).
 *   other arguments as sparse_mla_decode; opts may be NULL.
 */
nvmla_status sparse_mla_decode_fp8rows(const void* q_latent, const void* q_rope,
                                       const uint8_t* fp8_rows, const int32_t* row_idx,
                                       int32_t topk, int32_t T, int32_t H, float sm_scale,
                                       void* out, float* lse,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* err_word, const nvmla_decode_options* opts,
                                       nvmla_stream_t stream);

/* Workspace for sparse_mla_decode_fp8rows. */
size_t sparse_mla_decode_fp8rows_workspace_size(int32_t T, int32_t H, int32_t topk,
                                                const nvmla_decode_options* opts);

/*
 * nvmla_topk_select -- the step upstream of the decode: each query token's
 * top-k positions by score as the fixed-length, -1 padded list that
 * sparse_mla_decode consumes. [4-bit, item 3: 2048-slot lists, empty slots
 * padded; Serving, "A native NVFP4 sparse-MLA decode kernel": the decode
 * consumes the positions the sparse indexer selected.] The indexer's scores
 * need trained weights the pages do not give: they are an input here.
 *
 *   scores     (device) fp32 [T][row_stride], 4-byte aligned; token t's
 *              candidates are positions 0 .. length_t - 1 of row t.
 *   ncols      columns that hold scores (row_stride >= ncols >= 0,
 *              ncols <= NVMLA_MAX_TOPK_COLS).
 *   T          rows (0 .. NVMLA_MAX_TOKENS).
 *   lengths    (device, nullable) int32 [T]: length_t, clamped to
 *              [0, ncols]; NULL means ncols for every token.
 *   topk       1..2048, the list length.
 *   topk_idx   (device) int32 [T][topk], written.
 *
 * Row t of topk_idx holds the k = min(topk, length_t) positions with the
 * largest scores, equal scores ranked by lower position, in increasing
 * order, then -1 up to topk. -0.0 ranks as +0.0; NaN scores are ranked by
 * their bits (above +inf when positive) and are not meant as input.
 * T == 0 is a no-op. Returns NVMLA_OK or an error status (nothing launched).
 *
 * Each row runs on one cluster of 8 CTAs. Rows of up to 262,144 candidates
 * are read from global memory once (each CTA keeps its eighth in shared
 * memory) and need one exchange of candidates between the CTAs. Slower
 * cluster-wide passes, with the same result, serve rows where a CTA has
 * more than 1,024 scores at or above its cut, or fewer than k scores lie at
 * or above the largest cut (winners bunched in one eighth, heavy ties);
 * longer rows are walked in global memory by a radix select.
 */
nvmla_status nvmla_topk_select(const float* scores, int64_t row_stride, int32_t ncols,
                               const int32_t* lengths, int32_t T, int32_t topk,
                               int32_t* topk_idx, nvmla_stream_t stream);

/*
 * The FP8 cache the NVFP4 format is measured against: 576-byte rows
 * [num_pages][64][576] (32-byte aligned), bytes 0-511 the latent and
 * 512-575 the RoPE values, each one E4M3 byte (round to nearest even,
 * saturating at 448, sign of zero kept; no scale). [Serving, "Making room
 * for low-latency decode": 576 bytes per token for an FP8 row; KV, "KV
 * cache and data transfer": the FP8 decode at 13.7 us beside 12.0 us for
 * NVFP4.]
 *
 * fp8_mla_pack: arguments, checks and errors as nvfp4_mla_pack, writing
 * 576-byte rows.
 * sparse_mla_decode_fp8cache: arguments, results and errors as
 * sparse_mla_decode_ex over such a cache; it runs on the tcgen05 kernel
 * only: NVMLA_ERR_UNSUPPORTED unless H is a multiple of 64 (and for
 * impl = NVMLA_IMPL_MMA). The workspace is sized by
 * sparse_mla_decode_workspace_size_ex with impl = NVMLA_IMPL_TCGEN05.
 */
nvmla_status fp8_mla_pack(const void* latent_bf16, int64_t latent_stride,
                          const void* rope_bf16, int64_t rope_stride,
                          const int32_t* slot_mapping, int64_t n_tokens,
                          uint8_t* cache, int64_t num_pages,
                          int32_t* err_word, nvmla_stream_t stream);

nvmla_status sparse_mla_decode_fp8cache(const void* q_latent, const void* q_rope,
                                        const uint8_t* cache, int64_t num_pages,
                                        const int32_t* block_table, int32_t num_seqs,
                                        int32_t max_pages_per_seq,
                                        const int32_t* topk_idx, int32_t topk,
                                        const int32_t* q_seq_idx, const int32_t* seq_lens,
                                        int32_t T, int32_t H, float sm_scale,
                                        void* out, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* err_word, const nvmla_decode_options* opts,
                                        nvmla_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* nvmla_status_string(nvmla_status s);

/* Message of the calling thread's most recent failing call ("" if none). */
const char* nvmla_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t nvmla_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads). Lets benchmarks state how many GPU launches a call made. */
uint64_t nvmla_launch_count(void);

/* How this library was compiled: NVMLA_BUILD_DEBUG_BOUNDS is set in a build
 * with -DNVMLA_DEBUG_BOUNDS, whose tcgen05 decode checks every data-dependent
 * index against its buffer and reports a failure as NVMLA_ERRW_BOUNDS (for
 * tests; slower). The default build sets no flag. */
#define NVMLA_BUILD_DEBUG_BOUNDS 0x1
int32_t nvmla_build_flags(void);

#ifdef __cplusplus
}
#endif

#endif /* NVMLA_H_ */
