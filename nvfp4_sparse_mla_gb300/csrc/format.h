// Byte formats shared by the kernels and their host-side checks (plain C++:
// also compiled by the host compiler for the layout tests).
//
// "Prime Inference: Fast, Reliable Serving for Frontier Open Models",
// section "Making room for low-latency decode": a cache row holds the
// 512-value latent as 4-bit values with one FP8 scale per 16 values and the
// 64 RoPE values in FP8, 352 bytes, against 576 for an all-FP8 row.
#pragma once

namespace nvmla {

constexpr int kLatent = 512;           // latent (and value) dims
constexpr int kRope = 64;              // RoPE dims
constexpr int kDqk = kLatent + kRope;  // 576: query / key dims
constexpr int kRowBytes = 352;         // NVFP4 row: codes, scales, RoPE
constexpr int kCodeBytes = 256;        // E2M1 codes, two a byte
constexpr int kScaleOff = 256;         // 32 E4M3 scales, one per 16 values
constexpr int kRopeOff = 288;          // 64 E4M3 RoPE values
constexpr int kFp8RowBytes = 576;      // FP8 row: 512 latent then 64 RoPE E4M3 values
constexpr int kPage = 64;              // rows per cache page (block)

}  // namespace nvmla
