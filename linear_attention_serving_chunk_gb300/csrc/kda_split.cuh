// Layout of the per-(chunk, head) records that carry the state-independent
// part of a chunk from the parallel chunk-preparation pass to the sequential
// state pass of the two-pass tensor-core prefill (dk = dv = 128, C = 64).
//
// A record is the shared-memory image of the operands the state pass feeds
// to its three MMAs (128-byte-swizzled tiles, byte for byte as the tensor
// cores read them), so the state pass moves it with plain bulk copies:
//
//   A3   [-Wk ; -Q~]   128 rows x 128 K, fp16, K-major (two 64-column regions)
//   KP   K' = K e^{G_last - G}  [64 tok x 128 dk], fp16, MN-major
//   U    U = T diag(beta) V     [64 tok x 128 dv], fp16, MN-major
//   P    -P (64 r x 64 i, zero for i > r), fp16, MN-major: K-row i holds the
//        64 r's, i.e. the second MN block of the 128 x 64 operand [X ; -P]
//   G    gamma = e^{G_last}, 128 fp32 (one per key channel)
//
// Rows of a ragged last chunk beyond its length are zero in every tile.
#pragma once

#include <stdint.h>

namespace kda {

constexpr uint32_t kRecA3 = 0;
constexpr uint32_t kRecKP = 32 * 1024;
constexpr uint32_t kRecU = 48 * 1024;
constexpr uint32_t kRecP = 64 * 1024;
constexpr uint32_t kRecG = 72 * 1024;
constexpr uint32_t kRecBytes = 73 * 1024;

}  // namespace kda
