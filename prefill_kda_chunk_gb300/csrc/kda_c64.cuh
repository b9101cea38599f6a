// The 64-token chunk record and the operand layouts of the tcgen05 path.
//
// The recurrent kernel propagates the state once per 64 tokens. Each step is
// three groups of 5th-generation tensor-core MMAs with M = 128 (value
// channels in the accumulator's lanes), so the intra-chunk kernel hands over,
// per (64-token chunk, head), one record whose operand tiles are already in
// the tensor core's shared-memory layout and are copied byte for byte.
//
// Tile layout ("K-major, no swizzle"): a tile of R rows x E elements (bf16,
// E along the MMA's contraction dimension K) is a grid of 8-row x 8-element
// core matrices of 128 contiguous bytes each; the core matrix of rows
// [8a, 8a+8) and elements [8b, 8b+8) starts at a * (E * 16) + b * 128, and
// row r, element e inside it sits at (r % 8) * 16 + (e % 8) * 2. In a
// shared-memory descriptor the step between core matrices along K (leading
// byte offset) is then 128 and the step between 8-row groups (stride byte
// offset) E * 16; one MMA with K = 16 reads two core matrices along K, so
// the next K-step starts 256 bytes further.
#pragma once

#include <stdint.h>

namespace kda {
namespace c64 {

constexpr int kC = 64;   // tokens per chunk

// Record of one (chunk, head). With S the K x V state entering the chunk:
//   U = Ut - W S,  o = scale Qg S + scale P U,  S' = Diag(gamma) S + Kd^T U
constexpr int kRecB1 = 0;        // [scale Q e^G ; -W]: 128 rows (64 of Qg, then 64 of -W)
                                 //   x 128 keys, bf16 K-major tiles (32 KiB)
constexpr int kRecB2 = 32768;    // Kd^T = (K e^(G_last - G))^T: 128 key rows x 64 tokens (16 KiB)
constexpr int kRecB3 = 49152;    // scale P: 64 rows r x 64 tokens i, lower incl. diagonal (8 KiB);
                                 //   B2 and B3 together are one 192-row tile [Kd^T ; P]
constexpr int kRecUt = 57344;    // Ut^T = (T diag(beta) V)^T: [128 v][64 tok] bf16, the 16-byte
                                 //   granule j of row v stored at granule j ^ (v % 8) (16 KiB)
constexpr int kRecGam = 73728;   // exp(G_last): fp32 [128]
constexpr int kRecBytes = 74240;

// Byte offset of (row, element) in a K-major tile with `ext` elements per row.
__host__ __device__ constexpr uint32_t kmaj(int row, int e, int ext) {
    return static_cast<uint32_t>((row >> 3) * (ext * 16) + (e >> 3) * 128 + (row & 7) * 16 +
                                 (e & 7) * 2);
}

// Byte offset of granule j (tokens 8j..8j+7) of value row v of the Ut^T tile.
__host__ __device__ constexpr uint32_t ut_off(int v, int j) {
    return static_cast<uint32_t>(v * 128 + ((j ^ (v & 7)) << 4));
}

}  // namespace c64
}  // namespace kda
