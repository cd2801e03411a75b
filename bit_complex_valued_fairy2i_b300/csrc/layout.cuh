// Packed code layout (version 1) and small shared device helpers.
//
// A code plane (one matrix U or W, one stage t) of an n x m layer:
//   rows in groups of 8 (row group rg = j / 8, g = j % 8),
//   columns in blocks of 64 (block kb = k / 64),
//   one 128-byte tile of 32 words per (rg, kb); word (4g + q) holds 16 codes
//   of row j, each as two bits (sign, real-axis flag).
// Code c = 0..15 of a word, with s = c >> 2, h = (c >> 1) & 1, e = c & 1,
// is column  64 kb + 16 s + 8 h + 2 q + e  and sits in bits
// (15 + 16 e - 2 P, 14 + 16 e - 2 P) with P = 2 s + h.
// Why: in an mma.sync m16n8k16 bf16 A fragment whose row g is the real-axis
// row of output 8 rg + g and row g + 8 its imaginary-axis row, lane (g, q)
// holds for step s the columns 16 s + 2 q + {0, 1} (P = 2 s) and
// 16 s + 8 + 2 q + {0, 1} (P = 2 s + 1), two per register, low column in
// the low half.  Shifting the word left by 2 P puts both codes of pair P in
// bits (15, 14) and (31, 30); then `& 0xC000C000` is the real-axis register
// and `(w & 0x80008000) | (~w & 0x40004000)` the imaginary-axis register,
// as bfloat16 values in {+2, -2, +0, -0} (2.0 = 0x4000).
// Within a row group the 128-byte tiles are stored in chunks of four blocks
// so that lane (4g + q) finds its words of four consecutive blocks in 16
// contiguous bytes; the last chunk holds the remaining r = KB % 4 blocks
// with r words per lane.
#pragma once
#include <cstdint>

namespace f2i {

constexpr int kRowsPerGroup = 8;
constexpr int kColsPerBlock = 64;
constexpr int kTileBytes = 128;  // one (row group, column block)

__host__ __device__ __forceinline__ int64_t row_groups(int64_t n) { return (n + 7) / 8; }
__host__ __device__ __forceinline__ int64_t col_blocks(int64_t m) { return (m + 63) / 64; }
__host__ __device__ __forceinline__ int64_t plane_bytes(int64_t n, int64_t m) {
  return row_groups(n) * col_blocks(m) * kTileBytes;
}

// Byte offset inside a plane of the word of lane `lane` (= 4g + q) for row
// group rg and column block kb, in a plane with KB column blocks.
__host__ __device__ __forceinline__ int64_t word_offset(int64_t rg, int64_t kb, int lane, int64_t KB) {
  const int64_t base = rg * KB * kTileBytes;
  const int64_t full = KB >> 2;
  const int64_t c = kb >> 2;
  if (c < full) return base + c * 512 + lane * 16 + (kb & 3) * 4;
  const int64_t r = KB - (full << 2);
  return base + full * 512 + lane * (4 * r) + (kb - (full << 2)) * 4;
}

// Column offset inside the 64-column block of code c (0..15) of lane q.
__host__ __device__ __forceinline__ int code_col(int c, int q) {
  return 16 * (c >> 2) + 8 * ((c >> 1) & 1) + 2 * q + (c & 1);
}
// Shift that brings code c (0..15) of a word to bits 1..0.
__host__ __device__ __forceinline__ int code_shift(int c) {
  return 14 + 16 * (c & 1) - 2 * (2 * (c >> 2) + ((c >> 1) & 1));
}

// 2-bit internal code (sign << 1 | real_flag)  <->  canonical 0..3
// (0 = +1, 1 = -1, 2 = +i, 3 = -i).
__host__ __device__ __forceinline__ uint32_t canonical_from_bits(uint32_t v) {
  return ((v & 1u) ? 0u : 2u) + (v >> 1);
}

// Per-device error word (bit flags), read and cleared by fairy2i_sync_status.
enum : unsigned { kErrNonFinite = 1u, kErrTimeout = 2u };

}  // namespace f2i

__device__ unsigned int g_fairy2i_error_word;

__device__ __forceinline__ void f2i_raise(unsigned flag) { atomicOr(&g_fairy2i_error_word, flag); }
