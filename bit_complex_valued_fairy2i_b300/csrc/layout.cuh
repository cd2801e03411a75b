// Packed code layout (version 2) and small shared device helpers.
//
// A code plane (one matrix U or W, one stage t) of an n x m layer:
//   rows in tiles of 16 (row tile rt = j / 16; rows 16 rt + 8 rho + g with
//   rho in {0, 1}, g in 0..7), columns in blocks of 64 (block kb = k / 64),
//   one 256-byte tile per (rt, kb): 32 lanes, lane (g, q) = 4 g + q, each with
//   a sign word S and a flag word F (sign 1 = the code is -1 or -i, flag 1 =
//   the code is +i or -i).
//
// The words are laid out for the sparse tensor-core form of the layer.  With
// each code's real-axis and imaginary-axis slots interleaved along K, every
// two codes form a group of four K slots holding exactly two nonzeros, i.e.
// 2:4 structured sparsity: `mma.sp m16n8k32` takes the nonzero values (the
// signs, as bfloat16 +-2) from S and the slot indices (the axis flags) from F.
//   S of lane (g, q): for step s = 0..3 (16 columns each) and fragment
//     register i = 0..3 (rho = i & 1, h = i >> 1), r = 4 s + i: bit 15 - r is
//     the sign of row rho, column 64 kb + 16 s + 8 h + 2 q, and bit 31 - r the
//     sign of the next column.  Shifting S left by r puts the two signs of
//     register i of step s at bits 15 and 31.
//   F of lane (g, q): the lane supplies the metadata of steps
//     sA = 2 (q >> 1) + d (d = 0, 1) for column groups grp = 4 (q & 1) + n'
//     (n' = 0..3; group = columns 16 sA + 2 grp, + 1) of rows rho = 0, 1:
//     nibble nb = n' + 4 rho holds the flag of the even column at bit
//     4 nb + d and of the odd column at bit 4 nb + 2 + d.  The metadata word
//     of step sA is then ((F >> d) & 0x55555555) | 0x88888888 (indices
//     0/1 for the even code's real/imaginary slot, 2/3 for the odd code's).
// Storage per row tile: blocks in chunks of two, lane-major, so that a lane's
// (S, F) of two consecutive blocks are 16 contiguous bytes; an odd last block
// stores 8 bytes per lane.  Padding rows and columns hold zero bits.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace f2i {

// Programmatic dependent launch: let the next kernel in the stream launch, and
// wait until the previous one has completed with its writes visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One output value to y[i]: fp32, or (bf16 != 0) rounded to nearest even to
// bfloat16 in a buffer of bfloat16 elements (the same value the fp32 output
// holds, rounded once).
__device__ __forceinline__ void store_y(float* y, int64_t i, float v, int32_t bf16) {
  if (bf16) reinterpret_cast<__nv_bfloat16*>(y)[i] = __float2bfloat16_rn(v);
  else y[i] = v;
}

constexpr int kRowsPerTile = 16;
constexpr int kColsPerBlock = 64;
constexpr int kTileBytes = 256;  // one (row tile, column block)

__host__ __device__ __forceinline__ int64_t row_tiles(int64_t n) { return (n + 15) / 16; }
__host__ __device__ __forceinline__ int64_t col_blocks(int64_t m) { return (m + 63) / 64; }
__host__ __device__ __forceinline__ int64_t plane_bytes(int64_t n, int64_t m) {
  return row_tiles(n) * col_blocks(m) * kTileBytes;
}

// Byte offset inside a plane of the (S, F) pair of lane `lane` for row tile
// rt and column block kb, in a plane with KB column blocks.
__host__ __device__ __forceinline__ int64_t pair_offset(int64_t rt, int64_t kb, int lane, int64_t KB) {
  const int64_t base = rt * KB * kTileBytes;
  const int64_t fullc = KB >> 1;
  if ((kb >> 1) < fullc) return base + (kb >> 1) * 512 + lane * 16 + (kb & 1) * 8;
  return base + fullc * 512 + lane * 8;
}

// Bit of the sign of (row rho, column 16 s + 8 h + 2 q + e of a block) in the
// S word of lane (g, q).
__host__ __device__ __forceinline__ int sign_bit(int s, int h, int rho, int e) {
  return 15 + 16 * e - (4 * s + 2 * h + rho);
}
// The lane q and the bit of the axis flag of (row rho, column 16 s + 8 h +
// 2 q' + e) in an F word: group 4 h + q' of step s is supplied by lane
// q = h + 2 (s >> 1), nibble q' + 4 rho, bit (s & 1) + 2 e of the nibble.
__host__ __device__ __forceinline__ int flag_lane(int s, int h) { return h + 2 * (s >> 1); }
__host__ __device__ __forceinline__ int flag_bit(int s, int qp, int rho, int e) {
  return 4 * (qp + 4 * rho) + (s & 1) + 2 * e;
}

// ---------------------------------------------------------------------------
// Layout version 3: the table-lookup decode layout.
//
// The decode evaluates each plane's two signed sums per row, P = sum of
// sigma x and Q = sum of sigma tau x (sigma = the code's sign, tau = +1 on the
// real axis and -1 on the imaginary axis; A_re = (P + Q) / 2 and
// A_im = (P - Q) / 2), by looking up, for every group of 8 columns, the signed
// sum of those 8 activations selected by one byte of code bits.  A code plane
// therefore stores, per (row, group of 8 columns), a sign byte (bit c = sign
// of column 8 G + c, 1 = -1 or -i) and a q byte (sign XOR imaginary-axis
// flag).
//
// Rows come in tiles of 32 (row j = 32 tau + r, lane r of the decode) and
// columns in windows of 256 (32 groups; window w).  Inside a window the
// groups form blocks of 8 (block b = G >> 3, 64 columns); a window stores
// nb blocks (4, or for a last partial window 1, 2 or 4 with zero padding),
// as nb slots of 512 bytes: 32 rows x 16 bytes, sign bytes 0..7 then q bytes
// 8..15.  Slot jj of row r holds block b = jj ^ (a & (nb - 1)), a =
// (r >> 3) & 3, its group 8 b + ((r & 7) ^ i) in byte i.  Equivalently the
// byte (jj, i) of row r is group (r & (8 nb - 1)) ^ (8 jj + i): at every byte
// position the 32 rows of a full window name 32 different groups, so the 32
// lanes of a warp read 32 different tables.
// Byte order: [window][row tile][plane (X, t)][slot][row][16 bytes].
// ---------------------------------------------------------------------------
constexpr int kL3Rows = 32;
constexpr int kL3Cols = 256;
constexpr int kL3SlotBytes = 512;

__host__ __device__ __forceinline__ int64_t l3_tiles(int64_t n) { return (n + 31) / 32; }
__host__ __device__ __forceinline__ int64_t l3_windows(int64_t m) { return (m + 255) / 256; }
// Slots (blocks of 64 columns) stored for window w: 4, or 1, 2, 4 for a last
// partial window (3 blocks are padded to 4).
__host__ __device__ __forceinline__ int l3_slots(int64_t m, int64_t w) {
  const int64_t rest = m - 256 * w;
  if (rest >= 256) return 4;
  const int nc = (int)((rest + 63) / 64);
  return nc == 3 ? 4 : nc;
}
// Slots of all windows of one row tile and plane.
__host__ __device__ __forceinline__ int64_t l3_row_slots(int64_t m) {
  return 4 * (m / 256) + ((m % 256) ? l3_slots(m, m / 256) : 0);
}
__host__ __device__ __forceinline__ int64_t l3_codes_bytes(int64_t n, int64_t m, int T) {
  return l3_tiles(n) * 2 * T * kL3SlotBytes * l3_row_slots(m);
}
// Byte offset of slot 0 of (window w, row tile tau, plane p).
__host__ __device__ __forceinline__ int64_t l3_offset(int64_t n, int64_t m, int T, int64_t w, int64_t tau, int p) {
  const int nb = l3_slots(m, w);
  return w * l3_tiles(n) * 2 * T * 4 * kL3SlotBytes + (tau * 2 * T + p) * (int64_t)nb * kL3SlotBytes;
}
// Byte (within the 16 bytes of row r in slot jj) of group g of a window with
// nb slots, and the slot: the inverse of the rule above.
__host__ __device__ __forceinline__ int l3_slot_of(int g, int r, int nb) { return (g >> 3) ^ ((r >> 3) & (nb - 1)); }
__host__ __device__ __forceinline__ int l3_byte_of(int g, int r) { return (g & 7) ^ (r & 7); }

// Per-device error word (bit flags), read and cleared by fairy2i_sync_status.
// kErrConfig: a kernel found its launch configuration unusable (shared-memory
// placement) and did nothing.
enum : unsigned { kErrNonFinite = 1u, kErrTimeout = 2u, kErrConfig = 4u };

}  // namespace f2i

__device__ unsigned int g_fairy2i_error_word;

__device__ __forceinline__ void f2i_raise(unsigned flag) { atomicOr(&g_fairy2i_error_word, flag); }
