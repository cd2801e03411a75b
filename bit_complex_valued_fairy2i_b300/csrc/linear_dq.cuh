// Layer evaluation for large token counts from layout 3 by a dense GEMM of
// the dequantized real matrix.
//
// The quantized layer is y = U^ x + W^ conj(x) with U^ = sum over stages of
// (s_re b_re + i s_im b_im) ("Fairy2i: Ultra-Low-Bit LLM Quantization Using
// Complex Weights {±1, ±i}", Step 3: the stages add up to one matrix; "Industry
// implications").  Its real form acting on [Re x | Im x] is the matrix of
// Theorem 1 (same page, Step 1) rebuilt from U^, W^ (the inverse map):
//   R^11 = Re U^ + Re W^   R^12 = Im W^ - Im U^
//   R^21 = Im U^ + Im W^   R^22 = Re U^ - Re W^
// Every token is then one row of a dense real GEMM, y~ = R^ x~, which the
// 5th-generation tensor cores run in one of two forms:
//   bfloat16 (F16 = false): R^ = hi + lo, hi the bfloat16 rounding of R^
//     (formed in fp32) and lo the bfloat16 rounding of the remainder, so R^ is
//     carried to ~2^-18 relative; x as given.  Executed flops: 2 terms x
//     2 (2n)(2m) per token = 16 n m, against 16 n m T for the ternary form of
//     linear_prefill.cuh;
//   fp16 (F16 = true): one term, every row of R^ scaled by a power of two so
//     that its largest possible entry is below 2^15 and rounded once to fp16
//     (2^-11 relative); x scaled per token by a power of two into fp16 by
//     dq_x16_kernel (exact: a bfloat16 value has 8 significant bits), both
//     powers of two undone in the epilogue.  8 n m flops per token.
// Every product is exact in the fp32 accumulators.
//
// GEMM shape per tile: D[128 rows][256 tokens] += A[128][K] * B[256][K]^T
//   rows: 64 outputs j, row 2 jl = Re y_j, row 2 jl + 1 = Im y_j, so that one
//         decode of (U^, W^)[j][c] yields the entries of both rows for both
//         halves of x~;
//   K:    blocks of 64 columns in pairs (block c of Re x, block c of Im x),
//         the two stages of a pair filled by one decode;
//   A:    hi and lo (or the fp16 term), 128-byte swizzled K-major, written by 16 producer warps
//         from the codes (in shared memory) and the scales: per stage plane and
//         column a signed scale added on its axis, or, with at most 64 tokens,
//         one load per column and matrix from the row's value tables (the 16
//         sums a stage pair's sign and axis bits select);
//   codes: per window of 256 columns (4 k-block pairs), the layout-3 bytes of
//         the tile's two 32-row tiles (contiguous: 2 x 2T planes x the
//         window's slots x 512 bytes), one bulk copy (cp.async.bulk, the TMA
//         engine) into a ring of two stages, a window ahead of their decode;
//   B:    x [M][2m] bfloat16 (or its fp16 copy) by TMA through two maps, one per half of x~
//         (128-byte swizzle, zero fill past m columns and M tokens), so that
//         the columns of A past m (decoded from zero code bits) meet zeros;
//   D:    fp32 in TMEM, two accumulators of 256 columns (double buffered).
// Warp roles (23 warps, one CTA per SM, persistent over tiles): warp 0 TMA
// for B, warp 1 TMEM allocation and MMA issue, warps 2-17 A producers, warps
// 18-21 epilogue (tcgen05.ld, stores of y), warp 22 the code copies.  All
// mbarrier waits are bounded.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include "layout.cuh"
#include "linear_prefill.cuh"

namespace f2i {

constexpr int kDqMaxGroup = 8;
constexpr int kDqSchedMax = 2048;  // tiles a launch may list per CTA (longest first); more run round-robin
constexpr int kDqMaxCtas = 256;
constexpr int kDqBM = 128;  // real rows per tile (64 outputs)
constexpr int kDqBN = 256;  // tokens per MMA (at most; a launch takes N = M rounded up to 16 below 256)
constexpr int kDqBK = 64;   // columns per k-block
constexpr int kDqATerm = kDqBM * kDqBK * 2;   // 16 KB: one term of A
constexpr int kDqBStage = kDqBN * kDqBK * 2;  // 32 KB: x for one MMA
constexpr int kDqProducerWarps = 16;
constexpr int kDqThreads = 32 * (7 + kDqProducerWarps);
constexpr uint32_t kDqTmemCols = 512;
constexpr int kDqCStages = 2;  // code stages, one window each
// Code stage: 2 row tiles of 32 x 2T planes x 4 slots x 512 bytes.
__host__ __device__ constexpr uint32_t dq_c_stage(int T) { return 8192u * (uint32_t)T; }
// NT token tiles of N per decoded k-block pair: 1 (M <= 256, or T > 2; the
// two TMEM accumulators alternate between tiles) or 2 (M > 256 and T <= 2;
// one decode feeds two MMAs, the accumulators hold the tile's two token
// tiles).  SMALL (N <= 64, one token tile): the producers set the pace; B
// stages hold 64 tokens (8 KB) and the room goes to per-row value tables
// (dq_table_row).  Stages beside the code ring (A 32 KB each):
//   SMALL:           3 A and 3 B of 8 KB, value tables;
//   NT = 1, T <= 2:  3 A and 3 B of 32 KB;
//   otherwise:       2 A and 2 B of NT x 32 KB.
// An A stage holds hi and lo (32 KB), or with F16 the one term (16 KB) and
// then twice as many A stages.  (Value tables beyond SMALL, in the room the
// F16 stages leave, measured slower: 175.8 against 161.0 us per LLaMA-2-7B
// block at 256 tokens, 861 against 851 at 2048.)
template <bool F16>
__host__ __device__ constexpr uint32_t dq_a_stage_bytes() { return F16 ? kDqATerm : 2u * kDqATerm; }
template <int NT, int T, bool SMALL, bool F16>
__host__ __device__ constexpr int dq_a_stages() { return ((NT == 1 && T <= 2) || SMALL ? 3 : 2) * (F16 ? 2 : 1); }
template <bool SMALL, bool F16>
__host__ __device__ constexpr bool dq_tables() { return SMALL; }
template <int NT, int T, bool SMALL>
__host__ __device__ constexpr int dq_b_stages() { return (NT == 1 && T <= 2) || SMALL ? 3 : 2; }
template <int NT, bool SMALL>
__host__ __device__ constexpr uint32_t dq_b_stage_bytes() { return SMALL ? 64u * kDqBK * 2u : (uint32_t)NT * kDqBStage; }
// Value tables: for every row of the tile, matrix X and pair of stages, the 16
// (Re, Im) sums that the pair's sign and axis bits can select; row stride 16
// bytes past the tables, so that the rows of a warp start in different banks.
template <int T>
__host__ __device__ constexpr int dq_pairs() { return (T + 1) / 2; }
template <int T>
__host__ __device__ constexpr uint32_t dq_table_row() { return 2u * dq_pairs<T>() * 16u * 8u + 16u; }
template <int T, bool TAB>
__host__ __device__ constexpr uint32_t dq_table_bytes() { return TAB ? 64u * dq_table_row<T>() : 0u; }
template <int NT, int T, bool SMALL, bool F16>
__host__ __device__ constexpr size_t dq_smem_bytes() {
  return 1024 + (size_t)dq_a_stages<NT, T, SMALL, F16>() * dq_a_stage_bytes<F16>() +
         (size_t)dq_b_stages<NT, T, SMALL>() * dq_b_stage_bytes<NT, SMALL>() + (size_t)kDqCStages * dq_c_stage(T) +
         dq_table_bytes<T, dq_tables<SMALL, F16>()>() + 512;
}

struct DqProblem {
  const uint8_t* codes;  // layout 3
  const float* scales;
  float* y;
  const float* xfac;  // F16: per token, 2^-f of its fp16 copy (x scaled by 2^f)
  int32_t n, m;
  int64_t tile_begin;
  int32_t row_tiles;  // tiles of 64 outputs
  int32_t tok_tiles;  // tiles of NT x N tokens
  int32_t kpairs;     // blocks of 64 columns per half of x~
  int32_t out_bf16;   // y holds bfloat16 elements
};

struct DqParams {
  CUtensorMap tmap[2 * kDqMaxGroup];  // per problem: Re x and Im x, each a [M][m] view of x [M][2m]
  DqProblem p[kDqMaxGroup];
  int64_t total_tiles;
  int32_t count, T, M;
  int32_t N;        // tokens per MMA: a multiple of 16 in [16, 256]
  int32_t sched_n;  // 0: tile blockIdx.x + i gridDim.x; else the list below
  int32_t pad_;
  uint16_t cta_begin[kDqMaxCtas + 1];  // CTA b runs sched[cta_begin[b] .. cta_begin[b + 1])
  uint16_t sched[kDqSchedMax];
};

// The i-th tile of this CTA, or -1 past its last.
__device__ __forceinline__ int64_t dq_tile_id(const DqParams& P, int64_t i) {
  if (P.sched_n == 0) {
    const int64_t t = (int64_t)blockIdx.x + i * gridDim.x;
    return t < P.total_tiles ? t : -1;
  }
  const int64_t k = (int64_t)P.cta_begin[blockIdx.x] + i;
  return k < (int64_t)P.cta_begin[blockIdx.x + 1] ? (int64_t)P.sched[k] : -1;
}

struct DqTile {
  int pi;
  int rt, tt;
};
__device__ __forceinline__ DqTile dq_tile(const DqParams& P, int64_t tile) {
  int pi = 0;
  for (int i = 1; i < P.count; ++i)
    if (tile >= P.p[i].tile_begin) pi = i;
  const int64_t local = tile - P.p[pi].tile_begin;
  DqTile c;
  c.pi = pi;
  c.rt = (int)(local / P.p[pi].tok_tiles);
  c.tt = (int)(local - (int64_t)c.rt * P.p[pi].tok_tiles);
  return c;
}

// bfloat16 pairs of (a, b) rounded to nearest even (a in the low half), and
// of the remainders a - hi, b - hi (exact in fp32): hi + lo carries each value
// to 2^-18 relative.
__device__ __forceinline__ void dq_split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  uint32_t h, l;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(b), "f"(a));
  const float ra = a - __uint_as_float(h << 16), rb = b - __uint_as_float(h & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(rb), "f"(ra));
  hi = h;
  lo = l;
}

// fp16 pair of (a, b) rounded to nearest even, a in the low half.
__device__ __forceinline__ uint32_t dq_f16x2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// F16 form: the power of two e by which a row of R^ is scaled, from the bits
// of the row's 4T scales (non-negative): the largest scale times 2^e lies in
// [2^11, 2^12), so every entry of the scaled row (a signed sum of at most 2T
// <= 8 scales) is below 2^15 and stays in the fp16 range.  e is clamped to
// [-64, 64] (a row of zero scales gets 64), so 2^e and 2^-e are normal floats.
__device__ __forceinline__ int dq_row_exp(uint32_t max_bits) {
  return min(64, max(-64, 138 - (int)((max_bits >> 23) & 0xFFu)));
}
__device__ __forceinline__ float dq_pow2(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// One code of one stage added to (re, im): bit E of the sign word s and of
// the imaginary-axis flag word f (a group's column, in the byte of its plane);
// the value is +-s_re on the real axis or +-s_im on the imaginary one.
template <int E>
__device__ __forceinline__ void dq_code(float& re, float& im, uint32_t s, uint32_t f, uint32_t sre, uint32_t sim) {
  asm("{\n\t.reg .pred p;\n\t.reg .b32 t, v;\n\t"
      "and.b32 t, %2, %6;\n\t"
      "setp.ne.u32 p, t, 0;\n\t"
      "selp.b32 v, %5, %4, p;\n\t"
      "shl.b32 t, %3, %7;\n\t"
      "and.b32 t, t, 0x80000000;\n\t"
      "xor.b32 v, v, t;\n\t"
      "@p add.f32 %1, %1, v;\n\t"
      "@!p add.f32 %0, %0, v;\n\t}"
      : "+f"(re), "+f"(im)
      : "r"(f), "r"(s), "r"(sre), "r"(sim), "n"(1u << E), "n"(31 - E));
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// One code of one stage added to (re, im) as dq_code does (same operations):
// s the sign bit, f the imaginary-axis flag.
__device__ __forceinline__ void dq_add(float& re, float& im, uint32_t s, uint32_t f, uint32_t sre, uint32_t sim) {
  const float v = __uint_as_float((f ? sim : sre) ^ (s << 31));
  if (f) im = __fadd_rn(im, v);
  else re = __fadd_rn(re, v);
}
// Table index of column E from the word (sign, flag of stage 2k; sign, flag of
// stage 2k + 1) of bytes: bit 3 the first sign, 2 its flag, 1 the second
// sign, 0 its flag (the multiply gathers bit E of the four bytes, no carries).
template <int E>
__device__ __forceinline__ uint32_t dq_index(uint32_t w) {
  return (((w >> E) & 0x01010101u) * 0x08040201u) >> 24;
}
__device__ __forceinline__ uint32_t dq_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// The 8 codes of a group in one plane (bits B .. B + 7 of s and f).
template <int B>
__device__ __forceinline__ void dq_plane(float (&re)[8], float (&im)[8], uint32_t s, uint32_t f, uint32_t sre,
                                         uint32_t sim) {
  dq_code<B + 0>(re[0], im[0], s, f, sre, sim);
  dq_code<B + 1>(re[1], im[1], s, f, sre, sim);
  dq_code<B + 2>(re[2], im[2], s, f, sre, sim);
  dq_code<B + 3>(re[3], im[3], s, f, sre, sim);
  dq_code<B + 4>(re[4], im[4], s, f, sre, sim);
  dq_code<B + 5>(re[5], im[5], s, f, sre, sim);
  dq_code<B + 6>(re[6], im[6], s, f, sre, sim);
  dq_code<B + 7>(re[7], im[7], s, f, sre, sim);
}

template <int T, int NT, bool SMALL, bool F16>
__global__ void __launch_bounds__(kDqThreads, 1) linear_dq_kernel(const __grid_constant__ DqParams P) {
  extern __shared__ uint8_t dq_smem_raw[];
  constexpr int NP = 2 * T;
  constexpr int NW = (NP + 3) / 4;  // words holding one byte per plane
  static_assert(NT == 1 || T <= 2, "two token tiles per decode only for T <= 2 (shared memory)");
  static_assert(!SMALL || NT == 1, "small token tiles come one per decode");
  static_assert(dq_smem_bytes<NT, T, SMALL, F16>() <= 232448, "shared memory per CTA");
  constexpr int AS = dq_a_stages<NT, T, SMALL, F16>();
  constexpr uint32_t kAStage = dq_a_stage_bytes<F16>();
  constexpr int BS = dq_b_stages<NT, T, SMALL>();
  constexpr int CS = kDqCStages;
  constexpr uint32_t kBStage = dq_b_stage_bytes<NT, SMALL>();
  constexpr bool TAB = dq_tables<SMALL, F16>();
  constexpr uint32_t kCStage = dq_c_stage(T);

  const uint32_t raw = smem_u32(dq_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dq_smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + AS * kAStage;
  const uint32_t sC = sB + BS * kBStage;
  const uint32_t sTab = sC + CS * kCStage;  // value tables (TAB)
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(gbase + AS * kAStage + BS * kBStage + CS * kCStage + dq_table_bytes<T, TAB>());
  const uint32_t bar0 = smem_u32(bars);
  auto fullA = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto emptyA = [&](int s) { return bar0 + 8u * (uint32_t)(AS + s); };
  auto fullB = [&](int s) { return bar0 + 8u * (uint32_t)(2 * AS + s); };
  auto emptyB = [&](int s) { return bar0 + 8u * (uint32_t)(2 * AS + BS + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + 4);  // every issued MMA complete
  auto fullC = [&](int s) { return bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + 5 + s); };
  auto emptyC = [&](int s) { return bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + 5 + CS + s); };
  const uint32_t prod_bar = bar0 + 8u * (uint32_t)(2 * AS + 2 * BS + 5 + 2 * CS);  // the producer warps meet
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * AS + 2 * BS + 6 + 2 * CS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // accumulator of token tile `sub` of the lt-th tile, and how many tiles used it before
  auto acc_buf = [&](uint32_t lt, int sub) { return NT == 1 ? (int)(lt & 1u) : sub; };
  auto acc_use = [&](uint32_t lt) { return NT == 1 ? (lt >> 1) : lt; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < AS; ++s) {
      mbar_init(fullA(s), kDqProducerWarps);  // one arrive per producer warp
      mbar_init(emptyA(s), 1);                // tcgen05.commit
    }
    for (int s = 0; s < CS; ++s) {
      mbar_init(fullC(s), 1);                 // the code warp's arrive.expect_tx
      mbar_init(emptyC(s), kDqProducerWarps);  // one arrive per producer warp
    }
    mbar_init(prod_bar, kDqProducerWarps);
    for (int s = 0; s < BS; ++s) {
      mbar_init(fullB(s), 1);   // TMA arrive.expect_tx
      mbar_init(emptyB(s), 1);  // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4);
    }
    mbar_init(done_bar, 1);  // tcgen05.commit after the last MMA
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < 2 * P.count; ++i) tma_prefetch_map(&P.tmap[i]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kDqTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer: activations, k-blocks in pairs (Re x, Im x) ----------------
    if (lane == 0) {
      if constexpr (F16) pdl_wait();  // the fp16 copy of x comes from the conversion launch before
      uint32_t it = 0;
      bool ok = true;
      for (int64_t i = 0; ok; ++i) {
        const int64_t tile = dq_tile_id(P, i);
        if (tile < 0) break;
        const DqTile c = dq_tile(P, tile);
        const DqProblem& pr = P.p[c.pi];
        for (int kb = 0; ok && kb < 2 * pr.kpairs; ++kb, ++it) {
          const int s = (int)(it % BS);
          const uint32_t ph = (it / BS) & 1u;
          if (!mbar_wait(emptyB(s), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fullB(s), (uint32_t)NT * (uint32_t)P.N * (kDqBK * 2));
#pragma unroll
          for (int sub = 0; sub < NT; ++sub)
            tma_load_2d(sB + (uint32_t)s * kBStage + (uint32_t)sub * kDqBStage, &P.tmap[2 * c.pi + (kb & 1)], fullB(s),
                        (kb >> 1) * kDqBK, (c.tt * NT + sub) * P.N);
        }
      }
      for (uint32_t k = (it > (uint32_t)BS ? it - BS : 0u); k < it; ++k)
        if (!mbar_wait(fullB((int)(k % BS)), (k / BS) & 1u, abort_flag)) break;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: hi and lo (or the fp16 term) into one accumulator per token tile ----------------
    if (lane == 0) {
      const uint32_t idesc = F16 ? idesc_f16(kDqBM, P.N) : idesc_bf16(kDqBM, P.N);
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int64_t i = 0; ok; ++i, ++lt) {
        const int64_t tile = dq_tile_id(P, i);
        if (tile < 0) break;
        const DqTile c = dq_tile(P, tile);
        const int kbs = 2 * P.p[c.pi].kpairs;
        for (int sub = 0; ok && sub < NT; ++sub)
          if (!mbar_wait(acce_bar(acc_buf(lt, sub)), (acc_use(lt) & 1u) ^ 1u, abort_flag)) ok = false;
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int sa = (int)(it % AS), sb = (int)(it % BS);
          if (!mbar_wait(fullA(sa), (it / AS) & 1u, abort_flag) ||
              !mbar_wait(fullB(sb), (it / BS) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + (uint32_t)sa * kAStage;
#pragma unroll
          for (int sub = 0; sub < NT; ++sub) {
            const uint32_t d_tmem = tmem_base + (uint32_t)acc_buf(lt, sub) * kDqBN;
            const uint32_t b0 = sB + (uint32_t)sb * kBStage + (uint32_t)sub * kDqBStage;
#pragma unroll
            for (int kk = 0; kk < kDqBK / 16; ++kk) {
              tc_mma_bf16(d_tmem, sw128_desc(a0 + 32u * kk), sw128_desc(b0 + 32u * kk), idesc,
                          (kb > 0 || kk > 0) ? 1u : 0u);
              if constexpr (!F16)
                tc_mma_bf16(d_tmem, sw128_desc(a0 + kDqATerm + 32u * kk), sw128_desc(b0 + 32u * kk), idesc, 1u);
            }
          }
          tc_commit(emptyA(sa));
          tc_commit(emptyB(sb));
        }
        if (ok)
          for (int sub = 0; sub < NT; ++sub) tc_commit(accf_bar(acc_buf(lt, sub)));
      }
      // every issued MMA completes before the tensor memory is freed, also when
      // a wait gave up (then the epilogue may not have waited for them)
      tc_commit(done_bar);
      volatile int drain_flag = 0;
      mbar_wait(done_bar, 0, &drain_flag, 100000000ull);
    }
  } else if (warp < 2 + kDqProducerWarps) {
    // ---------------- A producers: codes + scales -> R^ hi / lo ----------------
    // Thread (jl, gq) owns output jl of the tile (rows 2 jl, 2 jl + 1) and
    // group gq (columns 8 gq .. 8 gq + 7) of every 64-column block: one byte
    // of signs and one of flags per stage plane, out of the row's 16-byte
    // layout-3 chunk in the code stage.  The eight lanes of a quarter warp
    // share jl and write the eight 16-byte chunks of a 128-byte row: no bank
    // conflicts.
    const int pt = tid - 64;  // 0..511
    const int jl = pt >> 3, gq = pt & 7;
    const uint32_t row0 = (uint32_t)(2 * jl), row1 = row0 + 1u;
    const uint32_t o0 = row0 * 128u + (((uint32_t)gq ^ (row0 & 7u)) << 4);
    const uint32_t o1 = row1 * 128u + (((uint32_t)gq ^ (row1 & 7u)) << 4);
    // in a code stage (a window of nb slots): row tile th = jl >> 5, row r =
    // jl & 31; plane p, slot q of the row at ((th 2T + p) nb + q) 512 + 16 r
    const int cth = jl >> 5, cr = jl & 31;
    const uint32_t cbyte = (uint32_t)(cr * 16 + l3_byte_of(gq, cr));
    uint32_t it = 0, itc = 0;  // itc: windows of codes consumed
    bool ok = true;
    // TAB: row jl's value tables
    constexpr int PAIRS = dq_pairs<T>();
    const uint32_t trow = sTab + (uint32_t)jl * dq_table_row<T>();
    uint32_t pbu = 0;  // uses of the producers' barrier
    auto producers_meet = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(prod_bar);
      const bool got = mbar_wait(prod_bar, pbu & 1u, abort_flag);
      ++pbu;
      return !__any_sync(0xffffffffu, !got);
    };
    for (int64_t i = 0; ok; ++i) {
      const int64_t tile = dq_tile_id(P, i);
      if (tile < 0) break;
      const DqTile c = dq_tile(P, tile);
      const DqProblem& pr = P.p[c.pi];
      const int64_t n = pr.n;
      const int64_t j = (int64_t)c.rt * 64 + jl;
      const bool live = j < n;
      // the row's scales as bits (zero past n): [plane][axis]
      uint32_t sre[NP], sim[NP];
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        sre[p] = live ? __float_as_uint(__ldg(pr.scales + (int64_t)(2 * p) * n + j)) : 0u;
        sim[p] = live ? __float_as_uint(__ldg(pr.scales + (int64_t)(2 * p + 1) * n + j)) : 0u;
      }
      if constexpr (F16) {  // the row's scales times 2^e (exact), so R^ is formed scaled
        uint32_t mb = 0;
#pragma unroll
        for (int p = 0; p < NP; ++p) mb = max(mb, max(sre[p], sim[p]));
        const float f = dq_pow2(dq_row_exp(mb));
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          sre[p] = __float_as_uint(__uint_as_float(sre[p]) * f);
          sim[p] = __float_as_uint(__uint_as_float(sim[p]) * f);
        }
      }
      if constexpr (TAB) {
        // the tables of row jl: for matrix X and stage pair k, entry idx (bits as
        // dq_index) holds the pair's (Re, Im) sum, accumulated like dq_code (from
        // 0, stage 2k first); thread gq writes entries gq and gq + 8 of each.
        // The producers meet before (the previous tile's tables are read out) and
        // after (the tables are complete).
        if (!producers_meet()) {
          ok = false;
          break;
        }
#pragma unroll
        for (int X = 0; X < 2; ++X)
#pragma unroll
          for (int k = 0; k < PAIRS; ++k) {
            const int p0 = X * T + 2 * k;
            const bool two = 2 * k + 1 < T;
            const int p1 = two ? p0 + 1 : p0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t idx = (uint32_t)(gq + 8 * h);
              float re = 0.0f, im = 0.0f;
              dq_add(re, im, (idx >> 3) & 1u, (idx >> 2) & 1u, sre[p0], sim[p0]);
              if (two) dq_add(re, im, (idx >> 1) & 1u, idx & 1u, sre[p1], sim[p1]);
              asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(trow + (uint32_t)((X * PAIRS + k) * 16 + idx) * 8u),
                           "f"(re), "f"(im)
                           : "memory");
            }
          }
        if (!producers_meet()) {
          ok = false;
          break;
        }
      }
      // the group's sign and q bytes of every stage plane for pair kp (zero
      // past n), read from the window's code stage one pair ahead of their
      // decode (plane p's byte at bits 8 (p & 3) of word p >> 2); a stage goes
      // back to the code warp when its window's last pair has been read
      auto fetch = [&](int kp, uint32_t(&sw)[NW], uint32_t(&qw)[NW]) -> bool {
        const uint32_t k = itc + (uint32_t)(kp >> 2);
        const int cs = (int)(k % CS);
        // one wait per window (its copy completes one phase of the barrier)
        if ((kp & 3) == 0 && __any_sync(0xffffffffu, !mbar_wait(fullC(cs), (k / CS) & 1u, abort_flag) ? 1 : 0))
          return false;
        const int nb = l3_slots(pr.m, kp >> 2);
        const int q = (kp & 3) ^ (cr >> 3 & (nb - 1));
        const uint32_t cb = sC + (uint32_t)cs * kCStage + (uint32_t)((cth * NP * nb + q) * 512) + cbyte;
#pragma unroll
        for (int w = 0; w < NW; ++w) sw[w] = qw[w] = 0u;
        if (live) {
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            sw[p >> 2] |= lds_u8(cb + 512u * (uint32_t)(nb * p)) << (8 * (p & 3));
            qw[p >> 2] |= lds_u8(cb + 512u * (uint32_t)(nb * p) + 8u) << (8 * (p & 3));
          }
        }
        return true;
      };
      uint32_t nsw[NW], nqw[NW];
      if (pr.kpairs > 0 && !fetch(0, nsw, nqw)) ok = false;
      for (int kp = 0; ok && kp < pr.kpairs; ++kp) {
        uint32_t sw[NW], fw[NW];  // signs, imaginary-axis flags
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          sw[w] = nsw[w];
          fw[w] = nsw[w] ^ nqw[w];
        }
        if ((kp & 3) == 3 || kp + 1 == pr.kpairs) {  // the window's last pair is in registers
          __syncwarp();
          if (lane == 0) mbar_arrive(emptyC((int)((itc + (uint32_t)(kp >> 2)) % CS)));
        }
        if (kp + 1 < pr.kpairs && !fetch(kp + 1, nsw, nqw)) {
          ok = false;
          break;
        }
        // (Re, Im) of U^ [0] and W^ [1] for the group's 8 columns, in fp32 (zero
        // scales past n); columns past m decode from zero bits and meet zero-filled x
        float re[2][8], im[2][8];
        if constexpr (TAB) {
          // per matrix and stage pair: the word of bytes (sign, flag of stage 2k;
          // sign, flag of stage 2k + 1), then one table load per column
#pragma unroll
          for (int X = 0; X < 2; ++X)
#pragma unroll
            for (int k = 0; k < PAIRS; ++k) {
              const int p0 = X * T + 2 * k;
              const bool two = 2 * k + 1 < T;
              const int p1 = two ? p0 + 1 : p0;
              uint32_t w = dq_prmt(sw[p0 >> 2], fw[p0 >> 2], (uint32_t)((p0 & 3) | ((4 + (p0 & 3)) << 4))) & 0xFFFFu;
              if (two) w |= dq_prmt(sw[p1 >> 2], fw[p1 >> 2], (uint32_t)((p1 & 3) | ((4 + (p1 & 3)) << 4))) << 16;
              const uint32_t tb = trow + (uint32_t)((X * PAIRS + k) * 16) * 8u;
              float2 v[8];
              v[0] = lds_f2(tb + 8u * dq_index<0>(w));
              v[1] = lds_f2(tb + 8u * dq_index<1>(w));
              v[2] = lds_f2(tb + 8u * dq_index<2>(w));
              v[3] = lds_f2(tb + 8u * dq_index<3>(w));
              v[4] = lds_f2(tb + 8u * dq_index<4>(w));
              v[5] = lds_f2(tb + 8u * dq_index<5>(w));
              v[6] = lds_f2(tb + 8u * dq_index<6>(w));
              v[7] = lds_f2(tb + 8u * dq_index<7>(w));
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                re[X][e] = k == 0 ? v[e].x : __fadd_rn(re[X][e], v[e].x);
                im[X][e] = k == 0 ? v[e].y : __fadd_rn(im[X][e], v[e].y);
              }
            }
        } else {
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int e = 0; e < 8; ++e) re[x][e] = im[x][e] = 0.0f;
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const uint32_t sb = sw[p >> 2], fb = fw[p >> 2];
            const int x = p < T ? 0 : 1;
            switch (p & 3) {  // resolved at compile time (the loop is unrolled)
              case 0: dq_plane<0>(re[x], im[x], sb, fb, sre[p], sim[p]); break;
              case 1: dq_plane<8>(re[x], im[x], sb, fb, sre[p], sim[p]); break;
              case 2: dq_plane<16>(re[x], im[x], sb, fb, sre[p], sim[p]); break;
              default: dq_plane<24>(re[x], im[x], sb, fb, sre[p], sim[p]); break;
            }
          }
        }
        // both stages of the pair: k-block 2 kp (Re x columns) and 2 kp + 1 (Im x columns)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int s = (int)(it % AS);
          const uint32_t ph = (it / AS) & 1u;
          ++it;
          // every lane polls the stage's barrier (no divergent branch)
          if (__any_sync(0xffffffffu, !mbar_wait(emptyA(s), ph ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          // row 2 jl: Re y, row 2 jl + 1: Im y
          //   Re x block: R^11 = ReU + ReW, R^21 = ImU + ImW
          //   Im x block: R^12 = ImW - ImU, R^22 = ReU - ReW
          if constexpr (F16) {
            uint32_t a0[4], a1[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              if (h == 0) {
                a0[e >> 1] = dq_f16x2(re[0][e] + re[1][e], re[0][e + 1] + re[1][e + 1]);
                a1[e >> 1] = dq_f16x2(im[0][e] + im[1][e], im[0][e + 1] + im[1][e + 1]);
              } else {
                a0[e >> 1] = dq_f16x2(im[1][e] - im[0][e], im[1][e + 1] - im[0][e + 1]);
                a1[e >> 1] = dq_f16x2(re[0][e] - re[1][e], re[0][e + 1] - re[1][e + 1]);
              }
            }
            const uint32_t st = sA + (uint32_t)s * kAStage;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o0), "r"(a0[0]), "r"(a0[1]), "r"(a0[2]),
                         "r"(a0[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o1), "r"(a1[0]), "r"(a1[1]), "r"(a1[2]),
                         "r"(a1[3])
                         : "memory");
          } else {
            uint32_t h0[4], l0[4], h1[4], l1[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              if (h == 0) {
                dq_split2(re[0][e] + re[1][e], re[0][e + 1] + re[1][e + 1], h0[e >> 1], l0[e >> 1]);
                dq_split2(im[0][e] + im[1][e], im[0][e + 1] + im[1][e + 1], h1[e >> 1], l1[e >> 1]);
              } else {
                dq_split2(im[1][e] - im[0][e], im[1][e + 1] - im[0][e + 1], h0[e >> 1], l0[e >> 1]);
                dq_split2(re[0][e] - re[1][e], re[0][e + 1] - re[1][e + 1], h1[e >> 1], l1[e >> 1]);
              }
            }
            const uint32_t st = sA + (uint32_t)s * kAStage;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o0), "r"(h0[0]), "r"(h0[1]), "r"(h0[2]),
                         "r"(h0[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o1), "r"(h1[0]), "r"(h1[1]), "r"(h1[2]),
                         "r"(h1[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + kDqATerm + o0), "r"(l0[0]), "r"(l0[1]),
                         "r"(l0[2]), "r"(l0[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + kDqATerm + o1), "r"(l1[0]), "r"(l1[1]),
                         "r"(l1[2]), "r"(l1[3])
                         : "memory");
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(fullA(s));
        }
      }
      itc += (uint32_t)((pr.kpairs + 3) / 4);
    }
  } else if (warp < 6 + kDqProducerWarps) {
    // ---------------- epilogue: D row 2 jl + part of token t -> y[t][part n + j] ----------------
    const int eq = warp & 3;  // TMEM lanes 32 eq .. 32 eq + 31
    const int rl = 32 * eq + lane;
    if constexpr (F16) pdl_wait();  // the tokens' factors come from the conversion launch
    const int jl = rl >> 1, part = rl & 1;
    uint32_t lt = 0;
    bool ok = true;
    for (int64_t i = 0; ok; ++i, ++lt) {
      const int64_t tile = dq_tile_id(P, i);
      if (tile < 0) break;
      const DqTile c = dq_tile(P, tile);
      const DqProblem& pr = P.p[c.pi];
      const int64_t j = (int64_t)c.rt * 64 + jl;
      const int64_t ystride = 2 * (int64_t)pr.n;
      float rfac = 1.0f;  // F16: 2^-e of the row's scaling (the producers' e, from the same scales)
      if constexpr (F16) {
        if (j < pr.n) {
          uint32_t mb = 0;
#pragma unroll
          for (int p = 0; p < 2 * NP; ++p) mb = max(mb, __float_as_uint(__ldg(pr.scales + (int64_t)p * pr.n + j)));
          rfac = dq_pow2(-dq_row_exp(mb));
        }
      }
      for (int sub = 0; sub < NT; ++sub) {
        const int b = acc_buf(lt, sub);
        bool got = true;
        if (lane == 0) got = mbar_wait(accf_bar(b), acc_use(lt) & 1u, abort_flag);
        got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(32 * eq) << 16) + (uint32_t)b * kDqBN;
        const int64_t tok0 = ((int64_t)c.tt * NT + sub) * P.N;
#pragma unroll 1
        for (int cc = 0; cc < (P.N + 31) / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(tbase + 32u * cc, v);
          tmem_ld_wait();
          if (j < pr.n) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int64_t tok = tok0 + 32 * cc + e;
              if (tok < P.M) {
                const float o = F16 ? __uint_as_float(v[e]) * rfac * __ldg(pr.xfac + tok) : __uint_as_float(v[e]);
                store_y(pr.y, tok * ystride + (int64_t)part * pr.n + j, o, pr.out_bf16);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(b));
      }
    }
  } else {
    // ---------------- code copies: each window's codes into the code ring ----------------
    // Window w of the tile's two 32-row tiles is one contiguous run of
    // layout 3 (tile-major inside the window): 2 x 2T planes x nb slots x 512
    // bytes (one tile's worth at the layer's last tile).
    uint32_t it = 0;
    bool ok = true;
    for (int64_t i = 0; ok && lane == 0; ++i) {
      const int64_t tile = dq_tile_id(P, i);
      if (tile < 0) break;
      const DqTile c = dq_tile(P, tile);
      const DqProblem& pr = P.p[c.pi];
      const int64_t n = pr.n, m = pr.m;
      const int ntile = (int)min((int64_t)2, l3_tiles(n) - 2 * (int64_t)c.rt);  // row tiles of 32 present
      const int nw = (pr.kpairs + 3) / 4;
      for (int w = 0; w < nw; ++w, ++it) {
        const int s = (int)(it % CS);
        if (!mbar_wait(emptyC(s), ((it / CS) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t bytes = (uint32_t)(ntile * NP * l3_slots(m, w)) * (uint32_t)kL3SlotBytes;
        mbar_arrive_expect_tx(fullC(s), bytes);
        bulk_load(sC + (uint32_t)s * kCStage, pr.codes + l3_offset(n, m, T, w, 2 * c.rt, 0), bytes, fullC(s));
      }
    }
    // no copy outlives the CTA: wait for the last stages to land
    if (lane == 0)
      for (uint32_t k = (it > (uint32_t)CS ? it - CS : 0u); k < it; ++k)
        if (!mbar_wait(fullC((int)(k % CS)), (k / CS) & 1u, abort_flag)) break;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kDqTmemCols);
  }
}

// ---------------------------------------------------------------------------
// The activations of the F16 form: per layer and token, x~ (2m bfloat16, m a
// multiple of 8) times 2^f as fp16 into xh, and 2^-f into xfac.  f puts the
// token's largest magnitude in [2^14, 2^15) (f = 0 for a token of zeros or
// with Inf/NaN, whose values then convert as they are; at most 64, so a token
// below 2^-50 keeps fewer significant bits).  Every finite bfloat16 value the
// scaling leaves at or above 2^-17 is exact in fp16 (8 significant bits).
// One CTA per (token, layer); two passes over the row (the second from cache).
constexpr int kDqXThreads = 256;
struct DqXParams {
  const uint16_t* x[kDqMaxGroup];
  uint16_t* xh[kDqMaxGroup];
  float* xfac[kDqMaxGroup];
  int32_t m[kDqMaxGroup];
  int32_t count, pad_;
};

__device__ __forceinline__ uint32_t dq_bf16x2_to_f16x2(uint32_t w, float f) {
  return dq_f16x2(__uint_as_float(w << 16) * f, __uint_as_float(w & 0xFFFF0000u) * f);
}

__global__ void __launch_bounds__(kDqXThreads) dq_x16_kernel(const __grid_constant__ DqXParams P) {
  pdl_launch_dependents();  // the GEMM may set up and decode codes meanwhile
  const int l = blockIdx.y;
  const int64_t t = blockIdx.x, m = P.m[l];
  const uint4* src = reinterpret_cast<const uint4*>(P.x[l] + t * 2 * m);
  uint4* dst = reinterpret_cast<uint4*>(P.xh[l] + t * 2 * m);
  const int chunks = (int)(m / 4);  // 16-byte chunks of the 2m values
  uint32_t mx = 0;                  // largest magnitude (bits), two lanes of 16
  for (int c = threadIdx.x; c < chunks; c += kDqXThreads) {
    const uint4 v = __ldg(src + c);
    mx = __vmaxu2(mx, v.x & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v.y & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v.z & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v.w & 0x7FFF7FFFu);
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
  __shared__ uint32_t wmax[kDqXThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
  __syncthreads();
  uint32_t b = 0;
#pragma unroll
  for (int w = 0; w < kDqXThreads / 32; ++w) b = max(b, wmax[w]);
  // a bfloat16 magnitude with biased exponent E lies in [2^(E-127), 2^(E-126))
  const int f = (b == 0 || b >= 0x7F80u) ? 0 : min(64, 141 - (int)(b >> 7));
  const float up = dq_pow2(f);
  if (threadIdx.x == 0) P.xfac[l][t] = dq_pow2(-f);
  for (int c = threadIdx.x; c < chunks; c += kDqXThreads) {
    const uint4 v = __ldg(src + c);
    uint4 o;
    o.x = dq_bf16x2_to_f16x2(v.x, up);
    o.y = dq_bf16x2_to_f16x2(v.y, up);
    o.z = dq_bf16x2_to_f16x2(v.z, up);
    o.w = dq_bf16x2_to_f16x2(v.w, up);
    dst[c] = o;
  }
}

}  // namespace f2i
