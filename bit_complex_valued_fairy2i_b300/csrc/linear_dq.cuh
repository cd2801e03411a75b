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
// 5th-generation tensor cores run with bfloat16 operands: R^ = hi + lo, hi the
// bfloat16 rounding of R^ (formed in fp32) and lo the bfloat16 rounding of the
// remainder, so R^ is carried to ~2^-18 relative and every product is exact
// in the fp32 accumulators.  Executed flops: 2 terms x 2 (2n)(2m) per token =
// 16 n m, against 16 n m T for the ternary form of linear_prefill.cuh.
//
// GEMM shape per tile: D[128 rows][256 tokens] += A[128][K] * B[256][K]^T
//   rows: 64 outputs j, row 2 jl = Re y_j, row 2 jl + 1 = Im y_j, so that one
//         decode of (U^, W^)[j][c] yields the entries of both rows for both
//         halves of x~;
//   K:    blocks of 64 columns in pairs (block c of Re x, block c of Im x),
//         the two stages of a pair filled by one decode;
//   A:    hi and lo, 128-byte swizzled K-major, written by 8 producer warps
//         from the layout-3 codes and the scales;
//   B:    x [M][2m] bfloat16 by TMA (128-byte swizzle, zero fill past the
//         edges); columns past m of a Re-x block are cancelled by zero rows of A;
//   D:    fp32 in TMEM, two accumulators of 256 columns (double buffered).
// Warp roles (14 warps, one CTA per SM, persistent over tiles): warp 0 TMA
// for B, warp 1 TMEM allocation and MMA issue, warps 2-9 A producers, warps
// 10-13 epilogue (tcgen05.ld, stores of y).  All mbarrier waits are bounded.
#pragma once
#include <cuda.h>
#include <cstdint>
#include "layout.cuh"
#include "linear_prefill.cuh"

namespace f2i {

constexpr int kDqMaxGroup = 8;
constexpr int kDqStages = 3;
constexpr int kDqBM = 128;  // real rows per tile (64 outputs)
constexpr int kDqBN = 256;  // tokens per tile
constexpr int kDqBK = 64;   // columns per k-block
constexpr int kDqATerm = kDqBM * kDqBK * 2;   // 16 KB: one term of A
constexpr int kDqAStage = 2 * kDqATerm;       // hi and lo
constexpr int kDqBStage = kDqBN * kDqBK * 2;  // 32 KB
constexpr int kDqProducerWarps = 8;
constexpr int kDqThreads = 32 * (6 + kDqProducerWarps);
constexpr uint32_t kDqTmemCols = 512;
constexpr size_t kDqSmemBytes = 1024 + (size_t)kDqStages * (kDqAStage + kDqBStage) + 256;

struct DqProblem {
  const uint8_t* codes;  // layout 3
  const float* scales;
  float* y;
  int32_t n, m;
  int64_t tile_begin;
  int32_t row_tiles;  // tiles of 64 outputs
  int32_t tok_tiles;  // tiles of 256 tokens
  int32_t kpairs;     // blocks of 64 columns per half of x~
  int32_t pad_;
};

struct DqParams {
  CUtensorMap tmap[kDqMaxGroup];  // x of each problem as a [M][2m] bfloat16 tensor
  DqProblem p[kDqMaxGroup];
  int64_t total_tiles;
  int32_t count, T, M, pad_;
};

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

// bfloat16 bits of v rounded to nearest even, and of the remainder.
__device__ __forceinline__ void dq_split(float v, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  const float hf = __bfloat162float(h);
  __nv_bfloat16 l = __float2bfloat16_rn(v - hf);  // v - hf is exact in fp32
  hi = (uint32_t)__bfloat16_as_ushort(h);
  lo = (uint32_t)__bfloat16_as_ushort(l);
}

template <int T>
__global__ void __launch_bounds__(kDqThreads, 1) linear_dq_kernel(const __grid_constant__ DqParams P) {
  extern __shared__ uint8_t dq_smem_raw[];
  constexpr int NP = 2 * T;
  constexpr uint32_t kIdesc = idesc_bf16(kDqBM, kDqBN);

  const uint32_t raw = smem_u32(dq_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dq_smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + kDqStages * kDqAStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kDqStages * (kDqAStage + kDqBStage));
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(kDqStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kDqStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kDqStages + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kDqStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(full_bar(s), 1 + kDqProducerWarps);  // TMA arrive.expect_tx + one arrive per producer warp
      mbar_init(empty_bar(s), 1);                    // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < P.count; ++i) tma_prefetch_map(&P.tmap[i]);
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
      uint32_t it = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
        const DqTile c = dq_tile(P, tile);
        const DqProblem& pr = P.p[c.pi];
        for (int kb = 0; ok && kb < 2 * pr.kpairs; ++kb, ++it) {
          const int s = (int)(it % kDqStages);
          const uint32_t ph = (it / kDqStages) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), (uint32_t)kDqBStage);
          const int col = (kb & 1) * pr.m + (kb >> 1) * kDqBK;
          tma_load_2d(sB + (uint32_t)s * kDqBStage, &P.tmap[c.pi], full_bar(s), col, c.tt * kDqBN);
        }
      }
      for (uint32_t k = (it > (uint32_t)kDqStages ? it - kDqStages : 0u); k < it; ++k)
        if (!mbar_wait(full_bar((int)(k % kDqStages)), (k / kDqStages) & 1u, abort_flag)) break;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: hi and lo into one accumulator ----------------
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x, ++lt) {
        const DqTile c = dq_tile(P, tile);
        const int kbs = 2 * P.p[c.pi].kpairs;
        const int b = (int)(lt & 1u);
        if (!mbar_wait(acce_bar(b), ((lt >> 1) & 1u) ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)b * kDqBN;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int s = (int)(it % kDqStages);
          const uint32_t ph = (it / kDqStages) & 1u;
          if (!mbar_wait(full_bar(s), ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + (uint32_t)s * kDqAStage, b0 = sB + (uint32_t)s * kDqBStage;
#pragma unroll
          for (int kk = 0; kk < kDqBK / 16; ++kk) {
            tc_mma_bf16(d_tmem, sw128_desc(a0 + 32u * kk), sw128_desc(b0 + 32u * kk), kIdesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
            tc_mma_bf16(d_tmem, sw128_desc(a0 + kDqATerm + 32u * kk), sw128_desc(b0 + 32u * kk), kIdesc, 1u);
          }
          tc_commit(empty_bar(s));
        }
        if (ok) tc_commit(accf_bar(b));
      }
    }
  } else if (warp < 2 + kDqProducerWarps) {
    // ---------------- A producers: codes + scales -> R^ hi / lo ----------------
    // Thread (jl, qt) owns output jl of the tile (rows 2 jl, 2 jl + 1) and
    // columns 16 qt .. 16 qt + 15 of every 64-column block, i.e. groups
    // 2 qt, 2 qt + 1 of the block: one 16-byte layout-3 chunk per plane.
    const int pt = tid - 64;  // 0..255
    const int jl = pt >> 2, qt = pt & 3;
    const uint32_t row0 = (uint32_t)(2 * jl), row1 = row0 + 1u;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
      const DqTile c = dq_tile(P, tile);
      const DqProblem& pr = P.p[c.pi];
      const int64_t n = pr.n, m = pr.m;
      const int64_t j = (int64_t)c.rt * 64 + jl;
      const bool live = j < n;
      const int r = (int)(j & 31);
      // the row's scales (zero past n): [plane][axis]
      float sre[NP], sim[NP];
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        sre[p] = live ? __ldg(pr.scales + (int64_t)(2 * p) * n + j) : 0.0f;
        sim[p] = live ? __ldg(pr.scales + (int64_t)(2 * p + 1) * n + j) : 0.0f;
      }
      for (int kp = 0; ok && kp < pr.kpairs; ++kp) {
        // decode 16 columns: (Re, Im) of U^ and W^ in fp32
        const int64_t c0 = (int64_t)kp * 64 + 16 * qt;  // first column of this thread
        float ur[16], ui[16], wr[16], wi[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) ur[e] = ui[e] = wr[e] = wi[e] = 0.0f;
        if (live && c0 < m) {
          const int64_t g0 = c0 >> 3;  // global group of the first 8 columns
          const int64_t w = g0 >> 5;
          const int gw = (int)(g0 & 31);
          const int nb = l3_slots(m, w);
          const uint32_t slot_off = (uint32_t)l3_slot_of(gw, r, nb) * kL3SlotBytes + (uint32_t)r * 16u;
          const int by0 = l3_byte_of(gw, r), by1 = l3_byte_of(gw + 1, r);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(pr.codes + l3_offset(n, m, T, w, j >> 5, p) + slot_off));
            const uint32_t sw[2] = {v.x, v.y}, qw[2] = {v.z, v.w};
            const uint32_t s16 = ((sw[by0 >> 2] >> (8 * (by0 & 3))) & 0xFFu) | (((sw[by1 >> 2] >> (8 * (by1 & 3))) & 0xFFu) << 8);
            const uint32_t q16 = ((qw[by0 >> 2] >> (8 * (by0 & 3))) & 0xFFu) | (((qw[by1 >> 2] >> (8 * (by1 & 3))) & 0xFFu) << 8);
            const uint32_t f16 = s16 ^ q16;  // imaginary-axis flags
            const bool isU = p < T;
            // columns past m read as zero (their codes are zero bits, i.e. +1)
            const uint32_t cmask = m - c0 >= 16 ? 0xFFFFu : ((1u << (uint32_t)(m - c0)) - 1u);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              if (!((cmask >> e) & 1u)) continue;
              const uint32_t sneg = (s16 >> e) & 1u, fim = (f16 >> e) & 1u;
              const float mag = fim ? sim[p] : sre[p];
              const float val = __uint_as_float(__float_as_uint(mag) ^ (sneg << 31));
              if (isU) {
                ur[e] += fim ? 0.0f : val;
                ui[e] += fim ? val : 0.0f;
              } else {
                wr[e] += fim ? 0.0f : val;
                wi[e] += fim ? val : 0.0f;
              }
            }
          }
        }
        // both stages of the pair: k-block 2 kp (Re x columns) and 2 kp + 1 (Im x columns)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int s = (int)(it % kDqStages);
          const uint32_t ph = (it / kDqStages) & 1u;
          ++it;
          bool got = true;
          if (lane == 0) got = mbar_wait(empty_bar(s), ph ^ 1u, abort_flag);
          got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
          if (!got) {
            ok = false;
            break;
          }
          // row 2 jl: Re y, row 2 jl + 1: Im y
          //   Re x block: R^11 = ReU + ReW, R^21 = ImU + ImW
          //   Im x block: R^12 = ImW - ImU, R^22 = ReU - ReW
          uint32_t h0[8], l0[8], h1[8], l1[8];  // packed pairs of bfloat16 for 16 columns
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float a0, a1, b0v, b1v;
            if (h == 0) {
              a0 = ur[e] + wr[e];
              a1 = ur[e + 1] + wr[e + 1];
              b0v = ui[e] + wi[e];
              b1v = ui[e + 1] + wi[e + 1];
            } else {
              a0 = wi[e] - ui[e];
              a1 = wi[e + 1] - ui[e + 1];
              b0v = ur[e] - wr[e];
              b1v = ur[e + 1] - wr[e + 1];
            }
            uint32_t x0, y0, x1, y1;
            dq_split(a0, x0, y0);
            dq_split(a1, x1, y1);
            h0[e >> 1] = x0 | (x1 << 16);
            l0[e >> 1] = y0 | (y1 << 16);
            dq_split(b0v, x0, y0);
            dq_split(b1v, x1, y1);
            h1[e >> 1] = x0 | (x1 << 16);
            l1[e >> 1] = y0 | (y1 << 16);
          }
          const uint32_t st = sA + (uint32_t)s * kDqAStage;
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const uint32_t cc = (uint32_t)(2 * qt + hc);  // 16-byte chunk of the 128-byte row
            const uint32_t o0 = row0 * 128u + ((cc ^ (row0 & 7u)) << 4), o1 = row1 * 128u + ((cc ^ (row1 & 7u)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o0), "r"(h0[4 * hc]), "r"(h0[4 * hc + 1]),
                         "r"(h0[4 * hc + 2]), "r"(h0[4 * hc + 3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + o1), "r"(h1[4 * hc]), "r"(h1[4 * hc + 1]),
                         "r"(h1[4 * hc + 2]), "r"(h1[4 * hc + 3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + kDqATerm + o0), "r"(l0[4 * hc]),
                         "r"(l0[4 * hc + 1]), "r"(l0[4 * hc + 2]), "r"(l0[4 * hc + 3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + kDqATerm + o1), "r"(l1[4 * hc]),
                         "r"(l1[4 * hc + 1]), "r"(l1[4 * hc + 2]), "r"(l1[4 * hc + 3])
                         : "memory");
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
        }
      }
    }
  } else {
    // ---------------- epilogue: D row 2 jl + part of token t -> y[t][part n + j] ----------------
    const int eq = warp & 3;  // TMEM lanes 32 eq .. 32 eq + 31
    const int rl = 32 * eq + lane;
    const int jl = rl >> 1, part = rl & 1;
    uint32_t lt = 0;
    for (int64_t tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x, ++lt) {
      const DqTile c = dq_tile(P, tile);
      const DqProblem& pr = P.p[c.pi];
      const int b = (int)(lt & 1u);
      const int64_t j = (int64_t)c.rt * 64 + jl;
      bool got = true;
      if (lane == 0) got = mbar_wait(accf_bar(b), (lt >> 1) & 1u, abort_flag);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * eq) << 16) + (uint32_t)b * kDqBN;
      const int64_t ystride = 2 * (int64_t)pr.n;
      float* ycol = pr.y + (int64_t)part * pr.n + j;
#pragma unroll 1
      for (int cc = 0; cc < kDqBN / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tbase + 32u * cc, v);
        tmem_ld_wait();
        if (j < pr.n) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int64_t tok = (int64_t)c.tt * kDqBN + 32 * cc + e;
            if (tok < P.M) ycol[tok * ystride] = __uint_as_float(v[e]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kDqTmemCols);
  }
}

}  // namespace f2i
