// Layer evaluation for small token counts (decode).
//
// y = sum_t [ s_re A_re + i s_im A_im ]_U + [ s_re conj(A_re) + i s_im conj(A_im) ]_W
// ("Fairy2i-W2" model card, y = Ux + W conj(x); "Fairy2i: Ultra-Low-Bit LLM
// Quantization Using Complex Weights {±1, ±i}", "Industry implications:
// multiplication-free inference"), where A_re / A_im are signed sums of x over
// the real-coded / imaginary-coded columns of one (matrix, stage) plane.
// In real terms, with a = Re x, b = Im x:
//   U plane: Re y += s_re <re-row, a> - s_im <im-row, b>
//            Im y += s_re <re-row, b> + s_im <im-row, a>
//   W plane: Re y += s_re <re-row, a> + s_im <im-row, b>
//            Im y += -s_re <re-row, b> + s_im <im-row, a>
// where re-row / im-row are the ternary {-1, 0, +1} rows of signs on the
// real-coded / imaginary-coded columns.
#pragma once
#include <cstdint>
#include "layout.cuh"

namespace f2i {

constexpr int kMaxGroup = 32;

struct LinearProblem {
  const uint8_t* codes;
  const float* scales;
  const uint16_t* x;  // bfloat16 bits [M][2m]
  float* y;           // [M][2n]
  int64_t n, m;
  int32_t T;
  int32_t cta_begin;   // first CTA of this problem in the launch
  int32_t rg_per_cta;  // row groups per CTA (decode partition)
  int32_t pad_;
};

struct LinearGroup {
  int32_t count;
  int32_t M;
  LinearProblem p[kMaxGroup];
};

__device__ __forceinline__ int find_problem(const LinearGroup& G) {
  int pi = 0;
  for (int i = 1; i < G.count; ++i)
    if ((int)blockIdx.x >= G.p[i].cta_begin) pi = i;
  return pi;
}

// Words of lane `lane` for chunk c (column blocks 4c .. 4c+3) of row group rg
// in one plane; nb = number of valid blocks (4 except in the tail chunk).
__device__ __forceinline__ uint4 load_chunk(const uint8_t* plane, int64_t rg, int64_t c, int lane, int64_t KB,
                                            int& nb) {
  const uint8_t* base = plane + rg * KB * kTileBytes;
  const int64_t full = KB >> 2;
  uint4 w = make_uint4(0, 0, 0, 0);
  if (c < full) {
    nb = 4;
    w = __ldcs(reinterpret_cast<const uint4*>(base + c * 512 + lane * 16));
  } else {
    const int r = (int)(KB - (full << 2));
    nb = r;
    const uint32_t* t = reinterpret_cast<const uint32_t*>(base + full * 512 + lane * 4 * r);
    w.x = __ldcs(t);
    if (r > 1) w.y = __ldcs(t + 1);
    if (r > 2) w.z = __ldcs(t + 2);
  }
  return w;
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int b) {
  return b == 0 ? w.x : b == 1 ? w.y : b == 2 ? w.z : w.w;
}

// Adds the y contributions of one plane for one token: ra/rb = <re-row, a/b>,
// ia/ib = <im-row, a/b>.
__device__ __forceinline__ void plane_epilogue(int X, float s_re, float s_im, float ra, float rb, float ia, float ib,
                                               float& y_re, float& y_im) {
  if (X == 0) {  // s_re A_re + i s_im A_im
    y_re += s_re * ra - s_im * ib;
    y_im += s_re * rb + s_im * ia;
  } else {  // s_re conj(A_re) + i s_im conj(A_im)
    y_re += s_re * ra + s_im * ib;
    y_im += -s_re * rb + s_im * ia;
  }
}

// ---------------------------------------------------------------------------
// ALGO_ADDSUB: CUDA cores, adds and subtracts only (the pages' inference
// arithmetic taken literally).  One warp per row group (8 rows); lane (g, q)
// owns row 8 rg + g and the 16 columns of its word in every block.  x is
// staged in shared memory as packed bfloat16 (a, b) pairs; each code flips
// the sign bit of a and b and adds them to the real-axis or the
// imaginary-axis accumulator.  A quad shuffle sums the four lanes of a row.
// Compute-bound at about 6-8 instructions per code per token.
// ---------------------------------------------------------------------------
constexpr int kAddSubWarps = 8;
constexpr int kAddSubTok = 2;

__global__ void __launch_bounds__(kAddSubWarps * 32) linear_addsub_kernel(const __grid_constant__ LinearGroup G) {
  extern __shared__ __align__(16) uint32_t xs[];  // [kAddSubTok][m_pad] (a | b << 16)
  const LinearProblem& P = G.p[find_problem(G)];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = P.n, m = P.m;
  const int T = P.T, M = G.M;
  const int64_t KB = col_blocks(m), m_pad = KB * 64, RG = row_groups(n);
  const int64_t rg = (int64_t)(blockIdx.x - P.cta_begin) * kAddSubWarps + warp;
  const int g = lane >> 2, q = lane & 3;
  const int64_t j = rg * 8 + g;
  const int64_t pbytes = plane_bytes(n, m);
  const int64_t nchunks = (KB + 3) >> 2;

  for (int tok0 = 0; tok0 < M; tok0 += kAddSubTok) {
    const int ntok = min(kAddSubTok, M - tok0);
    __syncthreads();
    for (int64_t idx = tid; idx < kAddSubTok * m_pad; idx += kAddSubWarps * 32) {
      const int tok = (int)(idx / m_pad);
      const int64_t k = idx - tok * m_pad;
      uint32_t v = 0;
      if (tok < ntok && k < m) {
        const uint16_t* xr = P.x + (int64_t)(tok0 + tok) * 2 * m;
        v = (uint32_t)xr[k] | ((uint32_t)xr[m + k] << 16);
      }
      xs[idx] = v;
    }
    __syncthreads();
    if (rg >= RG) continue;

    float y_re[kAddSubTok], y_im[kAddSubTok];
#pragma unroll
    for (int tk = 0; tk < kAddSubTok; ++tk) y_re[tk] = y_im[tk] = 0.0f;

    for (int plane = 0; plane < 2 * T; ++plane) {
      const int X = plane / T, t = plane - X * T;
      const uint8_t* pl = P.codes + (int64_t)plane * pbytes;
      float acc[kAddSubTok][4];
#pragma unroll
      for (int tk = 0; tk < kAddSubTok; ++tk) acc[tk][0] = acc[tk][1] = acc[tk][2] = acc[tk][3] = 0.0f;
      for (int64_t c = 0; c < nchunks; ++c) {
        int nb;
        const uint4 wv = load_chunk(pl, rg, c, lane, KB, nb);
        for (int b = 0; b < nb; ++b) {
          const uint32_t w = word_of(wv, b);
          const int64_t kbase = (4 * c + b) * 64;
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const uint32_t v = (w >> code_shift(cc)) & 3u;
            const uint32_t sgn = (v >> 1) << 31;
            const bool real = v & 1u;
            const int64_t k = kbase + code_col(cc, q);
#pragma unroll
            for (int tk = 0; tk < kAddSubTok; ++tk) {
              const uint32_t xv = xs[tk * m_pad + k];
              const float a = __uint_as_float((xv << 16) ^ sgn);
              const float bb = __uint_as_float((xv & 0xFFFF0000u) ^ sgn);
              acc[tk][0] += real ? a : 0.0f;
              acc[tk][1] += real ? bb : 0.0f;
              acc[tk][2] += real ? 0.0f : a;
              acc[tk][3] += real ? 0.0f : bb;
            }
          }
        }
      }
      float s_re = 0.0f, s_im = 0.0f;
      if (j < n) {
        s_re = P.scales[((int64_t)(X * T + t) * 2 + 0) * n + j];
        s_im = P.scales[((int64_t)(X * T + t) * 2 + 1) * n + j];
      }
#pragma unroll
      for (int tk = 0; tk < kAddSubTok; ++tk) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc[tk][u] += __shfl_xor_sync(0xffffffffu, acc[tk][u], 1);
          acc[tk][u] += __shfl_xor_sync(0xffffffffu, acc[tk][u], 2);
        }
        plane_epilogue(X, s_re, s_im, acc[tk][0], acc[tk][1], acc[tk][2], acc[tk][3], y_re[tk], y_im[tk]);
      }
    }
    if (q == 0 && j < n) {
      for (int tk = 0; tk < ntok; ++tk) {
        float* yr = P.y + (int64_t)(tok0 + tk) * 2 * n;
        yr[j] = y_re[tk];
        yr[n + j] = y_im[tk];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// ALGO_MMA: tensor-core decode with mma.sync m16n8k16 bf16:
//   A (16 x 16): row g = real-axis row of output 8 rg + g, row g + 8 its
//     imaginary-axis row; entries {+2, -2, +0, -0} (bfloat16 2.0 = 0x4000),
//     one shift and two LOP3 per pair of codes (see layout.cuh).
//   B (16 x 8): column 2 q' + p = part p (0: a = Re x, 1: b = Im x) of token
//     q' of the tile, taken unchanged from the bfloat16 activations.
//   D (16 x 8): fp32; lane (g, q) ends with <re-row, a>, <re-row, b>,
//     <im-row, a>, <im-row, b> of token q, each times 2.  Products of +-2 and
//     a bfloat16 are exact, so only the fp32 accumulation rounds.
// Partition: the host gives each problem of the launch a number of CTAs in
// proportion to its bytes and each CTA a run of `rg_per_cta` row groups, so
// that one wave fills the GPU with no output row split across CTAs.  The 8
// warps of a CTA split its (row group, column chunk) items evenly, stream
// the 2T code planes with 16-byte loads two items ahead, fold each row
// group's share into per-warp partial outputs in shared memory, and one
// fixed-order sum at the end writes y (bitwise reproducible).
// ---------------------------------------------------------------------------
constexpr int kMmaWarps = 8;
constexpr int kMaxRowGroupsPerCta = 16;

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Real-axis operand of the code pair in bits (15,14) / (31,30).
__device__ __forceinline__ uint32_t re_operand(uint32_t w) { return w & 0xC000C000u; }
// Imaginary-axis operand: keep the sign, set the 2.0 exponent bit where the
// real-axis flag is clear (one LOP3).
__device__ __forceinline__ uint32_t im_operand(uint32_t w) { return (w & 0x80008000u) | (~w & 0x40004000u); }

// Row stride (bfloat16 elements) of the staged activations: 16 bytes of
// padding make the 8 (token, part) rows of a tile hit distinct banks.
__host__ __device__ __forceinline__ int64_t x_stride(int64_t m) { return col_blocks(m) * 64 + 8; }

template <int NPL, int TILES>
__global__ void __launch_bounds__(kMmaWarps * 32, (NPL * TILES <= 4) ? 2 : 1)
    linear_mma_kernel(const __grid_constant__ LinearGroup G) {
  extern __shared__ __align__(16) unsigned char msm[];

  const LinearProblem& P = G.p[find_problem(G)];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int64_t n = P.n, m = P.m;
  const int T = P.T, M = G.M;
  const int64_t KB = col_blocks(m), RG = row_groups(n);
  const int64_t pbytes = plane_bytes(n, m);
  const int nch = (int)((KB + 3) >> 2);
  const int64_t rg_begin = (int64_t)(blockIdx.x - P.cta_begin) * P.rg_per_cta;
  const int64_t rg_end = min(RG, rg_begin + P.rg_per_cta);
  const int niter = (int)(rg_end - rg_begin);
  const int64_t xstr = x_stride(m);

  uint16_t* xs = reinterpret_cast<uint16_t*>(msm);  // [M][2][xstr]
  // red: [niter][kMmaWarps][TILES][32 lanes] x (re, im)
  float2* red = reinterpret_cast<float2*>(msm + (((size_t)M * 2 * xstr * sizeof(uint16_t) + 15) & ~(size_t)15));

  // This warp's contiguous share of the CTA's (row group, chunk) items,
  // walked with incremental counters.
  const int items = niter * nch;
  const int i0 = (int)((int64_t)items * warp / kMmaWarps), i1 = (int)((int64_t)items * (warp + 1) / kMmaWarps);
  const int full = (int)(KB >> 2);
  const int tail = (int)(KB - 4 * full);
  const uint32_t row_stride = (uint32_t)KB * kTileBytes;
  const uint32_t lane16 = (uint32_t)lane * 16u;
  const uint32_t tail_off = (uint32_t)full * 512u + (uint32_t)lane * 4u * (uint32_t)tail;
  const uint8_t* plane0 = P.codes + rg_begin * (int64_t)row_stride;

  auto load_at = [&](int r, int c, uint4 (&dst)[NPL]) {
    const uint32_t off = (uint32_t)r * row_stride + (c < full ? (uint32_t)c * 512u + lane16 : tail_off);
#pragma unroll
    for (int pl = 0; pl < NPL; ++pl) {
      const uint8_t* a = plane0 + pl * pbytes + off;
      if (c < full) {
        dst[pl] = __ldcs(reinterpret_cast<const uint4*>(a));
      } else {
        const uint32_t* t = reinterpret_cast<const uint32_t*>(a);
        dst[pl].x = __ldcs(t);
        dst[pl].y = tail > 1 ? __ldcs(t + 1) : 0u;
        dst[pl].z = tail > 2 ? __ldcs(t + 2) : 0u;
        dst[pl].w = 0u;
      }
    }
  };
  auto advance = [&](int& r, int& c) {
    if (++c == nch) {
      c = 0;
      ++r;
    }
  };

  // Start streaming codes before staging the activations.
  int rc = i0 / nch, cc = i0 - (i0 / nch) * nch;  // item being processed
  int rl = rc, cl = cc;                           // next item to load
  uint4 cur[NPL], nx1[NPL];
  if (i0 < i1) {
    load_at(rl, cl, cur);
    advance(rl, cl);
  }
  if (i0 + 1 < i1) {
    load_at(rl, cl, nx1);
    advance(rl, cl);
  }

  // Stage x (bfloat16, unchanged) and clear the partial outputs.
  {
    const bool vec = (m & 7) == 0 && ((reinterpret_cast<uintptr_t>(P.x) & 15) == 0);
    const int64_t rows = (int64_t)M * 2;
    if (vec) {
      const int64_t per_row = xstr >> 3;  // uint4 per staged row
      for (int64_t idx = tid; idx < rows * per_row; idx += kMmaWarps * 32) {
        const int64_t row = idx / per_row, k8 = (idx - row * per_row) << 3;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k8 < m) v = *reinterpret_cast<const uint4*>(P.x + (row >> 1) * 2 * m + (row & 1) * m + k8);
        *reinterpret_cast<uint4*>(xs + row * xstr + k8) = v;
      }
    } else {
      for (int64_t idx = tid; idx < rows * xstr; idx += kMmaWarps * 32) {
        const int64_t row = idx / xstr, k = idx - row * xstr;
        xs[idx] = k < m ? P.x[(row >> 1) * 2 * m + (row & 1) * m + k] : (uint16_t)0;
      }
    }
    for (int z = tid; z < niter * kMmaWarps * TILES * 32; z += kMmaWarps * 32) red[z] = make_float2(0.0f, 0.0f);
  }
  __syncthreads();

  // B rows of this lane: token 4 tl + (g >> 1), part g & 1 (zero past M).
  const uint16_t* xrow[TILES];
  uint32_t bmask[TILES];
#pragma unroll
  for (int tl = 0; tl < TILES; ++tl) {
    const int tok = 4 * tl + (g >> 1);
    const int tc = min(tok, M - 1);
    xrow[tl] = xs + ((int64_t)tc * 2 + (g & 1)) * xstr + 2 * q;
    bmask[tl] = tok < M ? 0xFFFFFFFFu : 0u;
  }

  float sc[NPL][2];
  auto load_scales = [&](int r) {
    const int64_t j = (rg_begin + r) * 8 + g;
#pragma unroll
    for (int pl = 0; pl < NPL; ++pl) {
      sc[pl][0] = j < n ? P.scales[((int64_t)pl * 2 + 0) * n + j] : 0.0f;
      sc[pl][1] = j < n ? P.scales[((int64_t)pl * 2 + 1) * n + j] : 0.0f;
    }
  };
  float acc[NPL][TILES][4];
#pragma unroll
  for (int pl = 0; pl < NPL; ++pl)
#pragma unroll
    for (int tl = 0; tl < TILES; ++tl) acc[pl][tl][0] = acc[pl][tl][1] = acc[pl][tl][2] = acc[pl][tl][3] = 0.0f;
  if (i0 < i1) load_scales(rc);

  // One 64-column block: four k16 steps, two code pairs per step.
  auto mma_block = [&](const uint32_t (&w)[NPL], int kk0) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t b01[TILES], b23[TILES];
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl) {
        b01[tl] = *reinterpret_cast<const uint32_t*>(xrow[tl] + kk0 + 16 * s) & bmask[tl];
        b23[tl] = *reinterpret_cast<const uint32_t*>(xrow[tl] + kk0 + 16 * s + 8) & bmask[tl];
      }
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const uint32_t w0 = w[pl] << (4 * s), w1 = w[pl] << (4 * s + 2);
        const uint32_t re0 = re_operand(w0), im0 = im_operand(w0);
        const uint32_t re1 = re_operand(w1), im1 = im_operand(w1);
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) mma_bf16(acc[pl][tl], re0, im0, re1, im1, b01[tl], b23[tl]);
      }
    }
  };

  for (int i = i0; i < i1; ++i) {
    uint4 nx2[NPL];
    if (i + 2 < i1) {
      load_at(rl, cl, nx2);
      advance(rl, cl);
    }
    const int kc = 256 * cc;  // first column of this chunk
    if (cc < full) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t w[NPL];
#pragma unroll
        for (int pl = 0; pl < NPL; ++pl) w[pl] = word_of(cur[pl], b);
        mma_block(w, kc + 64 * b);
      }
    } else {
#pragma unroll
      for (int b = 0; b < 3; ++b) {
        if (b < tail) {
          uint32_t w[NPL];
#pragma unroll
          for (int pl = 0; pl < NPL; ++pl) w[pl] = word_of(cur[pl], b);
          mma_block(w, kc + 64 * b);
        }
      }
    }

    // end of this warp's segment of row group rc: fold into y partials
    const int r = rc;
    advance(rc, cc);
    if (i + 1 == i1 || rc != r) {
      float y_re[TILES], y_im[TILES];
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl) y_re[tl] = y_im[tl] = 0.0f;
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const int X = pl / T;
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) {
          plane_epilogue(X, sc[pl][0], sc[pl][1], 0.5f * acc[pl][tl][0], 0.5f * acc[pl][tl][1],
                         0.5f * acc[pl][tl][2], 0.5f * acc[pl][tl][3], y_re[tl], y_im[tl]);
          acc[pl][tl][0] = acc[pl][tl][1] = acc[pl][tl][2] = acc[pl][tl][3] = 0.0f;
        }
      }
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl)
        red[((r * kMmaWarps + warp) * TILES + tl) * 32 + lane] = make_float2(y_re[tl], y_im[tl]);
      if (i + 1 < i1) load_scales(rc);
    }
#pragma unroll
    for (int pl = 0; pl < NPL; ++pl) {
      cur[pl] = nx1[pl];
      nx1[pl] = nx2[pl];
    }
  }
  __syncthreads();

  // fixed-order sum over the warps' partials, then store
  for (int e = tid; e < niter * TILES * 32; e += kMmaWarps * 32) {
    const int ln = e & 31;
    const int tl = (e >> 5) % TILES;
    const int r = (e >> 5) / TILES;
    const int tok = 4 * tl + (ln & 3);
    const int64_t j = (rg_begin + r) * 8 + (ln >> 2);
    float re = 0.0f, im = 0.0f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) {
      const float2 v = red[((r * kMmaWarps + w) * TILES + tl) * 32 + ln];
      re += v.x;
      im += v.y;
    }
    if (tok < M && j < n) {
      float* yr = P.y + (int64_t)tok * 2 * n;
      yr[j] = re;
      yr[n + j] = im;
    }
  }
}

}  // namespace f2i
