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
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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
  int32_t rg_per_cta;  // row groups per CTA (persistent partition)
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

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

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

// Adds y contributions of one plane for one token: ra/rb = <re-row, a/b>,
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
// owns row 8 rg + g and the columns 64 kb + 16 p + 4 q + i of every block.
// x is staged in shared memory as packed bfloat16 (a, b) pairs; each code
// flips the sign bit of a and b and adds them to the real-axis or the
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
          const int64_t kbase = (4 * c + b) * 64 + 4 * q;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t v = (w >> code_shift(i, p)) & 3u;
              const uint32_t sgn = (v >> 1) << 31;
              const bool real = v & 1u;
              const int64_t k = kbase + 16 * p + i;
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
// ALGO_MMA_FP8: tensor-core decode.  The same signed sums, computed by
// mma.sync m16n8k32 with e4m3 operands:
//   A (16 x 32): rows g = real-axis row of output 8 rg + g, rows g + 8 = its
//     imaginary-axis row; entries {+2, -2, +0, -0} made from the packed codes
//     by one LOP3 per four codes (bits (7,6) of a byte are (sign, real flag):
//     `w & 0xC0C0C0C0` keeps +-2 on real-coded columns, the complementary
//     LOP3 keeps +-2 on imaginary-coded ones).
//   B (32 x 8): columns = (token, part in {a, b}, hi/lo) for two tokens; the
//     bfloat16 x of each (token, part) is scaled by a power of two 2^s so its
//     largest magnitude lands in [128, 256) and split exactly into
//     hi = e4m3(x 2^s) and lo = e4m3(16 (x 2^s - hi)).
//   D (16 x 8): fp32.  <row, x_part> = 2^-s (D_hi + D_lo / 16) / 2.
//
// Persistent partition: the host gives each problem of the launch a number of
// CTAs proportional to its bytes, and each CTA a contiguous run of
// `rg_per_cta` row groups of one problem, so one launch fills the GPU in a
// single wave with balanced work and no output row split across CTAs.  Each
// CTA builds its problem's x fragments once in shared memory, then walks its
// row groups RGC at a time, the KS = 8 / RGC warps of a row group splitting
// its column chunks and reducing through shared memory.
// ---------------------------------------------------------------------------
constexpr int kMmaWarps = 8;

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// Imaginary-axis operand: keep the sign bit, set the 2.0 exponent bit where
// the real-axis flag is clear (one LOP3).
__device__ __forceinline__ uint32_t im_axis_operand(uint32_t w) {
  return (w & 0x80808080u) | (~w & 0x40404040u);
}

// Two floats -> two e4m3 (round to nearest even, saturating), low byte = a.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// hi/lo e4m3 split of 8 consecutive activations (already scaled by 2^s).
__device__ __forceinline__ void split8(const float (&v)[8], uint32_t (&hi)[2], uint32_t (&lo)[2]) {
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t h = 0, l = 0;
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const float a = v[4 * w + 2 * pr], b = v[4 * w + 2 * pr + 1];
      const uint32_t hb = e4m3x2(a, b);
      const float2 hf = e4m3x2_to_float2(hb);
      const uint32_t lb = e4m3x2((a - hf.x) * 16.0f, (b - hf.y) * 16.0f);
      h |= hb << (16 * pr);
      l |= lb << (16 * pr);
    }
    hi[w] = h;
    lo[w] = l;
  }
}

template <int TILES>
struct DecodeSmem {
  uint32_t absmax[2 * TILES][2];
  float inv[2 * TILES][2];  // 2^(-s-1) per (token, part)
  float up[2 * TILES][2];   // 2^s
};

// Builds the B fragments of x for all column steps in shared memory.
// xf (uint32 view): word h of lane (4g + q) of step st of tile tl at
// ((tl * nsteps + st) * 32 + lane) * 2 + h holds column g at rows
// 32 st + 16 h + 4 q + (0..3).
template <int TILES>
__device__ void build_x_fragments(const uint16_t* __restrict__ x, int64_t m, int M, int64_t nsteps,
                                  uint32_t* xf, DecodeSmem<TILES>& S) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int NT = kMmaWarps * 32;
  const bool vec = (m & 7) == 0 && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  // zero fill (padding columns, padding tokens)
  uint4* z = reinterpret_cast<uint4*>(xf);
  const int64_t nz = (int64_t)TILES * nsteps * 32 * 2 / 4;
  for (int64_t i = tid; i < nz; i += NT) z[i] = make_uint4(0, 0, 0, 0);
  if (tid < 4 * TILES) S.absmax[tid >> 1][tid & 1] = 0;
  __syncthreads();
  // largest magnitude per (token, part)
  for (int tp = 0; tp < 2 * M; ++tp) {
    const uint16_t* xr = x + (int64_t)(tp >> 1) * 2 * m + (tp & 1) * m;
    uint32_t mx = 0;
    if (vec) {
      for (int64_t k = (int64_t)tid * 8; k < m; k += NT * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) mx = max(mx, max(w[u] & 0x7FFFu, (w[u] >> 16) & 0x7FFFu));
      }
    } else {
      for (int64_t k = tid; k < m; k += NT) mx = max(mx, (uint32_t)(xr[k] & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) atomicMax(&S.absmax[tp >> 1][tp & 1], mx);
  }
  __syncthreads();
  if (tid < 4 * TILES) {
    const uint32_t mb = S.absmax[tid >> 1][tid & 1];
    const int ef = (int)(mb >> 7);
    int sh = ef > 0 ? 7 - (ef - 127) : 125;  // largest magnitude -> [128, 256)
    sh = max(-126, min(125, sh));
    S.inv[tid >> 1][tid & 1] = __uint_as_float((uint32_t)(126 - sh) << 23);  // 2^(-s-1)
    S.up[tid >> 1][tid & 1] = __uint_as_float((uint32_t)(127 + sh) << 23);   // 2^s
  }
  __syncthreads();
  // fragments: one work item = (token, part, 8 consecutive columns)
  const int64_t groups = (m + 7) >> 3;
  for (int64_t it = tid; it < (int64_t)2 * M * groups; it += NT) {
    const int tp = (int)(it / groups);
    const int64_t k0 = (it - (int64_t)tp * groups) << 3;
    const int tok = tp >> 1, part = tp & 1;
    const uint16_t* xr = x + (int64_t)tok * 2 * m + part * m;
    const float up = S.up[tok][part];
    float v[8];
    if (vec) {
      const uint4 raw = *reinterpret_cast<const uint4*>(xr + k0);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[2 * u] = __uint_as_float(w[u] << 16) * up;
        v[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u) * up;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (k0 + u < m) ? __uint_as_float((uint32_t)xr[k0 + u] << 16) * up : 0.0f;
    }
    uint32_t hi[2], lo[2];
    split8(v, hi, lo);
    const int64_t st = k0 >> 5;
    const int within = (int)(k0 & 31);
    const int h = within >> 4, q0 = (within & 15) >> 2;
    const int tl = tok >> 1;
    const int ghi = 4 * (tok & 1) + 2 * part;
    uint32_t* base = xf + ((int64_t)tl * nsteps + st) * 64 + h;
    base[(4 * ghi + q0) * 2] = hi[0];
    base[(4 * ghi + q0 + 1) * 2] = hi[1];
    base[(4 * (ghi + 1) + q0) * 2] = lo[0];
    base[(4 * (ghi + 1) + q0 + 1) * 2] = lo[1];
  }
  __syncthreads();
}

template <int NPL, int TILES, int RGC>
__global__ void __launch_bounds__(kMmaWarps * 32) linear_mma_fp8_kernel(const __grid_constant__ LinearGroup G) {
  constexpr int KS = kMmaWarps / RGC;
  extern __shared__ __align__(16) unsigned char msm[];
  __shared__ DecodeSmem<TILES> S;

  const LinearProblem& P = G.p[find_problem(G)];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = P.n, m = P.m;
  const int T = P.T, M = G.M;
  const int64_t KB = col_blocks(m), m_pad = KB * 64, nsteps = m_pad / 32, RG = row_groups(n);
  uint32_t* xf = reinterpret_cast<uint32_t*>(msm);  // [TILES][nsteps][32][2]
  float* red = reinterpret_cast<float*>(msm + (size_t)TILES * nsteps * 32 * sizeof(uint2));
  const uint2* xf2 = reinterpret_cast<const uint2*>(xf);

  build_x_fragments<TILES>(P.x, m, M, nsteps, xf, S);

  const int rgc = warp % RGC, ks = warp / RGC;
  const int g = lane >> 2, q = lane & 3;
  const int64_t pbytes = plane_bytes(n, m);
  const int64_t nchunks = (KB + 3) >> 2;
  const int64_t cps = (nchunks + KS - 1) / KS;
  const int64_t c0 = ks * cps, c1 = min(nchunks, c0 + cps);
  const int64_t rg_begin = (int64_t)(blockIdx.x - P.cta_begin) * P.rg_per_cta;
  const int64_t rg_end = min(RG, rg_begin + P.rg_per_cta);

  // Flat per-warp sequence of (row-group step r, chunk c) items with a
  // one-item prefetch that runs across row-group boundaries, so the loads of
  // the next row group are in flight during this one's reduction.
  const int64_t niter = (rg_end - rg_begin + RGC - 1) / RGC;
  const bool has_work = c0 < c1;
  uint4 cur[NPL];
  int nb = 4;
  if (has_work && niter > 0 && rg_begin + rgc < rg_end) {
#pragma unroll
    for (int pl = 0; pl < NPL; ++pl) cur[pl] = load_chunk(P.codes + pl * pbytes, rg_begin + rgc, c0, lane, KB, nb);
  }
  for (int64_t r = 0; r < niter; ++r) {
    const int64_t rg = rg_begin + r * RGC + rgc;
    const int64_t j = rg * 8 + g;
    const bool active = has_work && rg < rg_end;
    float y_re[TILES], y_im[TILES];
#pragma unroll
    for (int tl = 0; tl < TILES; ++tl) y_re[tl] = y_im[tl] = 0.0f;

    if (active) {
      float acc[NPL][TILES][4];
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl)
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) acc[pl][tl][0] = acc[pl][tl][1] = acc[pl][tl][2] = acc[pl][tl][3] = 0.0f;

      for (int64_t c = c0; c < c1; ++c) {
        // next item: (r, c + 1), else (r + 1, c0) when that row group exists
        uint4 nxt[NPL];
        int nbn = 4;
        const bool more_here = c + 1 < c1;
        const int64_t rg_next = rg + RGC;
        const bool more_next = !more_here && r + 1 < niter && rg_next < rg_end;
        if (more_here || more_next) {
          const int64_t rr = more_here ? rg : rg_next;
          const int64_t cc = more_here ? c + 1 : c0;
#pragma unroll
          for (int pl = 0; pl < NPL; ++pl) nxt[pl] = load_chunk(P.codes + pl * pbytes, rr, cc, lane, KB, nbn);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (b >= nb) break;
          const int64_t st = 2 * (4 * c + b);
          uint2 bx0[TILES], bx1[TILES];
#pragma unroll
          for (int tl = 0; tl < TILES; ++tl) {
            bx0[tl] = xf2[((int64_t)tl * nsteps + st) * 32 + lane];
            bx1[tl] = xf2[((int64_t)tl * nsteps + st + 1) * 32 + lane];
          }
#pragma unroll
          for (int pl = 0; pl < NPL; ++pl) {
            const uint32_t w0 = word_of(cur[pl], b);
            const uint32_t w1 = w0 << 2, w2 = w0 << 4, w3 = w0 << 6;
            const uint32_t r0 = w0 & 0xC0C0C0C0u, r1 = w1 & 0xC0C0C0C0u;
            const uint32_t r2 = w2 & 0xC0C0C0C0u, r3 = w3 & 0xC0C0C0C0u;
            const uint32_t i0 = im_axis_operand(w0), i1 = im_axis_operand(w1);
            const uint32_t i2 = im_axis_operand(w2), i3 = im_axis_operand(w3);
#pragma unroll
            for (int tl = 0; tl < TILES; ++tl) {
              mma_e4m3(acc[pl][tl], r0, i0, r1, i1, bx0[tl]);
              mma_e4m3(acc[pl][tl], r2, i2, r3, i3, bx1[tl]);
            }
          }
        }
        if (more_here || more_next) {
#pragma unroll
          for (int pl = 0; pl < NPL; ++pl) cur[pl] = nxt[pl];
          nb = nbn;
        }
      }

      // per-plane epilogue; lane q holds token 2 tl + (q >> 1), part q & 1
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const int X = pl / T, t = pl - X * T;
        float s_re = 0.0f, s_im = 0.0f;
        if (j < n) {
          s_re = P.scales[((int64_t)(X * T + t) * 2 + 0) * n + j];
          s_im = P.scales[((int64_t)(X * T + t) * 2 + 1) * n + j];
        }
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) {
          const int tok = 2 * tl + (q >> 1), part = q & 1;
          const float inv = S.inv[tok][part];
          const float vr = (acc[pl][tl][0] + acc[pl][tl][1] * 0.0625f) * inv;  // <re-row, x_part>
          const float vi = (acc[pl][tl][2] + acc[pl][tl][3] * 0.0625f) * inv;  // <im-row, x_part>
          if (part == 0) {
            y_re[tl] += s_re * vr;
            y_im[tl] += s_im * vi;
          } else if (X == 0) {
            y_re[tl] -= s_im * vi;
            y_im[tl] += s_re * vr;
          } else {
            y_re[tl] += s_im * vi;
            y_im[tl] -= s_re * vr;
          }
        }
      }
    }
    // combine parts a and b (lanes q, q ^ 1), then the column splits
#pragma unroll
    for (int tl = 0; tl < TILES; ++tl) {
      y_re[tl] += __shfl_xor_sync(0xffffffffu, y_re[tl], 1);
      y_im[tl] += __shfl_xor_sync(0xffffffffu, y_im[tl], 1);
    }
    if (KS > 1) {
      // red: [KS][RGC][TILES][2][32]
      if (ks > 0) {
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) {
          red[((((ks * RGC) + rgc) * TILES + tl) * 2 + 0) * 32 + lane] = y_re[tl];
          red[((((ks * RGC) + rgc) * TILES + tl) * 2 + 1) * 32 + lane] = y_im[tl];
        }
      }
      __syncthreads();
      if (ks == 0) {
        for (int s2 = 1; s2 < KS; ++s2) {
#pragma unroll
          for (int tl = 0; tl < TILES; ++tl) {
            y_re[tl] += red[((((s2 * RGC) + rgc) * TILES + tl) * 2 + 0) * 32 + lane];
            y_im[tl] += red[((((s2 * RGC) + rgc) * TILES + tl) * 2 + 1) * 32 + lane];
          }
        }
      }
      __syncthreads();  // red is reused by the next row groups
    }
    if (ks == 0 && rg < rg_end && j < n && (q & 1) == 0) {
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl) {
        const int tok = 2 * tl + (q >> 1);
        if (tok < M) {
          float* yr = P.y + (int64_t)tok * 2 * n;
          yr[j] = y_re[tl];
          yr[n + j] = y_im[tl];
        }
      }
    }
  }
}

}  // namespace f2i
