// Widely-linear conversion and phase-aware recursive residual quantization.
#pragma once
#include <cstdint>
#include "layout.cuh"

namespace f2i {

// ---------------------------------------------------------------------------
// Conversion ("Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights
// {±1, ±i}", Step 1, Theorem 1):
//   Re U = (R11 + R22)/2   Im U = (R21 - R12)/2
//   Re W = (R11 - R22)/2   Im W = (R12 + R21)/2
// One float32 rounding for the sum; the halving is exact.  Each work item is
// one row j and four columns, read as four 16-byte loads (one per block of
// R) and written as two 16-byte stores to each of U and W.  Pure streaming,
// HBM-bound: 16 bytes read and 16 written per complex (U, W) entry pair.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float half_sum(float a, float b) { return __fmul_rn(__fadd_rn(a, b), 0.5f); }
__device__ __forceinline__ float half_diff(float a, float b) { return __fmul_rn(__fsub_rn(a, b), 0.5f); }

__global__ void __launch_bounds__(256) convert_vec4_kernel(const float* __restrict__ R, int64_t n, int64_t m,
                                                           float4* __restrict__ U, float4* __restrict__ W) {
  const int64_t m4 = m >> 2;
  const int64_t total = n * m4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t j = idx / m4;
    const int64_t k = (idx - j * m4) << 2;
    const float* top = R + j * 2 * m;
    const float* bot = R + (n + j) * 2 * m;
    const float4 r11 = __ldcs(reinterpret_cast<const float4*>(top + k));
    const float4 r12 = __ldcs(reinterpret_cast<const float4*>(top + m + k));
    const float4 r21 = __ldcs(reinterpret_cast<const float4*>(bot + k));
    const float4 r22 = __ldcs(reinterpret_cast<const float4*>(bot + m + k));
    const int64_t o = (j * m + k) >> 1;  // float4 index of (j, k) in the pair layout
    U[o] = make_float4(half_sum(r11.x, r22.x), half_diff(r21.x, r12.x), half_sum(r11.y, r22.y), half_diff(r21.y, r12.y));
    U[o + 1] = make_float4(half_sum(r11.z, r22.z), half_diff(r21.z, r12.z), half_sum(r11.w, r22.w), half_diff(r21.w, r12.w));
    W[o] = make_float4(half_diff(r11.x, r22.x), half_sum(r12.x, r21.x), half_diff(r11.y, r22.y), half_sum(r12.y, r21.y));
    W[o + 1] = make_float4(half_diff(r11.z, r22.z), half_sum(r12.z, r21.z), half_diff(r11.w, r22.w), half_sum(r12.w, r21.w));
  }
}

__global__ void __launch_bounds__(256) convert_scalar_kernel(const float* __restrict__ R, int64_t n, int64_t m,
                                                             float2* __restrict__ U, float2* __restrict__ W) {
  const int64_t total = n * m;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t j = idx / m, k = idx - (idx / m) * m;
    const float r11 = R[j * 2 * m + k], r12 = R[j * 2 * m + m + k];
    const float r21 = R[(n + j) * 2 * m + k], r22 = R[(n + j) * 2 * m + m + k];
    U[idx] = make_float2(half_sum(r11, r22), half_diff(r21, r12));
    W[idx] = make_float2(half_diff(r11, r22), half_sum(r12, r21));
  }
}

// ---------------------------------------------------------------------------
// Quantization ("Fairy2i: Ultra-Low-Bit ...", Step 2 and Step 3).
// One CTA per (matrix, output row).  The row's residual lives in shared
// memory for all T stages; HBM sees one read of the row and one write of its
// codes and scales.
//
// Code of r = a + ib: argmax over (+1, -1, +i, -i) of Re(r conj(s)) =
// (a, -a, b, -b), first maximum.  Equivalently: real axis iff |a| >= |b|;
// negative iff the chosen component is < 0 (so -0 counts as +).
//
// Scale of an axis (mean |v| over the row's weights coded on it), exact and
// independent of summation order:
//   e   = exponent of the largest |v| (largest in [2^e, 2^(e+1)))
//   sum = sum of trunc(|v| 2^(48-e)) in int64, each term < 2^49
//   s   = float(double(sum) 2^(e-48) / count)       (0 if count or max is 0)
// ---------------------------------------------------------------------------

// Exponent e with v in [2^e, 2^(e+1)) for a positive float given by its bits.
__device__ __forceinline__ int float_exponent(uint32_t bits) {
  const uint32_t ef = bits >> 23;
  if (ef != 0) return (int)ef - 127;
  const uint32_t mant = bits & 0x7FFFFFu;  // subnormal: mant * 2^-149
  return (31 - __clz((int)mant)) - 149;
}

// trunc(v * 2^(48-e)) for 0 <= v < 2^(e+1), exactly, by integer shifts.
__device__ __forceinline__ long long scaled_trunc(uint32_t bits, int e) {
  const uint32_t ef = bits >> 23;
  uint64_t mant = bits & 0x7FFFFFu;
  int ev;  // v = mant * 2^ev
  if (ef == 0) {
    ev = -149;
  } else {
    mant |= 0x800000u;
    ev = (int)ef - 150;
  }
  const int sh = ev + 48 - e;
  if (sh >= 0) return (long long)(mant << sh);  // < 2^49 by the bound on v
  if (sh <= -64) return 0;
  return (long long)(mant >> (-sh));
}

template <typename Tv>
__device__ __forceinline__ Tv warp_sum(Tv v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int kQuantThreads = 256;

// Dynamic shared memory: m float2 residual entries, then m code bytes.
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(
    const float2* __restrict__ U, const float2* __restrict__ W, int64_t n, int64_t m, int T,
    uint8_t* __restrict__ codes, float* __restrict__ scales) {
  extern __shared__ __align__(16) unsigned char qsmem[];
  float2* row = reinterpret_cast<float2*>(qsmem);
  uint8_t* cbits = qsmem + m * sizeof(float2);
  constexpr int NW = kQuantThreads / 32;
  __shared__ uint32_t s_max[2][NW];
  __shared__ int s_cnt[2][NW];
  __shared__ long long s_sum[2][NW];
  __shared__ float s_scale[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int X = blockIdx.y;
  const int64_t j = blockIdx.x;
  const float2* src = (X == 0 ? U : W) + j * m;

  bool bad = false;
  for (int64_t k = tid; k < m; k += kQuantThreads) {
    const float2 v = src[k];
    bad |= !(isfinite(v.x) && isfinite(v.y));
    row[k] = v;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) f2i_raise(kErrNonFinite);
    return;  // whole CTA leaves together; the codes of this row stay unspecified
  }

  const int64_t KB = col_blocks(m);
  const int64_t pbytes = plane_bytes(n, m);
  const int64_t rg = j >> 3;
  const int g = (int)(j & 7);

  for (int t = 0; t < T; ++t) {
    // codes, per-axis maxima and counts
    uint32_t lmax0 = 0, lmax1 = 0;
    int lcnt0 = 0, lcnt1 = 0;
    for (int64_t k = tid; k < m; k += kQuantThreads) {
      const float2 v = row[k];
      const float ar = fabsf(v.x), ai = fabsf(v.y);
      const bool real = ar >= ai;
      const bool neg = real ? (v.x < 0.0f) : (v.y < 0.0f);
      cbits[k] = (uint8_t)(((neg ? 1 : 0) << 1) | (real ? 1 : 0));
      if (real) { lmax0 = max(lmax0, __float_as_uint(ar)); ++lcnt0; }
      else { lmax1 = max(lmax1, __float_as_uint(ai)); ++lcnt1; }
    }
    lmax0 = warp_max(lmax0); lmax1 = warp_max(lmax1);
    lcnt0 = warp_sum(lcnt0); lcnt1 = warp_sum(lcnt1);
    if (lane == 0) { s_max[0][warp] = lmax0; s_max[1][warp] = lmax1; s_cnt[0][warp] = lcnt0; s_cnt[1][warp] = lcnt1; }
    __syncthreads();
    uint32_t mx[2] = {0, 0};
    int cnt[2] = {0, 0};
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      mx[0] = max(mx[0], s_max[0][w]); mx[1] = max(mx[1], s_max[1][w]);
      cnt[0] += s_cnt[0][w]; cnt[1] += s_cnt[1][w];
    }
    const int e0 = mx[0] ? float_exponent(mx[0]) : 0;
    const int e1 = mx[1] ? float_exponent(mx[1]) : 0;

    // exact integer sums of |v| 2^(48-e)
    long long ls0 = 0, ls1 = 0;
    for (int64_t k = tid; k < m; k += kQuantThreads) {
      const float2 v = row[k];
      if (cbits[k] & 1u) ls0 += scaled_trunc(__float_as_uint(fabsf(v.x)), e0);
      else ls1 += scaled_trunc(__float_as_uint(fabsf(v.y)), e1);
    }
    ls0 = warp_sum(ls0); ls1 = warp_sum(ls1);
    if (lane == 0) { s_sum[0][warp] = ls0; s_sum[1][warp] = ls1; }
    __syncthreads();
    if (tid < 2) {
      const int a = tid;
      long long sum = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) sum += s_sum[a][w];
      float s = 0.0f;
      if (cnt[a] > 0 && mx[a] != 0) {
        const int e = a == 0 ? e0 : e1;
        const double mean = ldexp(__ll2double_rn(sum), e - 48) / (double)cnt[a];
        s = __double2float_rn(mean);
      }
      s_scale[a] = s;
      scales[((int64_t)(X * T + t) * 2 + a) * n + j] = s;
    }
    __syncthreads();

    // residual update r <- r - (s_re b_re + i s_im b_im), one float32 rounding
    const float s_re = s_scale[0], s_im = s_scale[1];
    for (int64_t k = tid; k < m; k += kQuantThreads) {
      const uint32_t c = cbits[k];
      float2 v = row[k];
      if (c & 1u) v.x = __fsub_rn(v.x, (c & 2u) ? -s_re : s_re);
      else v.y = __fsub_rn(v.y, (c & 2u) ? -s_im : s_im);
      row[k] = v;
    }

    // pack: word (kb, q) of row g holds the 16 columns 64 kb + code_col(c, q)
    uint8_t* plane = codes + (int64_t)(X * T + t) * pbytes;
    for (int64_t w = tid; w < KB * 4; w += kQuantThreads) {
      const int64_t kb = w >> 2;
      const int q = (int)(w & 3);
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int64_t k = kb * 64 + code_col(c, q);
        if (k < m) word |= (uint32_t)cbits[k] << code_shift(c);
      }
      *reinterpret_cast<uint32_t*>(plane + word_offset(rg, kb, 4 * g + q, KB)) = word;
    }
    __syncthreads();  // cbits and row are rewritten by the next stage
  }
}

// ---------------------------------------------------------------------------
// Canonical view of the packed codes: out[X][t][j][k] in {0: +1, 1: -1,
// 2: +i, 3: -i}.  One thread per packed word.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) unpack_codes_kernel(const uint8_t* __restrict__ codes, int64_t n, int64_t m,
                                                           int T, uint8_t* __restrict__ out) {
  const int64_t RG = row_groups(n), KB = col_blocks(m);
  const int64_t wpp = RG * KB * 32;
  const int64_t total = 2 * (int64_t)T * wpp;
  const int64_t pbytes = plane_bytes(n, m);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t plane = idx / wpp;
    const int64_t rem = idx - plane * wpp;
    const int64_t rg = rem / (KB * 32);
    const int64_t rem2 = rem - rg * KB * 32;
    const int64_t kb = rem2 >> 5;
    const int lane = (int)(rem2 & 31);
    const int64_t j = rg * 8 + (lane >> 2);
    if (j >= n) continue;
    const int q = lane & 3;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + plane * pbytes + word_offset(rg, kb, lane, KB));
    uint8_t* dst = out + (plane * n + j) * m;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int64_t k = kb * 64 + code_col(c, q);
      if (k < m) dst[k] = (uint8_t)canonical_from_bits((w >> code_shift(c)) & 3u);
    }
  }
}

}  // namespace f2i
