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

// trunc(v 2^(48-e)) for a finite v >= 0 below 2^(e+1), given the bits b of v
// and c = 102 + e, with 32-bit integer operations and one widening multiply:
// v = mant 2^(q-150) with q = max(exponent field, 1) and mant carrying the
// implicit bit when the exponent field is non-zero, so the value is
// mant 2^(q-c), a left shift of at most 25 or a truncating right shift.
__device__ __forceinline__ unsigned long long scaled_trunc_int(uint32_t b, int c) {
  const int q = max((int)(b >> 23), 1);
  const uint32_t mant = b - ((uint32_t)(q - 1) << 23);
  const int sh = q - c;
  const uint32_t hi = __funnelshift_rc(mant, 0u, (uint32_t)max(-sh, 0));  // mant >> (c - q), 0 past 31
  return (unsigned long long)hi * (unsigned long long)(1u << max(sh, 0));
}

// Column (inside its 64-column block) of weight c = 4 s + 2 h + e of the
// thread word q: 16 s + 8 h + 2 q + e, the columns whose signs share the sign
// word of lane (g, q) in the packed layout.
__host__ __device__ __forceinline__ int word_col(int c, int q) { return 16 * (c >> 2) + 8 * ((c >> 1) & 1) + 2 * q + (c & 1); }

// One CTA per (output row j, matrix X).  Thread t owns WPT words of the row;
// a word holds 16 weights (layout 2: columns 64 kb + word_col(c, q) of word
// w = 4 kb + q; layout 3: 16 consecutive columns) and, per stage, their
// sign bits and real-axis bits as two 16-bit masks.  The weights stay in
// registers through all T stages, so HBM sees one read of the row and one
// write of its codes and scales.  Per stage two block reductions (maxima;
// exact sums and counts), one barrier each; the scales are formed in every
// warp and passed on by shuffles.
constexpr int kQuantThreads = 512;  // words per thread: 1 for m <= 8192, 2 up to 16384
// One word per thread: at most 64 registers, so that 8 CTAs of 128 threads
// (m = 2048) share an SM and hide each other's row loads and barriers.

// Writes the zero 16-byte chunks of a padding row (j >= n) of layout 3: the
// last row tile's rows past n must read as zero codes.
__device__ __forceinline__ void l3_zero_row(uint8_t* codes, int64_t n, int64_t m, int T, int64_t j, int X) {
  const int64_t tau = j >> 5;
  const int r = (int)(j & 31);
  const int64_t W3 = l3_windows(m);
  for (int64_t idx = threadIdx.x; idx < W3 * 4 * T; idx += blockDim.x) {
    const int64_t win = idx / (4 * T);
    const int rem = (int)(idx - win * 4 * T);
    const int t = rem >> 2, jj = rem & 3;
    if (jj >= l3_slots(m, win)) continue;
    *reinterpret_cast<uint4*>(codes + l3_offset(n, m, T, win, tau, X * T + t) + jj * kL3SlotBytes + r * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

// FUSED = false: weights from complex U, W [n][m] (grid (rows, 2): row, matrix).
// FUSED = true:  weights computed from the real R [2n][2m] with the same
// float32 operations as the conversion kernel, so the codes and scales equal
// those of convert-then-quantize bit for bit (grid (2, rows): the two matrices
// of a row are neighbouring CTAs and share the R rows through L2).
// LAYOUT 2 or 3 selects the packed code layout written (the arithmetic is the
// same; only the column order of a thread's words and the final stores
// differ).  For layout 3 the grid has a row for every row of the last tile,
// and rows past n write zero chunks.
template <int WPT, bool FUSED, int LAYOUT>
__global__ void __launch_bounds__(kQuantThreads, WPT == 1 ? 2 : 1) quantize_words_kernel(
    const float2* __restrict__ U, const float2* __restrict__ W, const float* __restrict__ R, int64_t n, int64_t m,
    int T, uint8_t* __restrict__ codes, float* __restrict__ scales) {
  constexpr int E = 16 * WPT;  // weights per thread
  // one array per block-wide reduction of a stage: a reduction's array is
  // rewritten only after two other barriers, so one barrier per reduction
  __shared__ uint32_t s_mx[2][32];
  __shared__ unsigned long long s_sum[2][32];
  __shared__ uint32_t s_cnt[2][32];
  __shared__ float s_scale[2];

  const int tid = threadIdx.x;
  const int X = FUSED ? blockIdx.x : blockIdx.y;
  const int64_t j = FUSED ? blockIdx.y : blockIdx.x;
  if (LAYOUT == 3 && j >= n) {  // padding row of the last tile (block-uniform)
    l3_zero_row(codes, n, m, T, j, X);
    return;
  }
  const int64_t KB = col_blocks(m);
  const float2* src = FUSED ? nullptr : (X == 0 ? U : W) + j * m;
  const float* top = FUSED ? R + j * 2 * m : nullptr;        // R11 | R12 row
  const float* bot = FUSED ? R + (n + j) * 2 * m : nullptr;  // R21 | R22 row

  // column of weight e = 16 u + c of this thread (word u of WPT): layout 2
  // orders a word's columns as one sign word of the mma fragment, layout 3
  // takes 16 consecutive columns (two groups of 8)
  auto col_of = [&](int e) -> int64_t {
    const int64_t w = (int64_t)tid * WPT + (e >> 4);
    if (LAYOUT == 3) return w * 16 + (e & 15);
    return (w >> 2) * 64 + word_col(e & 15, (int)(w & 3));
  };
  float re[E], im[E];
  bool bad = false;
  uint32_t valid[WPT];
  // the weight of column k: from U or W, or formed from the four blocks of R
  // (default caching there: the row's other matrix, the neighbouring CTA,
  // reads the same R)
  auto weight = [&](int64_t k) -> float2 {
    if (FUSED) {
      const float r11 = __ldg(top + k), r12 = __ldg(top + m + k);
      const float r21 = __ldg(bot + k), r22 = __ldg(bot + m + k);
      return X == 0 ? make_float2(half_sum(r11, r22), half_diff(r21, r12))   // U
                    : make_float2(half_diff(r11, r22), half_sum(r12, r21));  // W
    }
    return __ldcs(src + k);
  };
  // A word whose 16 columns all lie inside the matrix is read two columns at
  // a time (its columns come in adjacent pairs k, k + 1 with k even): 16-byte
  // loads of U or W, 8-byte loads of the R blocks; m even keeps them aligned.
  // From R on layout 3 (16 consecutive columns, m a multiple of 4) it is
  // four columns per 16-byte load.  Other words are read one weight at a time.
  const bool pairs_aligned = (m & 1) == 0;
  const bool quads_aligned = FUSED && LAYOUT == 3 && (m & 3) == 0;
#pragma unroll
  for (int u = 0; u < WPT; ++u) {
    const int64_t w = (int64_t)tid * WPT + u;
    const bool whole = (w >> 2) < KB && (LAYOUT == 3 ? w * 16 + 16 <= m : (w >> 2) * 64 + 64 <= m);
    if (FUSED && LAYOUT == 3 && whole && quads_aligned) {
      valid[u] = 0xFFFFu;
#pragma unroll
      for (int c = 0; c < 16; c += 4) {
        const int e = 16 * u + c;
        const int64_t k = w * 16 + c;
        const float4 r11 = __ldg(reinterpret_cast<const float4*>(top + k));
        const float4 r12 = __ldg(reinterpret_cast<const float4*>(top + m + k));
        const float4 r21 = __ldg(reinterpret_cast<const float4*>(bot + k));
        const float4 r22 = __ldg(reinterpret_cast<const float4*>(bot + m + k));
        const float a11[4] = {r11.x, r11.y, r11.z, r11.w}, a12[4] = {r12.x, r12.y, r12.z, r12.w};
        const float a21[4] = {r21.x, r21.y, r21.z, r21.w}, a22[4] = {r22.x, r22.y, r22.z, r22.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          re[e + i] = X == 0 ? half_sum(a11[i], a22[i]) : half_diff(a11[i], a22[i]);
          im[e + i] = X == 0 ? half_diff(a21[i], a12[i]) : half_sum(a12[i], a21[i]);
          bad |= !(isfinite(re[e + i]) && isfinite(im[e + i]));
        }
      }
    } else if (whole && pairs_aligned) {
      valid[u] = 0xFFFFu;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        const int e = 16 * u + c;
        const int64_t k = col_of(e);
        float2 v0, v1;
        if (FUSED) {
          const float2 r11 = __ldg(reinterpret_cast<const float2*>(top + k));
          const float2 r12 = __ldg(reinterpret_cast<const float2*>(top + m + k));
          const float2 r21 = __ldg(reinterpret_cast<const float2*>(bot + k));
          const float2 r22 = __ldg(reinterpret_cast<const float2*>(bot + m + k));
          v0 = X == 0 ? make_float2(half_sum(r11.x, r22.x), half_diff(r21.x, r12.x))
                      : make_float2(half_diff(r11.x, r22.x), half_sum(r12.x, r21.x));
          v1 = X == 0 ? make_float2(half_sum(r11.y, r22.y), half_diff(r21.y, r12.y))
                      : make_float2(half_diff(r11.y, r22.y), half_sum(r12.y, r21.y));
        } else {
          const float4 v = __ldcs(reinterpret_cast<const float4*>(src + k));
          v0 = make_float2(v.x, v.y);
          v1 = make_float2(v.z, v.w);
        }
        bad |= !(isfinite(v0.x) && isfinite(v0.y) && isfinite(v1.x) && isfinite(v1.y));
        re[e] = v0.x;
        im[e] = v0.y;
        re[e + 1] = v1.x;
        im[e + 1] = v1.y;
      }
    } else {
      valid[u] = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int e = 16 * u + c;
        const int64_t k = col_of(e);
        float2 v = make_float2(0.0f, 0.0f);
        if ((w >> 2) < KB && k < m) {
          v = weight(k);
          valid[u] |= 1u << c;
        }
        bad |= !(isfinite(v.x) && isfinite(v.y));
        re[e] = v.x;
        im[e] = v.y;
      }
    }
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) f2i_raise(kErrNonFinite);
    return;  // whole CTA leaves together; the codes of this row stay unspecified
  }

  const int64_t pbytes = plane_bytes(n, m);
  const int g = (int)(j & 7), rho = (int)((j >> 3) & 1);
  const int64_t rt = j >> 4;

  const int lane = tid & 31, nwarps = (int)((blockDim.x + 31) >> 5);
  for (int t = 0; t < T; ++t) {
    // codes: real axis iff |Re| >= |Im|; negative iff the chosen component is
    // < 0 (-0 counts as +).  Columns outside the matrix hold (0, 0): real, not
    // negative, no weight in any maximum or sum; the masks drop them from the
    // counts and the imaginary flags.
    uint32_t sgn[WPT], realm[WPT];
    uint32_t mx0 = 0, mx1 = 0;
#pragma unroll
    for (int u = 0; u < WPT; ++u) sgn[u] = realm[u] = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e >> 4, c = e & 15;
      const float ar = fabsf(re[e]), ai = fabsf(im[e]);
      const bool real = ar >= ai;
      const bool neg = real ? (re[e] < 0.0f) : (im[e] < 0.0f);
      sgn[u] |= neg ? (1u << c) : 0u;
      realm[u] |= real ? (1u << c) : 0u;
      mx0 = max(mx0, real ? __float_as_uint(ar) : 0u);
      mx1 = max(mx1, real ? 0u : __float_as_uint(ai));
    }
    uint32_t cnt0 = 0, cnt1 = 0;
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      realm[u] &= valid[u];
      cnt0 += __popc(realm[u]);
      cnt1 += __popc(valid[u] & ~realm[u]);
    }
    // block maxima (one barrier)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx0 = max(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = max(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (lane == 0) {
      s_mx[0][tid >> 5] = mx0;
      s_mx[1][tid >> 5] = mx1;
    }
    __syncthreads();
    mx0 = s_mx[0][0];
    mx1 = s_mx[1][0];
    for (int w = 1; w < nwarps; ++w) {
      mx0 = max(mx0, s_mx[0][w]);
      mx1 = max(mx1, s_mx[1][w]);
    }
    const int e0 = mx0 ? float_exponent(mx0) : 0;
    const int e1 = mx1 ? float_exponent(mx1) : 0;

    // exact integer sums of trunc(|v| 2^(48-e)) (each term < 2^49).  Rows
    // with both maxima at or above 2^-79 take the fp32 path: t = |v| 2^(48-e)
    // is an exponent change (exact), a round-toward-zero add of 2^23
    // truncates it below 2^23 (above, t is an integer already), and
    // round-to-nearest adds of 1.5 2^55 and 1.5 2^39 split it exactly into
    // integer multiples of 2^32, 2^16 and 1; over at most 32 terms a thread's
    // sum of each part stays below 2^22 units, so the fp32 sums are exact.
    // Smaller rows take the integer-shift path (block-uniform branch).
    unsigned long long ls0 = 0, ls1 = 0;
    if (e0 >= -79 && e1 >= -79) {
      const float p0 = __int_as_float((48 - e0 + 127) << 23), p1 = __int_as_float((48 - e1 + 127) << 23);
      const float K1 = 54043195528445952.0f;  // 1.5 2^55
      const float K2 = 824633720832.0f;       // 1.5 2^39
      float a0 = 0.0f, b0 = 0.0f, z0 = 0.0f, a1 = 0.0f, b1 = 0.0f, z1 = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int u = e >> 4, c = e & 15;
        const bool isr = (realm[u] >> c) & 1u;
        const float t = __fmul_rn(isr ? fabsf(re[e]) : fabsf(im[e]), isr ? p0 : p1);
        const float tt = t < 8388608.0f ? __fsub_rn(__fadd_rz(t, 8388608.0f), 8388608.0f) : t;
        const float A = __fsub_rn(__fadd_rn(tt, K1), K1);
        const float r1 = __fsub_rn(tt, A);
        const float B = __fsub_rn(__fadd_rn(r1, K2), K2);
        const float C = __fsub_rn(r1, B);
        if (isr) {
          a0 = __fadd_rn(a0, A);
          b0 = __fadd_rn(b0, B);
          z0 = __fadd_rn(z0, C);
        } else {  // columns outside the matrix add 0
          a1 = __fadd_rn(a1, A);
          b1 = __fadd_rn(b1, B);
          z1 = __fadd_rn(z1, C);
        }
      }
      auto whole = [](float a, float b, float z) -> unsigned long long {
        const long long ia = __float2int_rz(__fmul_rn(a, 2.3283064365386963e-10f));  // a 2^-32
        const long long ib = __float2int_rz(__fmul_rn(b, 1.52587890625e-05f));       // b 2^-16
        return (unsigned long long)((ia << 32) + (ib << 16) + (long long)__float2int_rz(z));
      };
      ls0 = whole(a0, b0, z0);
      ls1 = whole(a1, b1, z1);
    } else {
      const int c0 = 102 + e0, c1 = 102 + e1;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int u = e >> 4, c = e & 15;
        const bool isr = (realm[u] >> c) & 1u;
        const unsigned long long val =
            scaled_trunc_int(__float_as_uint(isr ? fabsf(re[e]) : fabsf(im[e])), isr ? c0 : c1);
        if (isr) ls0 += val;
        else ls1 += val;  // columns outside the matrix add trunc(0) = 0
      }
    }
    // block sums and counts (one barrier)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, o);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, o);
      cnt0 += __shfl_xor_sync(0xffffffffu, cnt0, o);
      cnt1 += __shfl_xor_sync(0xffffffffu, cnt1, o);
    }
    if (lane == 0) {
      s_sum[0][tid >> 5] = ls0;
      s_sum[1][tid >> 5] = ls1;
      s_cnt[0][tid >> 5] = cnt0;
      s_cnt[1][tid >> 5] = cnt1;
    }
    __syncthreads();
    // threads 0 and 1 form the two scales (fp64: a handful of instructions on
    // a slow pipe, so one warp only) while the others store this stage's codes
    if (tid < 2) {
      unsigned long long sum = s_sum[tid][0];
      uint32_t cnt = s_cnt[tid][0];
      for (int w = 1; w < nwarps; ++w) {
        sum += s_sum[tid][w];
        cnt += s_cnt[tid][w];
      }
      const uint32_t mx = tid == 0 ? mx0 : mx1;
      const int ex = tid == 0 ? e0 : e1;
      float sc = 0.0f;
      if (cnt > 0 && mx != 0) sc = __double2float_rn(ldexp(__ll2double_rn((long long)sum), ex - 48) / (double)cnt);
      s_scale[tid] = sc;
      scales[((int64_t)(X * T + t) * 2 + tid) * n + j] = sc;
    }

    if (LAYOUT == 3) {
      // layout 3: the (4 / WPT) threads of a 64-column block assemble its
      // sign bytes and q bytes (q = sign XOR imaginary flag) into one 16-byte
      // chunk of the row, written once (no other row shares it)
      const int64_t w0 = (int64_t)tid * WPT;  // first word; all WPT words lie in block w0 >> 2
      const int64_t blk = w0 >> 2, win = blk >> 2;
      const int r = (int)(j & 31), nb = l3_slots(m, win < l3_windows(m) ? win : 0);
      unsigned long long S = 0, Q = 0;
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        const uint32_t s16 = sgn[u];
        const uint32_t q16 = s16 ^ (valid[u] & ~realm[u] & 0xFFFFu);
        const int g0 = (int)(((w0 + u) & 15) * 2);  // group of the word's first 8 columns in its window
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int pos = 8 * l3_byte_of(g0 + h, r);
          S |= (unsigned long long)((s16 >> (8 * h)) & 0xFFu) << pos;
          Q |= (unsigned long long)((q16 >> (8 * h)) & 0xFFu) << pos;
        }
      }
#pragma unroll
      for (int o = 1; o < 4 / WPT; o <<= 1) {
        S |= __shfl_xor_sync(0xffffffffu, S, o);
        Q |= __shfl_xor_sync(0xffffffffu, Q, o);
      }
      if ((tid & (4 / WPT - 1)) == 0 && win < l3_windows(m) && (blk & 3) < nb) {
        const int jj = l3_slot_of((int)((blk & 3) << 3), r, nb);
        *reinterpret_cast<uint4*>(codes + l3_offset(n, m, T, win, j >> 5, X * T + t) + jj * kL3SlotBytes + r * 16) =
            make_uint4((uint32_t)S, (uint32_t)(S >> 32), (uint32_t)Q, (uint32_t)(Q >> 32));
      }
    } else {
      // scatter the codes into the sign and flag words of the row's tile (the
      // plane was zeroed; the other row of each lane pair ORs its own bits)
      uint8_t* plane = codes + (int64_t)(X * T + t) * pbytes;
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        const int64_t w = (int64_t)tid * WPT + u;
        const int64_t kb = w >> 2;
        if (kb >= KB) continue;
        const int q = (int)(w & 3);
        uint32_t sw = 0, fw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int sidx = c >> 2, h = (c >> 1) & 1, e = c & 1;
          const uint32_t neg = (sgn[u] >> c) & 1u;
          const uint32_t imag = ((valid[u] & ~realm[u]) >> c) & 1u;  // padding columns stay zero
          sw |= neg << sign_bit(sidx, h, rho, e);
          fw[flag_lane(sidx, h)] |= imag << flag_bit(sidx, q, rho, e);
        }
        if (sw) atomicOr(reinterpret_cast<unsigned int*>(plane + pair_offset(rt, kb, 4 * g + q, KB)), sw);
#pragma unroll
        for (int ql = 0; ql < 4; ++ql)
          if (fw[ql]) atomicOr(reinterpret_cast<unsigned int*>(plane + pair_offset(rt, kb, 4 * g + ql, KB) + 4), fw[ql]);
      }
    }
    __syncthreads();
    const float s_re = s_scale[0], s_im = s_scale[1];

    // residual r <- r - (s_re b_re + i s_im b_im), one float32 rounding
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e >> 4, c = e & 15;
      const bool neg = (sgn[u] >> c) & 1u;
      const bool isr = (realm[u] >> c) & 1u;
      const float d = isr ? (neg ? -s_re : s_re) : (neg ? -s_im : s_im);
      const float upd = __fsub_rn(isr ? re[e] : im[e], d);
      re[e] = isr ? upd : re[e];
      im[e] = isr ? im[e] : upd;
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u)
      if (valid[u] != 0xFFFFu)  // columns outside the matrix stay (0, 0)
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (!((valid[u] >> c) & 1u)) re[16 * u + c] = im[16 * u + c] = 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Canonical view of the packed codes: out[X][t][j][k] in {0: +1, 1: -1,
// 2: +i, 3: -i}.  One thread per (plane, row tile, column block, lane).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) unpack_codes_kernel(const uint8_t* __restrict__ codes, int64_t n, int64_t m,
                                                           int T, uint8_t* __restrict__ out) {
  const int64_t RT = row_tiles(n), KB = col_blocks(m);
  const int64_t per_plane = RT * KB * 32;
  const int64_t total = 2 * (int64_t)T * per_plane;
  const int64_t pbytes = plane_bytes(n, m);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t plane = idx / per_plane;
    const int64_t rem = idx - plane * per_plane;
    const int64_t rt = rem / (KB * 32);
    const int64_t rem2 = rem - rt * KB * 32;
    const int64_t kb = rem2 >> 5;
    const int lane = (int)(rem2 & 31);
    const int g = lane >> 2, q = lane & 3;
    const uint8_t* pl = codes + plane * pbytes;
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(pl + pair_offset(rt, kb, lane, KB));
    uint32_t fw[4];
#pragma unroll
    for (int ql = 0; ql < 4; ++ql) fw[ql] = *reinterpret_cast<const uint32_t*>(pl + pair_offset(rt, kb, 4 * g + ql, KB) + 4);
#pragma unroll
    for (int rho = 0; rho < 2; ++rho) {
      const int64_t j = rt * 16 + 8 * rho + g;
      if (j >= n) continue;
      uint8_t* dst = out + (plane * n + j) * m;
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int64_t k = kb * 64 + 16 * s + 8 * h + 2 * q + e;
            if (k >= m) continue;
            const uint32_t sign = (sw >> sign_bit(s, h, rho, e)) & 1u;
            const uint32_t imag = (fw[flag_lane(s, h)] >> flag_bit(s, q, rho, e)) & 1u;
            dst[k] = (uint8_t)(2u * imag + sign);
          }
    }
  }
}

}  // namespace f2i
