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

// Column (inside its 64-column block) of weight c = 4 s + 2 h + e of the
// thread word q: 16 s + 8 h + 2 q + e, the columns whose signs share the sign
// word of lane (g, q) in the packed layout.
__host__ __device__ __forceinline__ int word_col(int c, int q) { return 16 * (c >> 2) + 8 * ((c >> 1) & 1) + 2 * q + (c & 1); }

// One CTA per (output row j, matrix X).  Thread t owns WPT words of the row;
// word w = 4 kb + q holds the 16 weights at columns 64 kb + word_col(c, q),
// each code as two bits (sign, real-axis flag) at bits (2c + 1, 2c).
// The weights stay in registers through all T stages, so HBM sees one read of
// the row and one write of its codes and scales, and each word is assembled as
// its codes are decided.  Row-wide maxima, counts and exact sums are block
// reductions (warp shuffles, then one value per warp in shared memory).
constexpr int kQuantThreads = 512;  // words per thread: 1 for m <= 8192, 2 up to 16384

template <typename Tv, typename Op>
__device__ __forceinline__ void block_reduce2(Tv& a, Tv& b, Tv* sa, Tv* sb, Op op) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = op(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = op(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if (lane == 0) {
    sa[warp] = a;
    sb[warp] = b;
  }
  __syncthreads();
  a = sa[0];
  b = sb[0];
  for (int w = 1; w < nw; ++w) {
    a = op(a, sa[w]);
    b = op(b, sb[w]);
  }
  __syncthreads();  // sa / sb are reused by the next reduction
}

// Sums of two 64-bit and two 32-bit values over the block in one round (the
// counts travel with the exact sums; both are needed only for the scale).
__device__ __forceinline__ void block_sum_ll2_u2(long long& a, long long& b, uint32_t& c, uint32_t& d,
                                                 long long* sa, long long* sb, uint32_t* sc, uint32_t* sd) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
    d += __shfl_xor_sync(0xffffffffu, d, o);
  }
  if (lane == 0) {
    sa[warp] = a;
    sb[warp] = b;
    sc[warp] = c;
    sd[warp] = d;
  }
  __syncthreads();
  a = sa[0];
  b = sb[0];
  c = sc[0];
  d = sd[0];
  for (int w = 1; w < nw; ++w) {
    a += sa[w];
    b += sb[w];
    c += sc[w];
    d += sd[w];
  }
  __syncthreads();  // the buffers are reused by the next reduction
}

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
__global__ void __launch_bounds__(kQuantThreads) quantize_words_kernel(
    const float2* __restrict__ U, const float2* __restrict__ W, const float* __restrict__ R, int64_t n, int64_t m,
    int T, uint8_t* __restrict__ codes, float* __restrict__ scales) {
  constexpr int E = 16 * WPT;  // weights per thread
  __shared__ uint32_t s_u[2][32];
  __shared__ long long s_l[2][32];
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
#pragma unroll
  for (int u = 0; u < WPT; ++u) valid[u] = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int64_t w = (int64_t)tid * WPT + (e >> 4);
    const int64_t k = col_of(e);
    float2 v = make_float2(0.0f, 0.0f);
    if ((w >> 2) < KB && k < m) {
      if (FUSED) {
        // default caching: the row's other matrix (the neighbouring CTA) reads the same R
        const float r11 = __ldg(top + k), r12 = __ldg(top + m + k);
        const float r21 = __ldg(bot + k), r22 = __ldg(bot + m + k);
        v = X == 0 ? make_float2(half_sum(r11, r22), half_diff(r21, r12))   // U
                   : make_float2(half_diff(r11, r22), half_sum(r12, r21));  // W
      } else {
        v = __ldcs(src + k);
      }
      valid[e >> 4] |= 1u << (e & 15);
    }
    bad |= !(isfinite(v.x) && isfinite(v.y));
    re[e] = v.x;
    im[e] = v.y;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) f2i_raise(kErrNonFinite);
    return;  // whole CTA leaves together; the codes of this row stay unspecified
  }

  const int64_t pbytes = plane_bytes(n, m);
  const int g = (int)(j & 7), rho = (int)((j >> 3) & 1);
  const int64_t rt = j >> 4;

  for (int t = 0; t < T; ++t) {
    // codes: real axis iff |Re| >= |Im|; negative iff the chosen component is < 0
    // (branch-free; columns outside the matrix keep zero code bits and count nowhere)
    uint32_t word[WPT], realm[WPT];
    uint32_t mx0 = 0, mx1 = 0, cnt0 = 0, cnt1 = 0;
#pragma unroll
    for (int u = 0; u < WPT; ++u) word[u] = realm[u] = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e >> 4, c = e & 15;
      const bool in = (valid[u] >> c) & 1u;
      const float ar = fabsf(re[e]), ai = fabsf(im[e]);
      const bool real = ar >= ai;
      const bool neg = real ? (re[e] < 0.0f) : (im[e] < 0.0f);
      const bool isr = in && real, isi = in && !real;
      word[u] |= (in ? (((neg ? 1u : 0u) << 1) | (real ? 1u : 0u)) : 0u) << (2 * c);
      realm[u] |= (isr ? 1u : 0u) << c;
      mx0 = max(mx0, isr ? __float_as_uint(ar) : 0u);
      mx1 = max(mx1, isi ? __float_as_uint(ai) : 0u);
      cnt0 += isr ? 1u : 0u;
      cnt1 += isi ? 1u : 0u;
    }
    block_reduce2(mx0, mx1, s_u[0], s_u[1], [](uint32_t x, uint32_t y) { return max(x, y); });
    const int e0 = mx0 ? float_exponent(mx0) : 0;
    const int e1 = mx1 ? float_exponent(mx1) : 0;

    // exact integer sums of trunc(|v| 2^(48-e)).  With 48 - e <= 127 the
    // power of two is a float, |v| 2^(48-e) < 2^49 is exact (an exponent
    // change) and the truncating conversion to u64 is exact; rows whose
    // maximum is below 2^-79 take the integer-shift path (block-uniform).
    long long ls0 = 0, ls1 = 0;
    if (e0 >= -79 && e1 >= -79) {
      const float sc0 = __int_as_float((48 - e0 + 127) << 23), sc1 = __int_as_float((48 - e1 + 127) << 23);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int u = e >> 4, c = e & 15;
        const bool isr = (realm[u] >> c) & 1u, in = (valid[u] >> c) & 1u;
        const float v = isr ? fabsf(re[e]) : fabsf(im[e]);
        const long long val = (long long)__float2ull_rz(__fmul_rn(v, isr ? sc0 : sc1));
        ls0 += isr ? val : 0ll;
        ls1 += (in && !isr) ? val : 0ll;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int u = e >> 4, c = e & 15;
        if (!((valid[u] >> c) & 1u)) continue;
        if ((realm[u] >> c) & 1u) ls0 += scaled_trunc(__float_as_uint(fabsf(re[e])), e0);
        else ls1 += scaled_trunc(__float_as_uint(fabsf(im[e])), e1);
      }
    }
    block_sum_ll2_u2(ls0, ls1, cnt0, cnt1, s_l[0], s_l[1], s_u[0], s_u[1]);
    if (tid < 2) {
      const long long sum = tid == 0 ? ls0 : ls1;
      const uint32_t cnt = tid == 0 ? cnt0 : cnt1;
      const uint32_t mx = tid == 0 ? mx0 : mx1;
      const int e = tid == 0 ? e0 : e1;
      float sc = 0.0f;
      if (cnt > 0 && mx != 0) sc = __double2float_rn(ldexp(__ll2double_rn(sum), e - 48) / (double)cnt);
      s_scale[tid] = sc;
      scales[((int64_t)(X * T + t) * 2 + tid) * n + j] = sc;
    }
    __syncthreads();
    const float s_re = s_scale[0], s_im = s_scale[1];
    __syncthreads();  // s_scale is rewritten by the next stage

    // residual r <- r - (s_re b_re + i s_im b_im), one float32 rounding
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int u = e >> 4, c = e & 15;
      const bool neg = (word[u] >> (2 * c + 1)) & 1u;
      const bool isr = (realm[u] >> c) & 1u;
      const float d = isr ? (neg ? -s_re : s_re) : (neg ? -s_im : s_im);
      const float upd = __fsub_rn(isr ? re[e] : im[e], d);
      re[e] = isr ? upd : re[e];
      im[e] = isr ? im[e] : upd;
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
        uint32_t s16 = 0;
#pragma unroll
        for (int c = 0; c < 16; ++c) s16 |= ((word[u] >> (2 * c + 1)) & 1u) << c;
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
      continue;
    }
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
        const uint32_t v = (word[u] >> (2 * c)) & 3u;  // (sign, real-axis flag)
        const uint32_t imag = (valid[u] >> c) & 1u & ~v;       // padding columns stay zero
        sw |= (v >> 1) << sign_bit(sidx, h, rho, e);
        fw[flag_lane(sidx, h)] |= imag << flag_bit(sidx, q, rho, e);
      }
      if (sw) atomicOr(reinterpret_cast<unsigned int*>(plane + pair_offset(rt, kb, 4 * g + q, KB)), sw);
#pragma unroll
      for (int ql = 0; ql < 4; ++ql)
        if (fw[ql]) atomicOr(reinterpret_cast<unsigned int*>(plane + pair_offset(rt, kb, 4 * g + ql, KB) + 4), fw[ql]);
    }
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
