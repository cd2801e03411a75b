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
  int32_t cta_begin;      // first CTA of this problem in the launch
  int32_t tiles_per_cta;  // row tiles per CTA (decode partition)
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

// Row stride (bfloat16 elements) of staged activations: 16 bytes of padding.
__host__ __device__ __forceinline__ int64_t x_stride(int64_t m) { return col_blocks(m) * 64 + 8; }

// Stages x ([M][2m] bfloat16) as rows (token, part) of x_stride(m) elements,
// zero past m, followed by `extra_rows` rows of zeros.
__device__ __forceinline__ void stage_x(uint16_t* xs, const uint16_t* x, int M, int64_t m, int extra_rows,
                                        int nthreads) {
  const int64_t xstr = x_stride(m);
  const int64_t rows = (int64_t)M * 2;
  const bool vec = (m & 7) == 0 && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  if (vec) {
    const int64_t per_row = xstr >> 3;
    for (int64_t idx = threadIdx.x; idx < (rows + extra_rows) * per_row; idx += nthreads) {
      const int64_t row = idx / per_row, k8 = (idx - row * per_row) << 3;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < rows && k8 < m) v = *reinterpret_cast<const uint4*>(x + (row >> 1) * 2 * m + (row & 1) * m + k8);
      *reinterpret_cast<uint4*>(xs + row * xstr + k8) = v;
    }
  } else {
    for (int64_t idx = threadIdx.x; idx < (rows + extra_rows) * xstr; idx += nthreads) {
      const int64_t row = idx / xstr, k = idx - row * xstr;
      xs[idx] = (row < rows && k < m) ? x[(row >> 1) * 2 * m + (row & 1) * m + k] : (uint16_t)0;
    }
  }
}

// ---------------------------------------------------------------------------
// ALGO_ADDSUB: CUDA cores, adds and subtracts only (the pages' inference
// arithmetic taken literally).  One warp per row tile of 16 rows; lane (g, q)
// owns rows g and g + 8 and, in every 64-column block, the 16 columns of its
// sign word; the axis flags come from the quad's flag words (shuffles).  x is
// staged in shared memory as packed bfloat16 (a, b) pairs; each code flips
// the sign bits of a and b and adds them to its axis accumulators.  A quad
// shuffle sums the four lanes of a row.  Issue-bound; a reference path.
// ---------------------------------------------------------------------------
constexpr int kAddSubWarps = 8;
constexpr int kAddSubTok = 2;

__global__ void __launch_bounds__(kAddSubWarps * 32) linear_addsub_kernel(const __grid_constant__ LinearGroup G) {
  extern __shared__ __align__(16) uint32_t xs[];  // [kAddSubTok][m_pad] (a | b << 16)
  const LinearProblem& P = G.p[find_problem(G)];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = P.n, m = P.m;
  const int T = P.T, M = G.M;
  const int64_t KB = col_blocks(m), m_pad = KB * 64, RT = row_tiles(n);
  const int64_t rt = (int64_t)(blockIdx.x - P.cta_begin) * kAddSubWarps + warp;
  const int g = lane >> 2, q = lane & 3;
  const int64_t pbytes = plane_bytes(n, m);

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
    if (rt >= RT) continue;

    float y_re[2][kAddSubTok], y_im[2][kAddSubTok];
#pragma unroll
    for (int rho = 0; rho < 2; ++rho)
#pragma unroll
      for (int tk = 0; tk < kAddSubTok; ++tk) y_re[rho][tk] = y_im[rho][tk] = 0.0f;

    for (int plane = 0; plane < 2 * T; ++plane) {
      const int X = plane / T, t = plane - X * T;
      const uint8_t* pl = P.codes + (int64_t)plane * pbytes;
      float acc[2][kAddSubTok][4];  // (ra, rb, ia, ib)
#pragma unroll
      for (int rho = 0; rho < 2; ++rho)
#pragma unroll
        for (int tk = 0; tk < kAddSubTok; ++tk) acc[rho][tk][0] = acc[rho][tk][1] = acc[rho][tk][2] = acc[rho][tk][3] = 0.0f;
      for (int64_t kb = 0; kb < KB; ++kb) {
        const uint2 own = *reinterpret_cast<const uint2*>(pl + pair_offset(rt, kb, lane, KB));
        uint32_t fq[4];
#pragma unroll
        for (int ql = 0; ql < 4; ++ql) fq[ql] = __shfl_sync(0xffffffffu, own.y, (lane & ~3) | ql);
#pragma unroll
        for (int rho = 0; rho < 2; ++rho)
#pragma unroll
          for (int s = 0; s < 4; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const uint32_t sgn = ((own.x >> sign_bit(s, h, rho, e)) & 1u) << 31;
                const bool imag = (fq[flag_lane(s, h)] >> flag_bit(s, q, rho, e)) & 1u;
                const int64_t k = kb * 64 + 16 * s + 8 * h + 2 * q + e;
#pragma unroll
                for (int tk = 0; tk < kAddSubTok; ++tk) {
                  const uint32_t xv = xs[tk * m_pad + k];
                  const float a = __uint_as_float((xv << 16) ^ sgn);
                  const float bb = __uint_as_float((xv & 0xFFFF0000u) ^ sgn);
                  acc[rho][tk][0] += imag ? 0.0f : a;
                  acc[rho][tk][1] += imag ? 0.0f : bb;
                  acc[rho][tk][2] += imag ? a : 0.0f;
                  acc[rho][tk][3] += imag ? bb : 0.0f;
                }
              }
      }
#pragma unroll
      for (int rho = 0; rho < 2; ++rho) {
        const int64_t j = rt * 16 + 8 * rho + g;
        float s_re = 0.0f, s_im = 0.0f;
        if (j < n) {
          s_re = P.scales[((int64_t)(X * T + t) * 2 + 0) * n + j];
          s_im = P.scales[((int64_t)(X * T + t) * 2 + 1) * n + j];
        }
#pragma unroll
        for (int tk = 0; tk < kAddSubTok; ++tk) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[rho][tk][u] += __shfl_xor_sync(0xffffffffu, acc[rho][tk][u], 1);
            acc[rho][tk][u] += __shfl_xor_sync(0xffffffffu, acc[rho][tk][u], 2);
          }
          plane_epilogue(X, s_re, s_im, acc[rho][tk][0], acc[rho][tk][1], acc[rho][tk][2], acc[rho][tk][3],
                         y_re[rho][tk], y_im[rho][tk]);
        }
      }
    }
#pragma unroll
    for (int rho = 0; rho < 2; ++rho) {
      const int64_t j = rt * 16 + 8 * rho + g;
      if (q == 0 && j < n) {
        for (int tk = 0; tk < ntok; ++tk) {
          float* yr = P.y + (int64_t)(tok0 + tk) * 2 * n;
          yr[j] = y_re[rho][tk];
          yr[n + j] = y_im[rho][tk];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// ALGO_MMA: 2:4-sparse tensor-core decode, mma.sp m16n8k32 bf16.
//   K is the interleave (column k, axis): slot 2k = real axis, 2k + 1 =
//   imaginary axis.  Each code is nonzero in exactly one of its two slots, so
//   every group of four slots (two codes) holds two nonzeros: the compressed
//   A values are the two codes' signs as bfloat16 +-2 (one LOP3 per register
//   from the sign word, shifted into place by a multiply), and the metadata
//   (slot indices) are the axis flags, one LOP3 per four steps from the flag
//   word.  A rows: output rows g and g + 8 of a 16-row tile.
//   B (32 x 8): column 4 t + c for token t of the pair: c = 0 -> (a_k, 0),
//   1 -> (0, a_k), 2 -> (b_k, 0), 3 -> (0, b_k) over slots (2k, 2k + 1), so D
//   columns are <re-row, a>, <im-row, a>, <re-row, b>, <im-row, b>.
//   Products of +-2 and a bfloat16 are exact; only the fp32 accumulation
//   rounds.  Steps 0-1 take metadata from quad lanes 0-1 (selector 0), steps
//   2-3 from lanes 2-3 (selector 1), which is how the flag words are laid out.
// Partition: the host gives each problem of the launch a number of CTAs in
// proportion to its bytes and each CTA a run of `tiles_per_cta` row tiles.
// A CTA has WARPS = 8 warps (two CTAs per SM) or 16 (one CTA per SM: twice the
// row tiles per CTA, so the whole-tile granularity of the partition costs less
// imbalance between SMs).  The warps of a CTA split its (row tile, two-block
// chunk) items evenly, stream the 2T code planes through a per-warp cp.async
// double buffer, fold each row tile's share into per-warp partial outputs in
// shared memory, and one fixed-order sum at the end writes y (bitwise
// reproducible for a given launch shape).
// ---------------------------------------------------------------------------
constexpr int kMmaWarps = 8;       // two CTAs per SM
constexpr int kMmaWarpsWide = 16;  // one CTA per SM
constexpr int kMaxTilesPerCta = 16;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// (x & m) | 0x40004000 in one LOP3 (m held in a register): the two signs at
// bits 15 and 31 become bfloat16 +-2.
__device__ __forceinline__ uint32_t sign_operand(uint32_t x, uint32_t m) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, 0x40004000, 0xEA;" : "=r"(r) : "r"(x), "r"(m));
  return r;
}
template <int SEL>
__device__ __forceinline__ void mma_sp_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[4],
                                            uint32_t e) {
  asm volatile(
      "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, %13;"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(e), "n"(SEL));
}

// Shared memory: per-warp rings [WARPS][2][NPL][32 lanes] x 16 bytes, then
// x staged as [2M + 1][x_stride(m)] bfloat16 (last row zero), then partials
// [tiles][WARPS][TILES][32 lanes][2 rows] float2.
template <int NPL, int TILES, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, (WARPS == kMmaWarps && NPL * TILES <= 8) ? 2 : 1)
    linear_mma_kernel(const __grid_constant__ LinearGroup G) {
  extern __shared__ __align__(16) unsigned char msm[];
  const LinearProblem& P = G.p[find_problem(G)];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int64_t n = P.n, m = P.m;
  const int T = P.T, M = G.M;
  const int64_t KB = col_blocks(m), RT = row_tiles(n);
  const int64_t pbytes = plane_bytes(n, m);
  const int nch = (int)((KB + 1) >> 1);  // two-block chunks per row tile
  const int64_t rt_begin = (int64_t)(blockIdx.x - P.cta_begin) * P.tiles_per_cta;
  const int64_t rt_end = min(RT, rt_begin + P.tiles_per_cta);
  const int niter = (int)(rt_end - rt_begin);
  const int64_t xstr = x_stride(m);
  constexpr uint32_t kSlot = NPL * 512u;

  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(msm);
  const uint32_t ring = sbase + (uint32_t)warp * 2u * kSlot;
  uint16_t* xs = reinterpret_cast<uint16_t*>(msm + WARPS * 2 * kSlot);
  float2* red = reinterpret_cast<float2*>(msm + WARPS * 2 * kSlot +
                                          (((size_t)(2 * M + 1) * xstr * sizeof(uint16_t) + 15) & ~(size_t)15));

  const int items = niter * nch;
  const int i0 = (int)((int64_t)items * warp / WARPS), i1 = (int)((int64_t)items * (warp + 1) / WARPS);
  const int fullc = (int)(KB >> 1);
  const uint32_t tile_row = (uint32_t)KB * kTileBytes;
  const uint8_t* plane0 = P.codes + rt_begin * (int64_t)tile_row;

  int ir = i0 / nch, ic = i0 - (i0 / nch) * nch;  // next item to load
  // byte offset of this lane's 16 bytes of the next item, inside plane 0
  uint32_t src_off = (uint32_t)ir * tile_row + (uint32_t)ic * 512u + (uint32_t)lane * 16u;
  const uint32_t pstride = (uint32_t)pbytes;  // a plane is below 4 GB
  auto issue = [&](int slot) {
    if (ic < fullc) {
      const uint32_t dst = ring + (uint32_t)slot * kSlot + (uint32_t)lane * 16u;
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) cp_async16(dst + pl * 512u, plane0 + (src_off + (uint32_t)pl * pstride));
    }
    cp_commit();
    src_off += 512u;
    if (++ic == nch) {
      ic = 0;
      ++ir;
      src_off = (uint32_t)ir * tile_row + (uint32_t)lane * 16u;
    }
  };
  if (i0 < i1) issue(0);

  // Staged activations: with 16-byte rows every piece is an asynchronous copy
  // (zero-filled past m and in the extra row), so all of a thread's pieces are
  // in flight at once instead of one load-store round trip each.
  if ((m & 7) == 0 && (reinterpret_cast<uintptr_t>(P.x) & 15) == 0) {
    const int64_t rows = (int64_t)M * 2, per_row = xstr >> 3;
    for (int64_t idx = tid; idx < (rows + 1) * per_row; idx += WARPS * 32) {
      const int64_t row = idx / per_row, k8 = (idx - row * per_row) << 3;
      const bool in = row < rows && k8 < m;
      const uint16_t* src = in ? P.x + (row >> 1) * 2 * m + (row & 1) * m + k8 : P.x;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(xs + row * xstr + k8);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16 : 0) : "memory");
    }
    cp_commit();
  } else {
    stage_x(xs, P.x, M, m, 1, WARPS * 32);
  }
  for (int z = tid; z < niter * WARPS * TILES * 64; z += WARPS * 32) red[z] = make_float2(0.0f, 0.0f);
  cp_wait<0>();  // the staged activations (and the first code item)
  __syncthreads();

  // B of this lane: token 2 tl + (g >> 2), part (g >> 1) & 1, upper half iff g odd
  const uint16_t* xp[TILES];
#pragma unroll
  for (int tl = 0; tl < TILES; ++tl) {
    const int tok = 2 * tl + (g >> 2);
    const int64_t row = tok < M ? (int64_t)tok * 2 + ((g >> 1) & 1) : (int64_t)2 * M;
    xp[tl] = xs + row * xstr + q;
  }
  // Run-time constants (M < 2^30): the multiplies below stay multiplies on the
  // FMA pipe instead of becoming shifts on the busier integer pipe.
  const uint32_t bmul = (g & 1) ? 65536u : 1u;
  const uint32_t smask = 0x80008000u + (uint32_t)(M >> 30);
  const uint32_t two = 2u + (uint32_t)(M >> 30);
  const uint32_t half_hi = 0x80000000u + (uint32_t)(M >> 30);  // umulhi(v, 2^31) = v >> 1

  float acc[NPL][TILES][4];
#pragma unroll
  for (int pl = 0; pl < NPL; ++pl)
#pragma unroll
    for (int tl = 0; tl < TILES; ++tl) acc[pl][tl][0] = acc[pl][tl][1] = acc[pl][tl][2] = acc[pl][tl][3] = 0.0f;
  int rc = i0 / nch, cc = i0 - (i0 / nch) * nch;  // item being computed

  // One 64-column block: four k32 steps of one sparse mma per plane and token pair.
  auto block = [&](const uint32_t (&S)[NPL], const uint32_t (&F)[NPL], int k0) {
    uint32_t mA[NPL], mB[NPL], Sx[NPL];
#pragma unroll
    for (int pl = 0; pl < NPL; ++pl) {
      mA[pl] = (F[pl] & 0x55555555u) | 0x88888888u;
      mB[pl] = (__umulhi(F[pl], half_hi) & 0x55555555u) | 0x88888888u;
      Sx[pl] = S[pl];
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t bf[TILES][4];
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl)
#pragma unroll
        for (int i = 0; i < 4; ++i) bf[tl][i] = (uint32_t)xp[tl][k0 + 16 * s + 4 * i] * bmul;
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        uint32_t a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[i] = sign_operand(Sx[pl], smask);
          Sx[pl] *= two;  // the next register's signs move to bits 15 and 31
        }
        const uint32_t e = (s & 1) ? mB[pl] : mA[pl];
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) {
          if (s < 2) mma_sp_bf16<0>(acc[pl][tl], a, bf[tl], e);
          else mma_sp_bf16<1>(acc[pl][tl], a, bf[tl], e);
        }
      }
    }
  };

  for (int i = i0; i < i1; ++i) {
    const int slot = (i - i0) & 1;
    if (i + 1 < i1) {
      issue(slot ^ 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    if (cc < fullc) {  // two blocks from the ring: (S, F) of block 2cc and 2cc + 1 per plane
      const unsigned char* rs = msm + (ring - sbase) + slot * kSlot + lane * 16;
      uint32_t S0[NPL], F0[NPL], S1[NPL], F1[NPL];
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const uint4 v = *reinterpret_cast<const uint4*>(rs + pl * 512);
        S0[pl] = v.x;
        F0[pl] = v.y;
        S1[pl] = v.z;
        F1[pl] = v.w;
      }
      block(S0, F0, 128 * cc);
      block(S1, F1, 128 * cc + 64);
    } else {  // odd last block: 8 bytes per lane, read directly
      uint32_t S[NPL], F[NPL];
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(plane0 + (uint32_t)pl * pstride + (uint32_t)rc * tile_row +
                                                              (uint32_t)fullc * 512u + (uint32_t)lane * 8u));
        S[pl] = v.x;
        F[pl] = v.y;
      }
      block(S, F, 128 * cc);
    }
    const int r = rc;
    if (++cc == nch) {
      cc = 0;
      ++rc;
    }
    if (i + 1 == i1 || rc != r) {
      // even lanes hold (ra, ia), odd lanes (rb, ib) of token 2 tl + (q >> 1), rows g and g + 8
      const int64_t j0 = (rt_begin + r) * 16 + g, j1 = j0 + 8;
      float yr[TILES][2], yi[TILES][2];
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl) yr[tl][0] = yr[tl][1] = yi[tl][0] = yi[tl][1] = 0.0f;
#pragma unroll
      for (int pl = 0; pl < NPL; ++pl) {
        const float sr0 = j0 < n ? __ldg(P.scales + ((int64_t)pl * 2 + 0) * n + j0) : 0.0f;
        const float si0 = j0 < n ? __ldg(P.scales + ((int64_t)pl * 2 + 1) * n + j0) : 0.0f;
        const float sr1 = j1 < n ? __ldg(P.scales + ((int64_t)pl * 2 + 0) * n + j1) : 0.0f;
        const float si1 = j1 < n ? __ldg(P.scales + ((int64_t)pl * 2 + 1) * n + j1) : 0.0f;
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl) {
          float o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) o[u] = __shfl_xor_sync(0xffffffffu, acc[pl][tl][u], 1);
          plane_epilogue(pl / T, sr0, si0, 0.5f * acc[pl][tl][0], 0.5f * o[0], 0.5f * acc[pl][tl][1], 0.5f * o[1],
                         yr[tl][0], yi[tl][0]);
          plane_epilogue(pl / T, sr1, si1, 0.5f * acc[pl][tl][2], 0.5f * o[2], 0.5f * acc[pl][tl][3], 0.5f * o[3],
                         yr[tl][1], yi[tl][1]);
          acc[pl][tl][0] = acc[pl][tl][1] = acc[pl][tl][2] = acc[pl][tl][3] = 0.0f;
        }
      }
#pragma unroll
      for (int tl = 0; tl < TILES; ++tl) {
        float2* dst = red + ((size_t)((r * WARPS + warp) * TILES + tl) * 32 + lane) * 2;
        dst[0] = make_float2(yr[tl][0], yi[tl][0]);
        dst[1] = make_float2(yr[tl][1], yi[tl][1]);
      }
    }
  }
  __syncthreads();

  // fixed-order sum over the warps' partials (even lanes), then store
  for (int e = tid; e < niter * TILES * 32; e += WARPS * 32) {
    const int ln = e & 31;
    if (ln & 1) continue;
    const int tl = (e >> 5) % TILES;
    const int r = (e >> 5) / TILES;
    const int tok = 2 * tl + ((ln & 3) >> 1);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int64_t j = (rt_begin + r) * 16 + 8 * rr + (ln >> 2);
      float re = 0.0f, im = 0.0f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float2 v = red[((size_t)((r * WARPS + w) * TILES + tl) * 32 + ln) * 2 + rr];
        re += v.x;
        im += v.y;
      }
      if (tok < M && j < n) {
        float* yrow = P.y + (int64_t)tok * 2 * n;
        yrow[j] = re;
        yrow[n + j] = im;
      }
    }
  }
}

}  // namespace f2i
