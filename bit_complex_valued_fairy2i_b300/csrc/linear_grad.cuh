// Input gradient of the layer, dL/dx = U^^H g + W^^T conj(g), for training
// through the quantized layer with the straight-through estimator
// ("Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights {±1, ±i}",
// quantization-aware training; "Fairy2i-W2" card, y = Ux + W conj(x)).
//
// The real form of the layer is a real matrix; its transpose is the real form
// of (U^^H, W^^T), so the gradient is a transposed product over the same packed
// codes.  Per row j and plane (matrix X, stage t) the row's gradient g_j is
// scaled once per axis:
//   U:  h_re = s_re g_j,          h_im = s_im (-i g_j)
//   W:  h_re = s_re conj(g_j),    h_im = s_im (i conj(g_j))
// and every code adds or subtracts the h of its axis into its column.
//
// Work split: one CTA per (layer, 64-column block, quarter of the row tiles,
// token pair); one launch may carry several layers (a decoder block's
// projections), each with its own codes, gradients and outputs.  A warp walks
// row tiles; lane (g, q) owns columns 16 s + 8 h + 2 q + e of rows g and g + 8
// (its sign word; the axis flags of its columns sit in the flag words of the
// four lanes of its quad, exchanged by shuffles).  Partial
// sums are reduced over the 8 lanes of a column, then over the warps in shared
// memory, then over the 4 CTAs of a thread-block cluster by rank 0 through
// distributed shared memory, always in a fixed order: the result is
// deterministic and no global scratch is used.
#pragma once
#include <cooperative_groups.h>

#include <cstdint>

#include "layout.cuh"

namespace f2i {

constexpr int kGxWarps = 8;
constexpr int kGxCluster = 4;  // CTAs per column block (row split); 4 measured faster than 2 or 8
constexpr int kGxMaxTokens = 16382;

constexpr int kGxMaxGroup = 32;

struct GradProblem {
  const uint8_t* codes;
  const float* scales;
  const float* g;  // [M][2n]
  float* gx;       // [M][2m]
  int64_t n, m;
  int32_t kb_begin;  // first blockIdx.x of this layer (its column blocks follow)
  int32_t pad_;
};

struct GradGroup {
  int32_t count, T, M, pad_;
  GradProblem p[kGxMaxGroup];
};

// TOK = tokens per CTA (1 or 2; a launch with more tokens uses TOK = 2 over token pairs).
template <int TOK>
__global__ void __cluster_dims__(1, kGxCluster, 1) __launch_bounds__(kGxWarps * 32)
    linear_grad_x_kernel(const __grid_constant__ GradGroup G) {
  namespace cg = cooperative_groups;
  __shared__ float red[kGxWarps][4][16][2][2];  // [warp][q][column][token][re, im]
  __shared__ float cta_sum[4][16][2][2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  int pi = 0;
  for (int i = 1; i < G.count; ++i)
    if ((int)blockIdx.x >= G.p[i].kb_begin) pi = i;
  const GradProblem& P = G.p[pi];
  const int64_t n = P.n, m = P.m;
  const int T = G.T, M = G.M;
  const int64_t KB = col_blocks(m), RT = row_tiles(n), pbytes = plane_bytes(n, m);
  const int kb = (int)blockIdx.x - P.kb_begin;
  const int rank = blockIdx.y % kGxCluster, tp = blockIdx.y / kGxCluster;
  const int t0 = TOK * tp;
  const bool has_t1 = TOK == 2 && t0 + 1 < M;
  const int64_t rt_begin = RT * rank / kGxCluster, rt_end = RT * (rank + 1) / kGxCluster;

  float acc[16][TOK][2];
#pragma unroll
  for (int c = 0; c < 16; ++c)
#pragma unroll
    for (int tk = 0; tk < TOK; ++tk) acc[c][tk][0] = acc[c][tk][1] = 0.0f;

  const float* g0 = P.g + (int64_t)t0 * 2 * n;
  const float* g1 = has_t1 ? g0 + 2 * n : g0;
  for (int64_t rt = rt_begin + warp; rt < rt_end; rt += kGxWarps) {
    const int64_t j0 = rt * 16 + g, j1 = j0 + 8;
    // gradient of rows j0, j1 for both tokens (zero past n)
    float ga[2][TOK], gb[2][TOK];  // [rho][token]
#pragma unroll
    for (int rho = 0; rho < 2; ++rho) {
      const int64_t j = rho ? j1 : j0;
      const bool ok = j < n;
      ga[rho][0] = ok ? __ldg(g0 + j) : 0.0f;
      gb[rho][0] = ok ? __ldg(g0 + n + j) : 0.0f;
      if (TOK == 2) {
        ga[rho][TOK - 1] = ok && has_t1 ? __ldg(g1 + j) : 0.0f;
        gb[rho][TOK - 1] = ok && has_t1 ? __ldg(g1 + n + j) : 0.0f;
      }
    }
    // planes in groups of four: the group's code words and scales are loaded before any is used
    for (int p0 = 0; p0 < 2 * T; p0 += 4) {
      uint2 wv[4];
      float sre[4][2], sim[4][2];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int p = p0 + pp;
        const bool pok = p < 2 * T;
        wv[pp] = pok ? __ldcs(reinterpret_cast<const uint2*>(P.codes + p * pbytes + pair_offset(rt, kb, lane, KB)))
                     : make_uint2(0u, 0u);
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          const int64_t j = rho ? j1 : j0;
          const bool ok = pok && j < n;
          sre[pp][rho] = ok ? __ldg(P.scales + (int64_t)(2 * p) * n + j) : 0.0f;
          sim[pp][rho] = ok ? __ldg(P.scales + (int64_t)(2 * p + 1) * n + j) : 0.0f;
        }
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int p = p0 + pp;
        if (p >= 2 * T) break;
        const int X = p / T;
        const uint32_t S = wv[pp].x;
        uint32_t Fq[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) Fq[qq] = __shfl_sync(0xffffffffu, wv[pp].y, (lane & ~3) | qq) >> (4 * q);
        // per row: the real-axis value hre and the difference him - hre of each token, complex
        float hre[2][TOK][2], hd[2][TOK][2];  // [rho][token][re, im]
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          const float s_re = sre[pp][rho], s_im = sim[pp][rho];
#pragma unroll
          for (int tk = 0; tk < TOK; ++tk) {
            const float a = ga[rho][tk], b = gb[rho][tk];
            const float him_re = s_im * b, him_im = X == 0 ? -s_im * a : s_im * a;
            hre[rho][tk][0] = s_re * a;
            hre[rho][tk][1] = X == 0 ? s_re * b : -s_re * b;
            hd[rho][tk][0] = him_re - hre[rho][tk][0];
            hd[rho][tk][1] = him_im - hre[rho][tk][1];
          }
        }
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 4 * s + 2 * h + e;  // column 16 s + 8 h + 2 q + e of the block
#pragma unroll
              for (int rho = 0; rho < 2; ++rho) {
                // sign bit of the code moved to bit 31: sgn = +-1.0; axis flag spread to a word
                // mask: sf = sgn for an imaginary-axis code, 0 otherwise.  The code then adds
                // sgn * hre + sf * (him - hre), i.e. +-(its axis' value), on the FMA pipe.
                const int kSign = 15 + 16 * e - (4 * s + 2 * h + rho);
                const int kFlag = 16 * rho + (s & 1) + 2 * e;
                const uint32_t sgn = ((S << (31 - kSign)) & 0x80000000u) | 0x3f800000u;
                const uint32_t fmask = (uint32_t)((int32_t)(Fq[h + 2 * (s >> 1)] << (31 - kFlag)) >> 31);
                const float fs = __uint_as_float(sgn), fsf = __uint_as_float(sgn & fmask);
#pragma unroll
                for (int tk = 0; tk < TOK; ++tk) {
                  acc[c][tk][0] = fmaf(fs, hre[rho][tk][0], acc[c][tk][0]);
                  acc[c][tk][0] = fmaf(fsf, hd[rho][tk][0], acc[c][tk][0]);
                  acc[c][tk][1] = fmaf(fs, hre[rho][tk][1], acc[c][tk][1]);
                  acc[c][tk][1] = fmaf(fsf, hd[rho][tk][1], acc[c][tk][1]);
                }
              }
            }
      }
    }
  }
  // over the 8 lanes g of each column (lane = 4 g + q), fixed butterfly order
#pragma unroll
  for (int c = 0; c < 16; ++c)
#pragma unroll
    for (int tk = 0; tk < TOK; ++tk)
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float v = acc[c][tk][part];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        acc[c][tk][part] = v;
      }
  if (g == 0) {
#pragma unroll
    for (int c = 0; c < 16; ++c)
#pragma unroll
      for (int tk = 0; tk < 2; ++tk) {
        red[warp][q][c][tk][0] = tk < TOK ? acc[c][tk < TOK ? tk : 0][0] : 0.0f;
        red[warp][q][c][tk][1] = tk < TOK ? acc[c][tk < TOK ? tk : 0][1] : 0.0f;
      }
  }
  __syncthreads();
  {  // over the warps, in warp order: 256 threads = 4 q x 16 columns x 2 tokens x 2 parts
    const int qq = tid >> 6, c = (tid >> 2) & 15, tk = (tid >> 1) & 1, part = tid & 1;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kGxWarps; ++w) v += red[w][qq][c][tk][part];
    cta_sum[qq][c][tk][part] = v;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (rank == 0) {  // over the cluster's CTAs, in rank order
    const int qq = tid >> 6, c = (tid >> 2) & 15, tk = (tid >> 1) & 1, part = tid & 1;
    float v = 0.0f;
    for (int r = 0; r < kGxCluster; ++r) {
      const float* peer = cluster.map_shared_rank(&cta_sum[0][0][0][0], r);
      v += peer[((qq * 16 + c) * 2 + tk) * 2 + part];
    }
    const int s = c >> 2, h = (c >> 1) & 1, e = c & 1;
    const int64_t col = (int64_t)kb * 64 + 16 * s + 8 * h + 2 * qq + e;
    const int t = t0 + tk;
    if (col < m && t < M) P.gx[(int64_t)t * 2 * m + part * m + col] = v;
  }
  cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

}  // namespace f2i
