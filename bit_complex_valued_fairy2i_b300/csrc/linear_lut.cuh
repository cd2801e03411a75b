// Layer evaluation by table lookup over layout 3 (decode token counts).
//
// The layer ("Fairy2i-W2" model card, y = Ux + W conj(x); "Fairy2i: Ultra-Low-
// Bit LLM Quantization Using Complex Weights {±1, ±i}", "Industry
// implications: multiplication-free inference") needs, per output row and
// code plane (matrix X, stage t), the two signed sums A_re (real-coded
// columns) and A_im (imaginary-coded columns) of x.  With sigma the code's
// sign and tau = +1 (real axis) or -1 (imaginary axis):
//   P = sum sigma x,  Q = sum sigma tau x,  A_re = (P + Q) / 2,  A_im = (P - Q) / 2.
// Both P and Q are sums of +-x only, so they are read from tables: for every
// group of 8 columns the 256 signed sums of its 8 activations, indexed by a
// byte of sign bits (P) or of sign-XOR-axis bits (Q).  Each lookup replaces 8
// complex adds; the inner loop per byte is one byte permute (the shared-memory
// address), one shared load and two fp32 adds of the fp16 table entry.
//
// Tables: one per (window of 256 columns, token), 32 groups x 256 entries of
// packed fp16 (re, im), entry e of group G at byte e * 256 + 4 G of a 64 KB
// region (two tables share a region, offset by 128 bytes).  Lane r of a warp
// owns row r of a 32-row tile; at each byte position of layout 3 the 32 rows
// name 32 different groups, so the 32 lanes hit 32 different banks.  The
// activations of a table are scaled by a power of two (the window maximum
// lands in [2^10, 2^11)) so that every entry is a normal fp16 number; each
// entry is the fp32 sum of its 8 terms rounded once to fp16, and the entries
// of two consecutive groups are added in fp16 before the fp32 accumulation.
//
// Work: a unit is (layer, window, row tile) = 32 rows x 256 columns x 2T
// planes.  Units are numbered window-major inside a layer and split evenly
// (by slot count) over one CTA per SM.  A CTA builds the tables of the
// windows its units touch, then its 16 warps take units in turn, streaming
// the codes through per-warp shared-memory rings (cp.async).  A unit's fp32
// accumulators become a partial output (scales applied): written to y for a
// layer of one window, otherwise to the caller's workspace, where a second
// kernel adds the windows of every row in window order.  Results are
// deterministic: every sum has a fixed order.
//
// The decode is launched as a programmatic dependent of the previous kernel
// in the stream: before griddepcontrol.wait a CTA only issues L2 prefetches
// of its codes (weights, never written by the decode) and of its first
// activations; every read of activations, codes into shared memory, and every
// write comes after it.  The reduction is an ordinary launch after it.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include "layout.cuh"

namespace f2i {

constexpr int kLutWarps = 16;
constexpr int kLutThreads = kLutWarps * 32;
constexpr int kLutMaxGroup = 32;
constexpr int kLutMaxCtas = 160;  // one CTA per SM (148 on B300); bounds the launch parameters
constexpr uint32_t kLutSmemBytes = 224u * 1024u;  // dynamic shared memory: covers [base, 224 KB) for any base

// Largest token count of one launch for T stages (fp32 accumulators and the
// double-buffered code words stay within 128 registers).
__host__ __device__ constexpr int lut_max_tokens(int T) { return T <= 2 ? 3 : T == 3 ? 2 : 1; }
// Tokens of the launch that starts at token t0 of M.  For T <= 2, launches of
// 2 tokens, the first of 3 when M is odd: per LLaMA-2-7B block, launches of 1,
// 2, 3 and 4 tokens took 17.5, 27.2, 41.0 and 59.0 us, so 2 or 3 tokens a
// launch cost the least per token.  Otherwise as many as lut_max_tokens.
__host__ __device__ constexpr int lut_launch_tokens(int64_t M, int64_t t0, int T) {
  return T > 2 ? (int)(M - t0 < lut_max_tokens(T) ? M - t0 : lut_max_tokens(T))
               : (t0 == 0 && M >= 3 && (M & 1)) ? 3 : (int)(M - t0 < 2 ? M - t0 : 2);
}

struct LutProblem {
  const uint8_t* codes;
  const float* scales;
  const uint16_t* x;  // bfloat16 [M][2m] (this launch's tokens)
  float* y;           // [M][2n], fp32 or (out_bf16) bfloat16 elements
  int32_t n, m;
  int32_t tiles;       // row tiles of 32 rows
  int32_t windows;     // column windows of 256
  int32_t unit_begin;  // first unit of the layer in the launch
  int32_t out_bf16;
  int64_t part_begin;  // first partial output (float2) in the workspace
};

// A run of a CTA's units inside one (layer, window).
struct LutSeg {
  int32_t unit, tau0;  // first unit; its row tile
  uint16_t win;
  uint8_t prob, nb;    // layer; slots of the window
};

struct LutParams {
  int32_t count, M, total_units, pad_;
  float2* partials;
  LutProblem p[kLutMaxGroup];
  int32_t cta_begin[kLutMaxCtas + 1];
  // every CTA's first batch of segments (up to two), computed on the host so
  // that no CTA starts with a serial search after the dependency wait
  LutSeg first[kLutMaxCtas][2];
  int32_t first_end[kLutMaxCtas];  // unit after the first batch
  uint8_t first_nseg[kLutMaxCtas];
};

// The window-combining pass: one thread per (row of a 32-row tile, token) of
// every layer with more than one window.
struct LutReduceProblem {
  float* y;            // fp32 or (out_bf16) bfloat16 elements
  const float2* part;  // [window][tile][token][32]
  int32_t n, tiles, windows, row_begin;  // row_begin: first padded row of the layer in the pass
  int32_t out_bf16, pad_;
};
struct LutReduceParams {
  int32_t count, M, total_rows, pad_;
  LutReduceProblem p[kLutMaxGroup];
};


__device__ __forceinline__ uint32_t lut_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
template <uint32_t OFF>
__device__ __forceinline__ uint32_t lut_lds(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}
template <uint32_t OFF>
__device__ __forceinline__ uint2 lut_lds2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(addr), "n"(OFF));
  return v;
}
// fp16x2 sum of two table entries (one rounding per half)
__device__ __forceinline__ uint32_t lut_hadd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// acc_re += lo(e), acc_im += hi(e): fp16 table entry added in fp32 (one rounding each)
__device__ __forceinline__ void lut_add(float& re, float& im, uint32_t e) {
  unsigned short lo, hi;
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(e));
  asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(re) : "h"(lo));
  asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(im) : "h"(hi));
}

__device__ __forceinline__ int lut_problem_of(const LutParams& P, int u) {
  int pi = 0;
  for (int i = 1; i < P.count; ++i)
    if (u >= P.p[i].unit_begin) pi = i;
  return pi;
}

// Shared-memory map: the warps' code rings from the bottom, the tables in the
// top one (M <= 2) or two (M = 3, 4) 64 KB regions below 224 KB.  Table set z
// of a resident segment s and token t, in region z >> 1 (256 bytes per entry
// index):
//   M = 1: two windows, slot S of set z at 4 S + 128 (z & 1);
//   M = 3 (and M = 2 at T > 2): one window, slot S of token t at
//   4 S + 128 (t & 1) of region t >> 1;
//   M = 2 at T <= 2: one window, the two tokens' entries of slot S side by
//   side at 8 S + 4 t, so one 8-byte load reads both.
//   (Pairs at M = 3 measured slower, 46.3 against 41.2 us per LLaMA-2-7B
//   block: the third token's loads then need more registers than the kernel
//   has; at T = 3 the pair kernel spills too.)
template <int T, int M>
__host__ __device__ constexpr bool lut_pairs() { return T <= 2 && M == 2; }
template <int M>
__host__ __device__ constexpr uint32_t lut_table_base() { return M <= 2 ? 160u * 1024u : 96u * 1024u; }
template <int M>
__host__ __device__ constexpr int lut_segments() { return M == 1 ? 2 : 1; }
template <int M>
__device__ __forceinline__ int lut_set(int s, int t) { return M == 1 ? s : t; }
// Shared-address part of set z that the lane's B word carries (bit 7 = the
// half) and the part given as an immediate offset of the loads.
template <int M>
__device__ __forceinline__ uint32_t lut_b_bits(int s) { return M == 1 ? ((uint32_t)s & 1u) << 7 : 0u; }
template <int T, int M, int t>
__host__ __device__ constexpr uint32_t lut_imm() {
  return lut_table_base<M>() + 65536u * (t >> 1) + (lut_pairs<T, M>() ? 0u : 128u * (t & 1));
}
// Bytes per slot of an entry row: 4, or 8 for token pairs.
template <int T, int M>
__host__ __device__ constexpr uint32_t lut_slot_stride() { return lut_pairs<T, M>() ? 8u : 4u; }
// Code ring of a warp: RING slots of 2T planes x 512 bytes (32 lanes x 16
// bytes) filled by cp.async; a slot is refilled after the evaluation that
// read it, so RING - 1 slots are in flight (at most 4 slots; the rings of the
// 16 warps stay below the tables with 2 KB to spare for the base).
__host__ __device__ constexpr uint32_t lut_slot_bytes(int T) { return 2u * T * 512u; }
template <int T, int M>
__host__ __device__ constexpr int lut_ring() {
  return (lut_table_base<M>() - 2048u) / (kLutWarps * lut_slot_bytes(T)) >= 4
             ? 4
             : (int)((lut_table_base<M>() - 2048u) / (kLutWarps * lut_slot_bytes(T)));
}

// One slot (8 groups x 2T planes) of a unit: for step i the lane reads group
// slot bj ^ i of every plane's table (P from the sign byte, Q from the q
// byte; bj and the XOR in units of the slot stride).  The entries of steps
// 2 k and 2 k + 1 are added in fp16 (one rounding; the activation scaling
// keeps the sum below 2^15) and the sum is added to the fp32 accumulators.
// With token pairs one 8-byte load serves both tokens.
template <int T, int M>
__device__ __forceinline__ void lut_slot(const uint4 (&c)[2 * T], uint32_t bj, float (&acc)[M][2 * T][4]) {
  static_assert(M <= 3, "at most three tokens per launch");
  constexpr uint32_t SW = lut_slot_stride<T, M>();
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint32_t b0 = bj ^ (SW * (uint32_t)i), b1 = bj ^ (SW * (uint32_t)(i + 1));
    const uint32_t sel0 = 0x7604u | ((uint32_t)(i & 3) << 4), sel1 = 0x7604u | ((uint32_t)((i + 1) & 3) << 4);
#pragma unroll
    for (int p = 0; p < 2 * T; ++p) {
      const uint32_t ws = i < 4 ? c[p].x : c[p].y, wq = i < 4 ? c[p].z : c[p].w;
      const uint32_t aP0 = lut_prmt(ws, b0, sel0), aP1 = lut_prmt(ws, b1, sel1);
      const uint32_t aQ0 = lut_prmt(wq, b0, sel0), aQ1 = lut_prmt(wq, b1, sel1);
      if constexpr (!lut_pairs<T, M>()) {
        lut_add(acc[0][p][0], acc[0][p][1], lut_hadd2(lut_lds<lut_imm<T, M, 0>()>(aP0), lut_lds<lut_imm<T, M, 0>()>(aP1)));
        lut_add(acc[0][p][2], acc[0][p][3], lut_hadd2(lut_lds<lut_imm<T, M, 0>()>(aQ0), lut_lds<lut_imm<T, M, 0>()>(aQ1)));
        if constexpr (M > 1) {
          lut_add(acc[1][p][0], acc[1][p][1],
                  lut_hadd2(lut_lds<lut_imm<T, M, 1>()>(aP0), lut_lds<lut_imm<T, M, 1>()>(aP1)));
          lut_add(acc[1][p][2], acc[1][p][3],
                  lut_hadd2(lut_lds<lut_imm<T, M, 1>()>(aQ0), lut_lds<lut_imm<T, M, 1>()>(aQ1)));
        }
        if constexpr (M > 2) {
          lut_add(acc[2][p][0], acc[2][p][1],
                  lut_hadd2(lut_lds<lut_imm<T, M, 2>()>(aP0), lut_lds<lut_imm<T, M, 2>()>(aP1)));
          lut_add(acc[2][p][2], acc[2][p][3],
                  lut_hadd2(lut_lds<lut_imm<T, M, 2>()>(aQ0), lut_lds<lut_imm<T, M, 2>()>(aQ1)));
        }
      } else {
        {
          const uint2 p0 = lut_lds2<lut_imm<T, M, 0>()>(aP0), p1 = lut_lds2<lut_imm<T, M, 0>()>(aP1);
          const uint2 q0 = lut_lds2<lut_imm<T, M, 0>()>(aQ0), q1 = lut_lds2<lut_imm<T, M, 0>()>(aQ1);
          lut_add(acc[0][p][0], acc[0][p][1], lut_hadd2(p0.x, p1.x));
          lut_add(acc[0][p][2], acc[0][p][3], lut_hadd2(q0.x, q1.x));
          lut_add(acc[1][p][0], acc[1][p][1], lut_hadd2(p0.y, p1.y));
          lut_add(acc[1][p][2], acc[1][p][3], lut_hadd2(q0.y, q1.y));
        }
      }
    }
  }
}

// The lane's group in window w (its first column), and whether two 16-byte
// loads fetch its 8 activations (m a multiple of 8, x 16-byte aligned, the
// group inside the layer).
__device__ __forceinline__ int64_t lut_group_col(const LutProblem& L, int w) {
  const int lane = threadIdx.x & 31;
  return 256 * (int64_t)w + 8 * (lane & (8 * l3_slots(L.m, w) - 1));
}
__device__ __forceinline__ bool lut_x_vector(const LutProblem& L, int64_t k0) {
  return (L.m & 7) == 0 && (reinterpret_cast<uintptr_t>(L.x) & 15) == 0 && k0 < L.m;
}
// Issues the two 16-byte loads (Re, Im) of the lane's group for token t, so
// that they are in flight before the codes; zeros where the build reads the
// activations one by one instead.
__device__ __forceinline__ void lut_fetch_x(const LutProblem& L, int w, int t, uint4& va, uint4& vb) {
  const int64_t k0 = lut_group_col(L, w);
  va = vb = make_uint4(0u, 0u, 0u, 0u);
  if (lut_x_vector(L, k0)) {
    const uint16_t* xa = L.x + (int64_t)t * 2 * L.m;
    va = *reinterpret_cast<const uint4*>(xa + k0);
    vb = *reinterpret_cast<const uint4*>(xa + L.m + k0);
  }
}

// Builds the table of (window w of layer L, token t) into set z from the
// lane's activations (va, vb from lut_fetch_x): warp h writes entries
// 16 h .. 16 h + 15 of every slot (lane = slot).  Slot S holds group
// S & (8 nb - 1): a partial window's groups are repeated over all 32 slots, so
// that the lanes that share a group read different banks.  Returns the factor
// 2^e that undoes the activation scaling.
template <bool PAIRS>
__device__ __forceinline__ float lut_build(const LutProblem& L, int w, int t, int z, uint32_t tbase, uint4 va,
                                           uint4 vb) {
  const int lane = threadIdx.x & 31, h = threadIdx.x >> 5;
  const int64_t m = L.m;
  const int64_t k0 = lut_group_col(L, w);
  const uint16_t* xa = L.x + (int64_t)t * 2 * m;
  float a[8], b[8];
  if (lut_x_vector(L, k0)) {
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      a[2 * c] = __uint_as_float(wa[c] << 16);
      a[2 * c + 1] = __uint_as_float(wa[c] & 0xFFFF0000u);
      b[2 * c] = __uint_as_float(wb[c] << 16);
      b[2 * c + 1] = __uint_as_float(wb[c] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const bool in = k0 + c < m;
      a[c] = in ? __uint_as_float((uint32_t)xa[k0 + c] << 16) : 0.0f;
      b[c] = in ? __uint_as_float((uint32_t)xa[m + k0 + c] << 16) : 0.0f;
    }
  }
  // window maximum over finite magnitudes (every warp holds the whole window)
  float mx = 0.0f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float fa = fabsf(a[c]), fb = fabsf(b[c]);
    mx = fmaxf(mx, isfinite(fa) ? fa : 0.0f);
    mx = fmaxf(mx, isfinite(fb) ? fb : 0.0f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  // e: mx 2^-e in [2^10, 2^11), so an entry (8 terms) stays below 2^14 and
  // the fp16 sum of two entries below 2^15; clamped so that 2^-e and 2^e are
  // normal floats
  int e = 0;
  if (mx > 0.0f) {
    const int ex = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // a subnormal maximum gives -127, then the clamp
    e = max(ex - 10, -126);
  }
  const float down = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    a[c] *= down;
    b[c] *= down;
  }
  // entry (16 h + l) = sum over c of (bit c set ? -1 : +1) (a_c, b_c)
  float hr = 0.0f, hi = 0.0f;
#pragma unroll
  for (int c = 4; c < 8; ++c) {
    const bool neg = (h >> (c - 4)) & 1;
    hr += neg ? -a[c] : a[c];
    hi += neg ? -b[c] : b[c];
  }
  float pr[4], pi[4], qr[4], qi[4];  // +-x0 +-x1 and +-x2 +-x3, index = the two sign bits
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    pr[v] = ((v & 1) ? -a[0] : a[0]) + ((v & 2) ? -a[1] : a[1]);
    pi[v] = ((v & 1) ? -b[0] : b[0]) + ((v & 2) ? -b[1] : b[1]);
    qr[v] = ((v & 1) ? -a[2] : a[2]) + ((v & 2) ? -a[3] : a[3]) + hr;
    qi[v] = ((v & 1) ? -b[2] : b[2]) + ((v & 2) ? -b[3] : b[3]) + hi;
  }
  // slot = lane: 4 bytes apart in the set's own half-row, or (PAIRS) 8 apart
  // beside the pair's other token
  const uint32_t set_addr =
      tbase + ((uint32_t)z >> 1) * 65536u + (PAIRS ? ((uint32_t)z & 1u) * 4u : ((uint32_t)z & 1u) * 128u);
  const uint32_t sw = PAIRS ? 8u : 4u;
#pragma unroll
  for (int l = 0; l < 16; ++l) {
    const float er = pr[l & 3] + qr[l >> 2], ei = pi[l & 3] + qi[l >> 2];
    const __half2 hv = __floats2half2_rn(er, ei);
    const uint32_t addr = set_addr + (uint32_t)(16 * h + l) * 256u + sw * (uint32_t)lane;
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(*reinterpret_cast<const uint32_t*>(&hv)) : "memory");
  }
  return __uint_as_float((uint32_t)(127 + e) << 23);  // 2^e
}

template <int T, int M>
__global__ void __launch_bounds__(kLutThreads, 1) linear_lut_kernel(const __grid_constant__ LutParams P) {
  extern __shared__ __align__(16) uint8_t lsm[];
  constexpr int NP = 2 * T;
  constexpr int S = lut_segments<M>();
  constexpr int RING = lut_ring<T, M>();
  constexpr uint32_t SLOT = lut_slot_bytes(T);
  __shared__ int s_nseg;
  __shared__ int s_unit[S + 1];  // unit range of each resident segment
  __shared__ int s_prob[S], s_win[S], s_tau0[S], s_nb[S];
  __shared__ const uint8_t* s_codes[S];  // codes of the segment's first unit
  __shared__ float s_pow[S][M];          // 2^e per (segment, token)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // rings at [base, ...), tables at [lut_table_base, 224 KB): all inside this
  // CTA's dynamic shared memory
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(lsm);
  const uint32_t ring_base = (base + 15u) & ~15u;
  if (base + kLutSmemBytes < 224u * 1024u || ring_base + kLutWarps * RING * SLOT > lut_table_base<M>()) {
    if (tid == 0) f2i_raise(kErrConfig);  // refuse rather than address memory outside the CTA's buffer
    return;
  }
  const uint32_t ring0 = ring_base + (uint32_t)warp * RING * SLOT + (uint32_t)lane * 16u;
  const int u_end = P.cta_begin[blockIdx.x + 1];
  int u = P.cta_begin[blockIdx.x];
  pdl_launch_dependents();
  // Before the dependency wait only L2 prefetches (the L2 is coherent, so a
  // prefetch never exposes stale data): warp w the codes of unit u + w, warp
  // 15 the activations of the first window for every token.
  if (lane == 0 && u < u_end) {
    const LutProblem& L0 = P.p[P.first[blockIdx.x][0].prob];
    const int w0 = P.first[blockIdx.x][0].win;
    if (warp < kLutWarps - 1 && u + warp < u_end) {
      const int uu = u + warp;
      const int pi = uu < L0.unit_begin + (w0 + 1) * L0.tiles ? P.first[blockIdx.x][0].prob : lut_problem_of(P, uu);
      const LutProblem& L = P.p[pi];
      const int w = (uu - L.unit_begin) / L.tiles;
      const uint8_t* cp0 = L.codes + l3_offset(L.n, L.m, T, w, uu - L.unit_begin - w * L.tiles, 0);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cp0),
                   "r"((uint32_t)(NP * l3_slots(L.m, w)) * (uint32_t)kL3SlotBytes)
                   : "memory");
    } else if (warp == kLutWarps - 1 && (L0.m & 7) == 0 && (reinterpret_cast<uintptr_t>(L0.x) & 15) == 0) {
      const int64_t k0 = 256 * (int64_t)w0;
      const uint32_t bytes = (uint32_t)(min((int64_t)256, (int64_t)L0.m - k0) * 2) & ~15u;
      for (int t = 0; t < M && bytes > 0; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(L0.x + (int64_t)t * 2 * L0.m + h * L0.m + k0),
                       "r"(bytes)
                       : "memory");
    }
  }
  pdl_wait();
  bool first_batch = true;
  while (u < u_end) {
    if (first_batch) {  // the host's segments: one thread per segment
      const int nseg0 = P.first_nseg[blockIdx.x];
      if (tid < nseg0) {
        const LutSeg& g = P.first[blockIdx.x][tid];
        const LutProblem& L = P.p[g.prob];
        s_unit[tid] = g.unit;
        s_prob[tid] = g.prob;
        s_win[tid] = g.win;
        s_tau0[tid] = g.tau0;
        s_nb[tid] = g.nb;
        s_codes[tid] = L.codes + l3_offset(L.n, L.m, T, g.win, g.tau0, 0);
      }
      if (tid == 0) {
        s_nseg = nseg0;
        s_unit[nseg0] = P.first_end[blockIdx.x];
      }
      first_batch = false;
    } else if (tid == 0) {
      int s = 0, uu = u;
      while (s < S && uu < u_end) {
        const int pi = lut_problem_of(P, uu);
        const LutProblem& L = P.p[pi];
        const int w = (uu - L.unit_begin) / L.tiles;
        s_unit[s] = uu;
        s_prob[s] = pi;
        s_win[s] = w;
        s_tau0[s] = uu - L.unit_begin - w * L.tiles;
        s_nb[s] = l3_slots(L.m, w);
        s_codes[s] = L.codes + l3_offset(L.n, L.m, T, w, s_tau0[s], 0);
        uu = min(u_end, L.unit_begin + (w + 1) * L.tiles);
        ++s;
      }
      s_nseg = s;
      s_unit[s] = uu;
    }
    __syncthreads();
    const int nseg = s_nseg;
    const int ub = s_unit[0], ue = s_unit[nseg];
    // a unit's codes (2T planes x nb slots, contiguous, consecutive tiles of a
    // segment one after another): pointer to lane 0's bytes
    auto unit_codes = [&](int uu, int& seg, int& nb) -> const uint8_t* {
      seg = 0;
#pragma unroll
      for (int k = 1; k < S; ++k)
        if (k < nseg && uu >= s_unit[k]) seg = k;
      nb = s_nb[seg];
      return s_codes[seg] + (uint32_t)(uu - s_unit[seg]) * ((uint32_t)(NP * nb) * (uint32_t)kL3SlotBytes);
    };

    // load cursor: the warp's units (ub + warp, + 16, ...) slot by slot into
    // its ring, RING - 1 slots ahead of evaluation; every call commits one group
    int lu = ub + warp, ljj = 0, lnb = 4, lseg = 0, lk = 0;
    const uint8_t* lcp = lu < ue ? unit_codes(lu, lseg, lnb) + lane * 16 : nullptr;
    auto issue = [&]() {
      if (lcp != nullptr) {
        const uint32_t dst = ring0 + (uint32_t)lk * SLOT;
#pragma unroll
        for (int p = 0; p < NP; ++p)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + (uint32_t)p * 512u),
                       "l"(lcp + (p * lnb + ljj) * kL3SlotBytes)
                       : "memory");
        if (++ljj == lnb) {
          ljj = 0;
          lu += kLutWarps;
          lcp = lu < ue ? unit_codes(lu, lseg, lnb) + lane * 16 : nullptr;
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      lk = lk + 1 == RING ? 0 : lk + 1;
    };
    // the activations of the tables first, then the codes: HBM streams while
    // the tables are built, and the activations do not queue behind the codes
    uint4 xva[S][M], xvb[S][M];
#pragma unroll
    for (int s = 0; s < S; ++s)
#pragma unroll
      for (int t = 0; t < M; ++t)
        if (s < nseg) lut_fetch_x(P.p[s_prob[s]], s_win[s], t, xva[s][t], xvb[s][t]);
#pragma unroll
    for (int r = 0; r < RING - 1; ++r) issue();

#pragma unroll
    for (int s = 0; s < S; ++s)
#pragma unroll
      for (int t = 0; t < M; ++t)
        if (s < nseg) {
          const float pw =
              lut_build<lut_pairs<T, M>()>(P.p[s_prob[s]], s_win[s], t, lut_set<M>(s, t), lut_table_base<M>(),
                                        xva[s][t], xvb[s][t]);
          if (tid == 0) s_pow[s][t] = pw;
        }
    __syncthreads();

    int ck = 0;  // ring slot evaluated next
    for (int uu = ub + warp; uu < ue; uu += kLutWarps) {
      int s, nb;
      unit_codes(uu, s, nb);
      const int pi = s_prob[s], w = s_win[s];
      const LutProblem& L = P.p[pi];
      const int tau = s_tau0[s] + (uu - s_unit[s]);
      const int64_t j = 32 * (int64_t)tau + lane;
      const bool row_in = j < L.n;
      // slot lane ^ (8 jj + i): group (lane & (8 nb - 1)) ^ (8 jj + i), bank = slot
      const uint32_t bbase = lut_slot_stride<T, M>() * (uint32_t)lane | lut_b_bits<M>(s);

      float acc[M][NP][4];
#pragma unroll
      for (int t = 0; t < M; ++t)
#pragma unroll
        for (int p = 0; p < NP; ++p) acc[t][p][0] = acc[t][p][1] = acc[t][p][2] = acc[t][p][3] = 0.0f;
      // the row's scales, in flight while the unit's slots are evaluated
      float sc[2 * NP];
#pragma unroll
      for (int k = 0; k < 2 * NP; ++k) sc[k] = row_in ? __ldg(L.scales + (int64_t)k * L.n + j) : 0.0f;
#pragma unroll 1
      for (int jj = 0; jj < nb; ++jj) {
        asm volatile("cp.async.wait_group %0;" ::"n"(RING - 2) : "memory");
        uint4 cw[NP];
        const uint32_t src = ring0 + (uint32_t)ck * SLOT;
#pragma unroll
        for (int p = 0; p < NP; ++p)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(cw[p].x), "=r"(cw[p].y), "=r"(cw[p].z), "=r"(cw[p].w)
                       : "r"(src + (uint32_t)p * 512u)
                       : "memory");
        ck = ck + 1 == RING ? 0 : ck + 1;
        lut_slot<T, M>(cw, bbase ^ (lut_slot_stride<T, M>() * 8u * (uint32_t)jj), acc);
        // refill the slot read one evaluation earlier (its registers are consumed)
        issue();
      }

      // epilogue: A_re = (P + Q) / 2, A_im = (P - Q) / 2 per plane, the row's
      // axis scales, then the window's 2^e (the 1/2 folded in)
      float yre[M], yim[M];
#pragma unroll
      for (int t = 0; t < M; ++t) yre[t] = yim[t] = 0.0f;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const int X = p / T;
        const float s_re = sc[2 * p], s_im = sc[2 * p + 1];
#pragma unroll
        for (int t = 0; t < M; ++t) {
          const float ra = acc[t][p][0] + acc[t][p][2], rb = acc[t][p][1] + acc[t][p][3];  // 2 A_re
          const float ia = acc[t][p][0] - acc[t][p][2], ib = acc[t][p][1] - acc[t][p][3];  // 2 A_im
          if (X == 0) {
            yre[t] += s_re * ra - s_im * ib;
            yim[t] += s_re * rb + s_im * ia;
          } else {
            yre[t] += s_re * ra + s_im * ib;
            yim[t] += -s_re * rb + s_im * ia;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < M; ++t) {
        const float f = 0.5f * s_pow[s][t];
        yre[t] *= f;
        yim[t] *= f;
      }
      const int64_t n2 = 2 * (int64_t)L.n;
      if (L.windows == 1) {
        if (row_in)
#pragma unroll
          for (int t = 0; t < M; ++t) {
            store_y(L.y, t * n2 + j, yre[t], L.out_bf16);
            store_y(L.y, t * n2 + L.n + j, yim[t], L.out_bf16);
          }
      } else {  // a partial output, combined over windows by lut_reduce_kernel
        float2* part = P.partials + L.part_begin;
#pragma unroll
        for (int t = 0; t < M; ++t)
          __stcg(part + (((int64_t)w * L.tiles + tau) * M + t) * 32 + lane, make_float2(yre[t], yim[t]));
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the batch

    u = ue;
    if (u < u_end) __syncthreads();  // the tables are rebuilt for the next segments
  }
}

// Sums the partial outputs of every row over the layer's windows and writes
// y.  Four threads per (row, token): thread q adds windows q, q + 4, ... in
// order, then the four sums are added as (s0 + s1) + (s2 + s3); a fixed order.
__global__ void __launch_bounds__(256) lut_reduce_kernel(const __grid_constant__ LutReduceParams R) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = (int64_t)R.total_rows * R.M * 4;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
    const int64_t idx = base + threadIdx.x;  // every thread of a warp takes the loop (shuffles below)
    const bool live = idx < total;
    const int64_t item = live ? idx >> 2 : 0;
    const int q = (int)(idx & 3);
    const int row = (int)(item / R.M), t = (int)(item - (int64_t)row * R.M);
    int pi = 0;
    for (int i = 1; i < R.count; ++i)
      if (row >= R.p[i].row_begin) pi = i;
    const LutReduceProblem& L = R.p[pi];
    const int r = row - L.row_begin, tau = r >> 5, lane = r & 31;
    float sr = 0.0f, si = 0.0f;
    if (live) {
      float2 v[6];
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        const int w = q + 4 * k;
        v[k] = w < L.windows ? __ldcg(L.part + (((int64_t)w * L.tiles + tau) * R.M + t) * 32 + lane)
                             : make_float2(0.0f, 0.0f);
      }
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        sr += v[k].x;
        si += v[k].y;
      }
      for (int w = q + 24; w < L.windows; w += 4) {  // layers of more than 24 windows
        const float2 u = __ldcg(L.part + (((int64_t)w * L.tiles + tau) * R.M + t) * 32 + lane);
        sr += u.x;
        si += u.y;
      }
    }
    // (s0 + s1) + (s2 + s3) over the four threads of the item
    sr += __shfl_xor_sync(0xffffffffu, sr, 1);
    si += __shfl_xor_sync(0xffffffffu, si, 1);
    sr += __shfl_xor_sync(0xffffffffu, sr, 2);
    si += __shfl_xor_sync(0xffffffffu, si, 2);
    if (live && q == 0 && r < L.n) {
      store_y(L.y, (int64_t)t * 2 * L.n + r, sr, L.out_bf16);
      store_y(L.y, (int64_t)t * 2 * L.n + L.n + r, si, L.out_bf16);
    }
  }
}

// Canonical codes of a layout-3 layer: out[plane][j][k] = 2 imag + sign.
__global__ void __launch_bounds__(256) unpack_codes_l3_kernel(const uint8_t* __restrict__ codes, int64_t n, int64_t m,
                                                              int T, uint8_t* __restrict__ out) {
  const int64_t G = (m + 7) / 8;
  const int64_t total = 2 * (int64_t)T * n * G;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t plane = idx / (n * G);
    const int64_t rem = idx - plane * n * G;
    const int64_t j = rem / G, g8 = rem - (rem / G) * G;
    const int64_t win = g8 >> 5;
    const int g = (int)(g8 & 31), r = (int)(j & 31), nb = l3_slots(m, win);
    const uint8_t* c = codes + l3_offset(n, m, T, win, j >> 5, (int)plane) + l3_slot_of(g, r, nb) * kL3SlotBytes +
                       r * 16 + l3_byte_of(g, r);
    const uint32_t s = c[0], q = c[8];
    uint8_t* dst = out + (plane * n + j) * m + 8 * g8;
#pragma unroll
    for (int b = 0; b < 8; ++b)
      if (8 * g8 + b < m) dst[b] = (uint8_t)(2u * (((s ^ q) >> b) & 1u) + ((s >> b) & 1u));
  }
}

}  // namespace f2i
