// Batch decode (1 to 8 tokens) of the widely-linear layer on the fifth-generation
// tensor core with 2:4 structured sparsity ("Fairy2i: Ultra-Low-Bit LLM
// Quantization Using Complex Weights {±1, ±i}", "Industry implications:
// multiplication-free inference"; "Fairy2i-W2" card, y = Ux + W conj(x)).
//
// Formulation.  Every complex code c of a row owns two K slots, (real axis,
// imaginary axis); exactly one of them holds the code's sign, so every two
// codes form a 2:4-sparse group of four slots.  `tcgen05.mma.sp` of
// kind::f8f6f4 takes the signs as compressed e4m3 +-1 values (A, in tensor
// memory) and the axis flags as the sparse metadata (also in tensor memory),
// K = 64 slots = 32 codes per instruction.  B holds, per token, the columns
//   j = 0: Re x on the real slot      j = 1: Im x on the real slot
//   j = 2: Re x on the imaginary slot j = 3: Im x on the imaginary slot
// so D gives per output row the four signed sums
//   sum_real-coded sign Re x, sum_real sign Im x, sum_imag sign Re x,
//   sum_imag sign Im x,
// from which the row and axis scales form the U and W terms (W acting on
// conj(x) only flips signs).  x (bfloat16) is represented exactly by two e4m3
// terms: x 2^s = hi + lo / 16 with a per-token power of two 2^s that puts
// max |x| in [128, 256); hi and lo sit in separate B columns (8 per token).
//
// The 2T code planes of U and W (stages t) are stacked in the 128 TMEM lanes:
// lane = plane * R + row, R = 64 / T (T = 1, 2), 16 (T = 3, 4).  A tile is R
// output rows; one CTA owns a tile over the whole K range, so every output is
// reduced in a fixed order with no cross-CTA step.
//
// The element order of the compressed A row inside one MMA equals the column
// order: from the version-2 sign words of a lane quad, PRMT gathers the bytes
// that hold one half of the steps (a word per two lanes), and a shift by
// 4 (s & 1) + 2 h + rho brings four signs to bits 7, 15, 23, 31; the flag words
// are already in metadata nibble form (bit 0 / bit 2 = the axis flags of the
// two codes of a group).
//
// Roles (19 warps): 0 TMA loads of code chunks (8 lanes), 1 and 18 MMA issue
// (alternate chunks; warp 1 also allocates TMEM), 2-9 expansion of codes into
// A and metadata (two warps per lane quarter, alternate chunks), 10-13
// epilogue, 14-17 construction of B from x (every fourth chunk each).
#pragma once
#include <cuda.h>

#include <cstdint>

#include "layout.cuh"
#include "linear_prefill.cuh"  // PTX wrappers for mbarrier, TMA, TMEM and tcgen05

namespace f2i {

constexpr int kTdMaxGroup = 8;
constexpr int kTdMaxTokens = 8;
constexpr int kTdAStages = 16;  // shared-memory ring of code chunks (4 KB each)
constexpr int kTdTStages = 4;   // stages of A + metadata in TMEM and B in shared memory (one chunk each)
constexpr int kTdThreads = 608;  // 19 warps
constexpr int kTdBuilders = 4;   // B-construction warps (chunk c goes to builder c % 4)
constexpr int kTdLoaders = 8;    // loader lanes (lane l issues chunks l, l + 8, ...)
constexpr int kTdMaxCtas = 160;
constexpr int kTdMaxSched = 6144;
constexpr int kTdMaxLocal = 1024;  // tile entries of one CTA (copied to shared memory)
constexpr uint32_t kTdTmemCols = 512;
constexpr uint32_t kTdAccCol = 256;  // accumulators: 2 buffers x nsub x N columns
constexpr int kTdAStageBytes = 4096;
constexpr int kTdRedBytes = 2 * 128 * kTdMaxTokens * 8;

struct TdProblem {
  const float* scales;
  const uint16_t* x;  // bfloat16 [M][2m]
  float* y;           // [M][2n]
  int32_t n, m, KB, tiles;
};

struct TdParams {
  CUtensorMap cmap[kTdMaxGroup];  // full two-block chunks: 5-D view (u32, g, chunk, row tile, plane)
  CUtensorMap tmap[kTdMaxGroup];  // odd last block: 4-D view (u32, g, row tile, plane)
  TdProblem p[kTdMaxGroup];
  int32_t count, T, R, M;
  int32_t N, nsub, bstage_bytes;
  uint16_t off[kTdMaxCtas + 1];  // schedule of CTA i: sched[off[i] .. off[i + 1])
  uint16_t sched[kTdMaxSched];   // (problem << 13) | tile
};

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, "
      "%7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
      "%6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// D[tmem] (+)= A[tmem] (2:4 sparse, metadata in tmem) * B[smem], e4m3 inputs, fp32 D.
__device__ __forceinline__ void tc_mma_sp_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t meta_tmem,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.sp.cta_group::1.kind::f8f6f4 [%0], [%1], %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(meta_tmem), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// ((x << sh) & 0x80808080) | c: four signs at bits 7, 15, 23, 31 become e4m3
// +-1 (c = 0x38383838 in a register).
__device__ __forceinline__ uint32_t e4m3_signs(uint32_t x, uint32_t sh, uint32_t c) {
  uint32_t r;
  asm("{\n\t.reg .b32 t;\n\t"
      "shl.b32 t, %1, %2;\n\t"
      "lop3.b32 %0, t, 0x80808080, %3, 0xEA;\n\t}"
      : "=r"(r)
      : "r"(x), "r"(sh), "r"(c));
  return r;
}
// (x & 0x55555555) | c: metadata word from a flag word (c = 0x88888888 in a register).
__device__ __forceinline__ uint32_t meta_word(uint32_t x, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x55555555, %2, 0xEA;" : "=r"(r) : "r"(x), "r"(c));
  return r;
}

// Two floats to e4m3 (round to nearest even, saturating): the low byte holds lo.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi_byte, float lo_byte) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi_byte), "f"(lo_byte));
  return r;
}
// e4m3 pair back to two floats (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t v, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t v16 = (uint16_t)v;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v16));
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}

// Bounded wait taken by a whole warp with one outcome for all lanes (every
// lane observes the phase, so each gets the acquire ordering); gives up as
// mbar_wait does.  A warp-uniform outcome keeps the warp-collective tcgen05
// instructions that follow from running with part of the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t limit_ns = 2000000000ull) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, 20000u))) return true;
    if ((i & 15) == 0) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          stop = 1;
        } else if (global_ns() - t0 > limit_ns) {
          *abort_flag = 1;
          f2i_raise(kErrTimeout);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

struct TdSmem {
  uint64_t a_full[kTdAStages], a_empty[kTdAStages];  // code chunks in shared memory
  // Stage ts (chunk c goes to stage c % 4) = TMEM A + metadata columns and a B buffer.
  uint64_t s_full[kTdTStages];   // A + metadata written (4 expander warps) and B built (1 builder warp)
  uint64_t s_empty[kTdTStages];  // the chunk's MMAs are done with the stage (one commit)
  uint64_t acc_full[2], acc_empty[2];
  uint64_t red_full[2];  // the four epilogue warps have written their plane sums of a tile
  uint64_t done[2];
  uint32_t xmax[kTdMaxGroup][kTdMaxTokens];
  float scale[kTdMaxGroup][kTdMaxTokens];  // 2^s
  float inv[kTdMaxGroup][kTdMaxTokens];    // 2^-s (NaN when x has a non-finite entry)
  uint16_t sched[kTdMaxLocal];  // this CTA's tile entries: (problem << 13) | tile
  int32_t kb[kTdMaxGroup];      // column blocks per problem
  uint32_t tmem_base;
  int abort_flag;
};

// Position in the CTA's chunk sequence (tile entry e, chunk c of the tile).
struct TdCursor {
  int e, c;
};
// Chunk counts come from the shared-memory copies of the schedule and of the column-block counts
// (dynamically indexed kernel parameters would go through the constant cache).
__device__ __forceinline__ int td_nch(const uint16_t* sched, const int32_t* kb, int e) {
  return (kb[sched[e] >> 13] + 1) >> 1;
}
__device__ __forceinline__ void td_advance(const uint16_t* sched, const int32_t* kb, TdCursor& cur, int steps,
                                           int t_end) {
  while (steps > 0 && cur.e < t_end) {
    const int left = td_nch(sched, kb, cur.e) - cur.c;
    if (steps < left) {
      cur.c += steps;
      return;
    }
    steps -= left;
    ++cur.e;
    cur.c = 0;
  }
}

__global__ void __launch_bounds__(kTdThreads, 1) linear_tc_decode_kernel(const __grid_constant__ TdParams P) {
  extern __shared__ __align__(1024) uint8_t td_smem_raw[];
  uint8_t* base = td_smem_raw + ((1024 - (smem_u32(td_smem_raw) & 1023)) & 1023);
  uint8_t* a_ring = base;                                      // kTdAStages x 4 KB
  uint8_t* b_ring = a_ring + kTdAStages * kTdAStageBytes;      // kTdTStages x bstage_bytes
  float2* red = reinterpret_cast<float2*>(b_ring + kTdTStages * P.bstage_bytes);  // [2][128][8]
  TdSmem& S = *reinterpret_cast<TdSmem*>(reinterpret_cast<uint8_t*>(red) + kTdRedBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int t_begin = 0, t_end = P.off[cta + 1] - P.off[cta];  // local tile entries in S.sched
  const int T = P.T, R = P.R, M = P.M, N = P.N, nsub = P.nsub;
  volatile int* abort_flag = &S.abort_flag;

  // ---- setup: barriers, TMEM, per-token scales of x ----
  if (tid < kTdMaxGroup * kTdMaxTokens) (&S.xmax[0][0])[tid] = 0u;
  for (int i = tid; i < t_end; i += kTdThreads) S.sched[i] = P.sched[P.off[cta] + i];
  if (tid < kTdMaxGroup) S.kb[tid] = tid < P.count ? P.p[tid].KB : 0;
  if (tid == 0) {
    S.abort_flag = 0;
    for (int i = 0; i < kTdAStages; ++i) {
      mbar_init(smem_u32(&S.a_full[i]), 1);
      mbar_init(smem_u32(&S.a_empty[i]), 4);
    }
    for (int i = 0; i < kTdTStages; ++i) {
      mbar_init(smem_u32(&S.s_full[i]), 5);
      mbar_init(smem_u32(&S.s_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.acc_full[i]), 2);
      mbar_init(smem_u32(&S.acc_empty[i]), 4);
      mbar_init(smem_u32(&S.red_full[i]), 4);
      mbar_init(smem_u32(&S.done[i]), 1);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane < P.count) {
    tma_prefetch_map(&P.cmap[lane]);
    tma_prefetch_map(&P.tmap[lane]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTdTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  // max |x| per (problem, token) over the problems this CTA touches: bfloat16
  // magnitudes compare as integers (v & 0x7fff), NaN above every finite value.
  {
    uint32_t used = 0;
    for (int e = t_begin; e < t_end; ++e) used |= 1u << (S.sched[e] >> 13);
    for (int i = 0; i < P.count; ++i) {
      if (!((used >> i) & 1u)) continue;
      const TdProblem& pr = P.p[i];
      const int64_t row = 2 * (int64_t)pr.m;
      for (int t = 0; t < M; ++t) {
        const uint16_t* xr = pr.x + t * row;
        uint32_t mx = 0;
        if ((pr.m & 7) == 0) {
          const uint4* x4 = reinterpret_cast<const uint4*>(xr);
          const int64_t nv = row / 8;
          for (int64_t k0 = tid; k0 < nv; k0 += 4 * kTdThreads) {  // four loads in flight per thread
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int64_t k = k0 + (int64_t)u * kTdThreads;
              v[u] = k < nv ? __ldg(x4 + k) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              mx = __vmaxu2(mx, v[u].x & 0x7fff7fffu);
              mx = __vmaxu2(mx, v[u].y & 0x7fff7fffu);
              mx = __vmaxu2(mx, v[u].z & 0x7fff7fffu);
              mx = __vmaxu2(mx, v[u].w & 0x7fff7fffu);
            }
          }
        } else {
          for (int64_t k = tid; k < row; k += kTdThreads) mx = max(mx, (uint32_t)(__ldg(xr + k) & 0x7fffu));
        }
        mx = max(mx & 0xffffu, mx >> 16);
        for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(&S.xmax[i][t], mx);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid < kTdMaxGroup * kTdMaxTokens) {
    const uint32_t mx = (&S.xmax[0][0])[tid];
    int s = 0;
    if (mx >= 0x80u && mx < 0x7f80u) s = 7 - ((int)(mx >> 7) - 127);  // max |x| 2^s in [128, 256)
    else if (mx > 0u && mx < 0x80u) s = 126;                           // subnormal bfloat16 only
    s = max(-120, min(126, s));
    (&S.scale[0][0])[tid] = __int_as_float((s + 127) << 23);
    (&S.inv[0][0])[tid] = mx >= 0x7f80u ? __int_as_float(0x7fc00000) : __int_as_float((127 - s) << 23);
  }
  __syncthreads();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ---- TMA producer: one code chunk (2T planes x R rows x 128 columns) per stage; loader lane l
    // takes chunks l, l + 8, ... ----
    if (lane < kTdLoaders) {
      const int Rt = R >> 4;
      const uint32_t full_bytes = 512u * Rt * 2 * T, tail_bytes = 256u * Rt * 2 * T;
      TdCursor cur{t_begin, 0};
      td_advance(S.sched, S.kb, cur, lane, t_end);
      for (uint32_t chunk = lane; cur.e < t_end; chunk += kTdLoaders) {
        if (*abort_flag) break;
        const int pi = S.sched[cur.e] >> 13, tile = S.sched[cur.e] & 8191;
        const int full = S.kb[pi] >> 1;
        const uint32_t s = chunk % kTdAStages;
        if (!mbar_wait(smem_u32(&S.a_empty[s]), ((chunk / kTdAStages) & 1) ^ 1, abort_flag)) break;
        const uint32_t bar = smem_u32(&S.a_full[s]);
        const uint32_t dst = smem_u32(a_ring + s * kTdAStageBytes);
        if (cur.c < full) {
          mbar_arrive_expect_tx(bar, full_bytes);
          tma_load_5d(dst, &P.cmap[pi], bar, 0, 0, cur.c, tile * Rt, 0);
        } else {
          mbar_arrive_expect_tx(bar, tail_bytes);
          tma_load_4d(dst, &P.tmap[pi], bar, 0, 0, tile * Rt, 0);
        }
        td_advance(S.sched, S.kb, cur, kTdLoaders, t_end);
      }
    }
  } else if (warp == 1 || warp == 18) {
    // ---- MMA issue: two issuing threads take alternate chunks, each accumulating into its own
    // sub-accumulators (a thread's barrier wait lets its own MMAs drain; the other thread's MMAs keep
    // the tensor core busy meanwhile).  Issuer q uses subs 2q, 2q + 1 (nsub = 4) or q (nsub = 2). ----
    const int q = warp == 1 ? 0 : 1;
    if (lane == 0) {
      const uint32_t idesc = (1u << 2) | (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((128u >> 4) << 24);
      const uint64_t bdesc_hi = ((uint64_t)((uint32_t)N) << 16) | ((uint64_t)(128u >> 4) << 32) | ((uint64_t)1 << 46);
      const uint32_t kstep_b16 = (uint32_t)N * 4u;  // 64 N bytes >> 4
      const uint32_t bstage16 = (uint32_t)P.bstage_bytes >> 4;
      const uint32_t bring16 = (smem_u32(b_ring) & 0x3FFFFu) >> 4;
      const uint32_t sub_a = nsub == 4 ? (uint32_t)(2 * q * N) : (uint32_t)(q * N);
      const uint32_t sub_b = nsub == 4 ? sub_a + (uint32_t)N : sub_a;
      uint32_t chunk = 0;
      int tl = 0;
      bool ok = true;
      for (int e = t_begin; e < t_end && ok; ++e, ++tl) {
        const int pi = S.sched[e] >> 13;
        const int KB = S.kb[pi], full = KB >> 1, nch = (KB + 1) >> 1;
        const int abuf = tl & 1;
        if (!mbar_wait(smem_u32(&S.acc_empty[abuf]), ((tl >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t acc = tmem + kTdAccCol + (uint32_t)(abuf * nsub * N);
        const uint32_t d0 = acc + sub_a, d1 = acc + sub_b;
        uint32_t acc_flag = 0;
        for (int c = 0; c < nch; ++c, ++chunk) {
          if ((int)(chunk & 1) != q) continue;
          const uint32_t ts = chunk % kTdTStages;
          if (!mbar_wait(smem_u32(&S.s_full[ts]), (chunk / kTdTStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_col = tmem + 32u * ts, m_col = tmem + 128u + 8u * ts;
          const uint64_t bd = bdesc_hi | (uint64_t)(bring16 + ts * bstage16);
          tc_mma_sp_f8(d0, a_col, bd, m_col, idesc, acc_flag);
          tc_mma_sp_f8(d1, a_col + 8u, bd + kstep_b16, m_col + 2u, idesc, nsub == 4 ? acc_flag : 1u);
          if (c < full) {
            tc_mma_sp_f8(d0, a_col + 16u, bd + 2u * kstep_b16, m_col + 4u, idesc, 1u);
            tc_mma_sp_f8(d1, a_col + 24u, bd + 3u * kstep_b16, m_col + 6u, idesc, 1u);
          }
          acc_flag = 1u;
          tc_commit(smem_u32(&S.s_empty[ts]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&S.acc_full[abuf]));
      }
      tc_commit(smem_u32(&S.done[q]));
      mbar_wait(smem_u32(&S.done[q]), 0, abort_flag);
    }
  } else if (warp < 10) {
    // ---- expansion: codes of one lane quad -> e4m3 signs (A) + metadata in TMEM ----
    const int par = (warp - 2) >> 2;
    const int lq = warp & 3;  // TMEM lane quarter of this warp
    const int l = lq * 32 + lane;
    const int p = l / R, r = l % R;
    const bool valid = p < 2 * T;
    const int rt_l = r >> 4, rho = (r >> 3) & 1, g = r & 7;
    const int flat = (p * (R >> 4) + rt_l) * 8 + g;  // 64-byte row of this lane quad in a chunk stage
    const uint32_t sw = (uint32_t)((g >> 1) & 3);
    const uint32_t sh0 = (uint32_t)rho, sh1 = 2u + rho, sh2 = 4u + rho, sh3 = 6u + rho;
    const uint32_t selr = rho ? 0x7632u : 0x5410u;
    const uint32_t c38 = 0x38383838u, c88 = 0x88888888u;
    const uint32_t lane_addr = tmem + ((uint32_t)(lq * 32) << 16);
    uint32_t chunk = 0;
    bool ok = true;
    for (int e = t_begin; e < t_end && ok; ++e) {
      const int pi = S.sched[e] >> 13;
      const int KB = S.kb[pi], full = KB >> 1, nch = (KB + 1) >> 1;
      for (int c = 0; c < nch; ++c, ++chunk) {
        if ((int)(chunk & 1) != par) continue;
        const uint32_t s = chunk % kTdAStages, ts = chunk % kTdTStages;
        if (!mbar_wait_warp(smem_u32(&S.a_full[s]), (chunk / kTdAStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        uint32_t Sw[2][4], Fw[2][4];
        const bool isfull = c < full;
        if (valid && isfull) {
          const uint8_t* st = a_ring + s * kTdAStageBytes + flat * 64;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + (((uint32_t)qq ^ sw) << 4));
            Sw[0][qq] = v.x;
            Fw[0][qq] = v.y;
            Sw[1][qq] = v.z;
            Fw[1][qq] = v.w;
          }
        } else if (valid) {
          const uint8_t* st = a_ring + s * kTdAStageBytes + flat * 32;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint2 v = *reinterpret_cast<const uint2*>(st + qq * 8);
            Sw[0][qq] = v.x;
            Fw[0][qq] = v.y;
            Sw[1][qq] = 0u;
            Fw[1][qq] = 0u;
          }
        } else {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) Sw[0][qq] = Fw[0][qq] = Sw[1][qq] = Fw[1][qq] = 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.a_empty[s]));
        if (!mbar_wait_warp(smem_u32(&S.s_empty[ts]), ((chunk / kTdTStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t a[32], mt[8];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t P1a = prmt(Sw[b][0], Sw[b][1], 0x7531u), P1b = prmt(Sw[b][2], Sw[b][3], 0x7531u);
          const uint32_t P2a = prmt(Sw[b][0], Sw[b][1], 0x6420u), P2b = prmt(Sw[b][2], Sw[b][3], 0x6420u);
          const uint32_t Q0 = prmt(Fw[b][0], Fw[b][1], selr), Q1 = prmt(Fw[b][2], Fw[b][3], selr);
#pragma unroll
          for (int kap = 0; kap < 2; ++kap) {
            const uint32_t xa = kap ? P2a : P1a, xb = kap ? P2b : P1b, Q = kap ? Q1 : Q0;
            const int ks = 2 * b + kap;
            a[8 * ks + 0] = e4m3_signs(xa, sh0, c38);  // w = 0, h = 0
            a[8 * ks + 1] = e4m3_signs(xb, sh0, c38);
            a[8 * ks + 2] = e4m3_signs(xa, sh1, c38);  // w = 0, h = 1
            a[8 * ks + 3] = e4m3_signs(xb, sh1, c38);
            a[8 * ks + 4] = e4m3_signs(xa, sh2, c38);  // w = 1, h = 0
            a[8 * ks + 5] = e4m3_signs(xb, sh2, c38);
            a[8 * ks + 6] = e4m3_signs(xa, sh3, c38);  // w = 1, h = 1
            a[8 * ks + 7] = e4m3_signs(xb, sh3, c38);
            mt[2 * ks] = meta_word(Q, c88);
            mt[2 * ks + 1] = meta_word(Q >> 1, c88);
          }
        }
        tmem_st32(lane_addr + 32u * ts, a);
        tmem_st8(lane_addr + 128u + 8u * ts, mt);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.s_full[ts]));
      }
    }
  } else if (warp < 14) {
    // ---- epilogue: scales, U/W combination, fixed-order sum over planes ----
    const int lq = warp & 3;
    const int l = lq * 32 + lane;
    const int p = l / R, r = l % R;
    const bool valid = p < 2 * T;
    const int X = valid ? p / T : 0, ts_ = valid ? p % T : 0;
    const uint32_t lane_addr = tmem + ((uint32_t)(lq * 32) << 16);
    const int et = tid - 320;  // 0..127
    int tl = 0;
    uint32_t chunk0 = 0;  // first chunk of the tile in the CTA's sequence
    for (int e = t_begin; e < t_end; ++e, ++tl) {
      const int pi = S.sched[e] >> 13, tile = S.sched[e] & 8191;
      const TdProblem& pr = P.p[pi];
      const int nch = (pr.KB + 1) >> 1;
      // Sub-accumulators written in this tile: issuer q took a chunk iff the tile has two chunks or
      // its one chunk has parity q.
      const bool q0 = nch >= 2 || (chunk0 & 1) == 0, q1 = nch >= 2 || (chunk0 & 1) == 1;
      chunk0 += (uint32_t)nch;
      const int row = tile * R + r;
      float s_re = 0.f, s_im = 0.f;
      if (valid && row < pr.n) {
        const int64_t base = ((int64_t)(X * T + ts_) * 2) * pr.n + row;
        s_re = __ldg(pr.scales + base);
        s_im = __ldg(pr.scales + base + pr.n);
      }
      const int abuf = tl & 1;
      if (!mbar_wait_warp(smem_u32(&S.acc_full[abuf]), (tl >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      float2* rb = red + (size_t)abuf * 128 * kTdMaxTokens + (size_t)l * kTdMaxTokens;
      const uint32_t acc0 = lane_addr + kTdAccCol + (uint32_t)(abuf * nsub * N);
      for (int sl = 0; sl < N / 16; ++sl) {
        float d[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = 0.f;
        for (int sb = 0; sb < nsub; ++sb) {
          const bool written = (nsub == 4 ? (sb < 2 ? q0 : q1) : (sb == 0 ? q0 : q1));
          if (!written) continue;
          uint32_t v[16];
          tmem_ld16(acc0 + (uint32_t)(sb * N + sl * 16), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) d[j] += __uint_as_float(v[j]);
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int t = sl * 2 + tt;
          if (t < M) {
            const float iv = S.inv[pi][t];
            const float v0 = fmaf(d[8 * tt + 4], 0.0625f, d[8 * tt + 0]) * iv;
            const float v1 = fmaf(d[8 * tt + 5], 0.0625f, d[8 * tt + 1]) * iv;
            const float v2 = fmaf(d[8 * tt + 6], 0.0625f, d[8 * tt + 2]) * iv;
            const float v3 = fmaf(d[8 * tt + 7], 0.0625f, d[8 * tt + 3]) * iv;
            float re, im;
            if (X == 0) {
              re = s_re * v0 - s_im * v3;
              im = s_re * v1 + s_im * v2;
            } else {
              re = s_re * v0 + s_im * v3;
              im = s_im * v2 - s_re * v1;
            }
            rb[t] = make_float2(re, im);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&S.acc_empty[abuf]));
        mbar_arrive(smem_u32(&S.red_full[abuf]));
      }
      if (!mbar_wait_warp(smem_u32(&S.red_full[abuf]), (tl >> 1) & 1, abort_flag)) break;
      const float2* rbuf = red + (size_t)abuf * 128 * kTdMaxTokens;
      for (int idx = et; idx < R * M; idx += 128) {
        const int rr = idx % R, t = idx / R;
        const int orow = tile * R + rr;
        if (orow >= pr.n) continue;
        float re = 0.f, im = 0.f;
        for (int pp = 0; pp < 2 * T; ++pp) {
          const float2 v = rbuf[(size_t)(pp * R + rr) * kTdMaxTokens + t];
          re += v.x;
          im += v.y;
        }
        float* yr = pr.y + (int64_t)t * 2 * pr.n;
        yr[orow] = re;
        yr[pr.n + orow] = im;
      }
    }
  } else if (warp < 14 + kTdBuilders) {
    // ---- B construction: x (bfloat16) -> hi/lo e4m3 columns, one chunk of 128 columns per stage.
    // Lane task: 4 consecutive columns of one token. ----
    const int par = warp - 14;
    uint32_t chunk = 0;
    bool ok = true;
    for (int e = t_begin; e < t_end && ok; ++e) {
      const int pi = S.sched[e] >> 13;
      const TdProblem& pr = P.p[pi];
      const int nch = (pr.KB + 1) >> 1;
      const bool vec = (pr.m & 3) == 0;
      for (int c = 0; c < nch; ++c, ++chunk) {
        if ((int)(chunk % kTdBuilders) != par) continue;
        const uint32_t ts = chunk % kTdTStages;
        if (!mbar_wait_warp(smem_u32(&S.s_empty[ts]), ((chunk / kTdTStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* bst = b_ring + ts * P.bstage_bytes;
        for (int t = 0; t < M; ++t) {
          const int col0 = c * 128 + lane * 4;
          const uint16_t* xr = pr.x + (int64_t)t * 2 * pr.m;
          uint2 rv, iv;
          if (vec && col0 + 4 <= pr.m) {
            rv = __ldg(reinterpret_cast<const uint2*>(xr + col0));
            iv = __ldg(reinterpret_cast<const uint2*>(xr + pr.m + col0));
          } else {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int cc = col0 + k;
              w[k] = cc < pr.m ? (uint32_t)__ldg(xr + cc) | ((uint32_t)__ldg(xr + pr.m + cc) << 16) : 0u;
            }
            rv = make_uint2((w[0] & 0xffffu) | (w[1] << 16), (w[2] & 0xffffu) | (w[3] << 16));
            iv = make_uint2((w[0] >> 16) | (w[1] & 0xffff0000u), (w[2] >> 16) | (w[3] & 0xffff0000u));
          }
          const float sc = S.scale[pi][t];
          uint32_t wh[2], wl[2];  // bytes [re(2k), im(2k), re(2k+1), im(2k+1)] of hi and of lo
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const uint32_t re2 = k2 ? rv.y : rv.x, im2 = k2 ? iv.y : iv.x;
            uint32_t h[2], lo[2];
#pragma unroll
            for (int o = 0; o < 2; ++o) {
              const float fr = __uint_as_float(o ? (re2 & 0xffff0000u) : (re2 << 16)) * sc;
              const float fi = __uint_as_float(o ? (im2 & 0xffff0000u) : (im2 << 16)) * sc;
              h[o] = cvt_e4m3x2(fi, fr);
              float hr, hi;
              e4m3x2_to_f32(h[o], hr, hi);
              lo[o] = cvt_e4m3x2((fi - hi) * 16.f, (fr - hr) * 16.f);
            }
            wh[k2] = h[0] | (h[1] << 16);
            wl[k2] = lo[0] | (lo[1] << 16);
          }
          // 4 columns = half a 16-byte core-matrix row: K-step lane / 8, core column (lane / 2) % 4,
          // byte offset 8 (lane % 2); rows 8t + 4 hl + j.
          uint8_t* dst = bst + (lane >> 3) * (N * 64) + ((lane >> 1) & 3) * (N * 16) + t * 128 + (lane & 1) * 8;
#pragma unroll
          for (int hl = 0; hl < 2; ++hl) {
            const uint32_t* w = hl ? wl : wh;
            uint2* d2 = reinterpret_cast<uint2*>(dst + hl * 64);
            d2[0] = make_uint2(w[0] & 0x00ff00ffu, w[1] & 0x00ff00ffu);
            d2[2] = make_uint2((w[0] >> 8) & 0x00ff00ffu, (w[1] >> 8) & 0x00ff00ffu);
            d2[4] = make_uint2((w[0] << 8) & 0xff00ff00u, (w[1] << 8) & 0xff00ff00u);
            d2[6] = make_uint2(w[0] & 0xff00ff00u, w[1] & 0xff00ff00u);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.s_full[ts]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTdTmemCols);
  }
}

}  // namespace f2i
