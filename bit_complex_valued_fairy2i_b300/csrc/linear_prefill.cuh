// Layer evaluation for large token counts (prefill) on the 5th-generation
// tensor cores: tcgen05.mma with TMEM accumulators, TMA-staged activations.
//
// The multiplication-free sum ("Fairy2i: Ultra-Low-Bit LLM Quantization Using
// Complex Weights {±1, ±i}", "Industry implications: multiplication-free
// inference": B_re, B_im in {-1, 0, 1}) is, over many tokens, a dense ternary
// contraction.  Per output row j and code plane (X, t) there are two ternary
// rows, re-row and im-row (disjoint supports), and per token four dot products
// <re-row, a>, <re-row, b>, <im-row, a>, <im-row, b> (a = Re x, b = Im x).
// They are combined with the plane's scales exactly as in the decode path:
//   U plane: Re y += s_re <re, a> - s_im <im, b>,  Im y += s_re <re, b> + s_im <im, a>
//   W plane: Re y += s_re <re, a> + s_im <im, b>,  Im y += -s_re <re, b> + s_im <im, a>
//
// GEMM shape per tile:  D[128 code rows][256] += A[128][K] * B[256][K]^T
//   A: code rows (output jj, plane p, axis a) at row RO*jj + 2p + a, entries
//      bfloat16 {+2, -2, +0, -0} expanded from the packed codes by the
//      producer warps (128-byte swizzled, K-major).  The codes reach shared
//      memory by the TMA engine: per window of 4 column-block pairs, one bulk
//      copy (cp.async.bulk) per (16-row tile, plane) of the tile's contiguous
//      layout-2 run, into a ring of two stages, a window ahead of their use.
//   B: the activations viewed as [2M][m] (row 2*token + part), which is the
//      caller's x [M][2m] unchanged; loaded by TMA, 128-byte swizzled.
//   D: fp32 in TMEM, two accumulators of 256 columns (double buffered).
// Every product is exact (+-2 times a bfloat16); only the fp32 accumulation
// rounds.  The factor 2 is removed with the scale (exact).
//
// Warp roles (15 warps, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer for B
//   warp 1      TMEM allocation; one thread issues tcgen05.mma / commit
//   warps 2-9   A producers: codes -> swizzled bfloat16 tiles (two groups of
//               four warps, alternate k-blocks)
//   warps 10-13 epilogue: tcgen05.ld, scales, reduction over the RO code
//               rows of each output (lane shuffles), stores y
//   warp 14     bulk copies of the codes
// All mbarrier waits are bounded (about 2 s); a wait that gives up raises the
// timeout flag of the device error word and every role winds down.
#pragma once
#include <cuda.h>
#include <cstdint>
#include "layout.cuh"

namespace f2i {

constexpr int kPfMaxGroup = 8;
constexpr int kPfStages = 4;
constexpr int kPfBM = 128;  // code rows per tile (MMA M)
constexpr int kPfBN = 256;  // activation rows per tile = 128 tokens x (a, b) (MMA N)
constexpr int kPfBK = 64;   // columns per k-block: one 128-byte swizzle row of bfloat16
constexpr int kPfTokens = kPfBN / 2;
constexpr int kPfAStage = kPfBM * kPfBK * 2;  // 16 KB
constexpr int kPfBStage = kPfBN * kPfBK * 2;  // 32 KB
constexpr int kPfProducerWarps = 8;
constexpr int kPfProducerGroups = 2;  // groups fill alternate k-blocks concurrently
constexpr int kPfGroupWarps = kPfProducerWarps / kPfProducerGroups;
constexpr int kPfThreads = 32 * (7 + kPfProducerWarps);
constexpr uint32_t kPfTmemCols = 512;  // two 256-column fp32 accumulators
// Code ring: two stages of a window of kPfWinPairs column-block pairs for
// every (16-row tile, plane) of a tile: 2 x 2 planes (T = 1, two row tiles),
// 4 (T = 2) or at most 8 (T = 3, 4) runs of 4 x 512 bytes.
constexpr int kPfCStages = 2;
constexpr int kPfWinPairs = 4;
constexpr uint32_t kPfCStage = 8u * kPfWinPairs * 512u + 128u;
// Run idx (= 16-row tile x 2T + plane) of a code stage starts 16 (idx & 7)
// bytes past its slot, so that the quads' 16-byte words of different planes
// fall in different bank groups.
__host__ __device__ __forceinline__ uint32_t pf_run_off(int idx) {
  return (uint32_t)idx * (kPfWinPairs * 512u) + 16u * (uint32_t)(idx & 7);
}
constexpr size_t kPfSmemBytes = 1024 /* alignment slack */ + (size_t)kPfStages * (kPfAStage + kPfBStage) +
                                (size_t)kPfCStages * kPfCStage + 256 /* barriers, TMEM address */;

struct PrefillProblem {
  const uint8_t* codes;
  const float* scales;
  float* y;
  int64_t n, m;
  int64_t tile_begin;  // first tile index of this problem within the launch
  int64_t row_tiles;
  int32_t tok_tiles, kblocks;
};

struct PrefillParams {
  CUtensorMap tmap[kPfMaxGroup];  // x of each problem as a [2M][m] bfloat16 tensor
  PrefillProblem p[kPfMaxGroup];
  int64_t total_tiles;
  int32_t count, T, M, pad_;
};

// ---- PTX wrappers -----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As above, but the thread may be suspended for up to `ns` nanoseconds while
// the phase is incomplete (it resumes as soon as the phase completes), so
// waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `parity` to complete.  Gives up after `limit_ns`
// (about 2 s by default), or soon after another role of the CTA has given up
// (`abort_flag`); then the device error word gets the timeout flag and false
// is returned.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        f2i_raise(kErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Bulk copy (no tensor map) of `bytes` from global to this CTA's shared
// memory, completing on mbarrier `bar` (16-byte aligned ends, multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bfloat16 inputs, fp32 accumulation.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// (x & m) | 0x40004000 in one LOP3 (m held in a register): the signs at bits
// 15 and 31 become bfloat16 +-2.
__device__ __forceinline__ uint32_t sign_operand_pf(uint32_t x, uint32_t m) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, 0x40004000, 0xEA;" : "=r"(r) : "r"(x), "r"(m));
  return r;
}

// (x & m) | f in one LOP3 (m = 0x80008000 held in a register; f has bits at
// 14 and 30 only): the signs of x at 15 and 31 and the flags of f form
// bfloat16 {+-2, +-0}.
__device__ __forceinline__ uint32_t real_operand_pf(uint32_t x, uint32_t m, uint32_t f) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(m), "r"(f));  // (x & m) | f
  return r;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 1024-byte groups of eight (stride byte offset 1024).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1 << 46;            // descriptor version of the sm_100 family
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 D, bfloat16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with fp16 A and B (type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- tile bookkeeping ----------------------------------------------------

struct PfTile {
  int pi;
  int64_t rt;
  int tt;
};
__device__ __forceinline__ PfTile pf_tile(const PrefillParams& P, int64_t tile) {
  int pi = 0;
  for (int i = 1; i < P.count; ++i)
    if (tile >= P.p[i].tile_begin) pi = i;
  const int64_t local = tile - P.p[pi].tile_begin;
  PfTile c;
  c.pi = pi;
  c.rt = local / P.p[pi].tok_tiles;
  c.tt = (int)(local - c.rt * P.p[pi].tok_tiles);
  return c;
}

// First 16-row layout-2 tile of tile rt, J outputs per tile (J = 32: two row
// tiles; 16: one; 8: half of one).
template <int J>
__host__ __device__ __forceinline__ int64_t pf_first_row_tile(int64_t rt) {
  return J >= 16 ? rt * (J / 16) : rt / (16 / J);
}

// ---- the kernel -------------------------------------------------------------

// RO = code rows per output: 4T rounded up to a power of two (4, 8, 16).
template <int RO>
__global__ void __launch_bounds__(kPfThreads, 1) linear_tcgen05_kernel(const __grid_constant__ PrefillParams P) {
  extern __shared__ uint8_t pf_smem_raw[];
  constexpr int J = kPfBM / RO;  // outputs per tile
  constexpr uint32_t kIdesc = idesc_bf16(kPfBM, kPfBN);

  const uint32_t raw = smem_u32(pf_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = pf_smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + kPfStages * kPfAStage;
  const uint32_t sC = sB + kPfStages * kPfBStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kPfStages * (kPfAStage + kPfBStage) + kPfCStages * kPfCStage);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(kPfStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kPfStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kPfStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (uint32_t)(2 * kPfStages + 4);  // every issued MMA complete
  auto fullC = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kPfStages + 5 + s); };
  auto emptyC = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kPfStages + 5 + kPfCStages + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPfStages + 5 + 2 * kPfCStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = P.T;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(full_bar(s), 1 + kPfGroupWarps);  // TMA arrive.expect_tx + one arrive per warp of the producing group
      mbar_init(empty_bar(s), 1); // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);  // tcgen05.commit
      mbar_init(acce_bar(b), 4);  // one arrive per epilogue warp
    }
    mbar_init(done_bar, 1);  // tcgen05.commit after the last MMA
    for (int s = 0; s < kPfCStages; ++s) {
      mbar_init(fullC(s), 1);                 // the code warp's arrive.expect_tx
      mbar_init(emptyC(s), kPfProducerWarps);  // one arrive per producer warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < P.count; ++i) tma_prefetch_map(&P.tmap[i]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kPfTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2 && warp < 2 + kPfProducerWarps) {
    // zero every A stage once: code rows that no output uses (T = 3) stay zero
    const int i = tid - 64;
    for (uint32_t off = (uint32_t)i * 16u; off < (uint32_t)(kPfStages * kPfAStage); off += 32u * kPfProducerWarps * 16u)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sA + off), "r"(0u) : "memory");
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer: activations ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
        const PfTile c = pf_tile(P, tile);
        const int kbs = P.p[c.pi].kblocks;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int s = (int)(it % kPfStages);
          const uint32_t ph = (it / kPfStages) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), (uint32_t)kPfBStage);
          tma_load_2d(sB + (uint32_t)s * kPfBStage, &P.tmap[c.pi], full_bar(s), kb * kPfBK, c.tt * kPfBN);
        }
      }
      // let copies still in flight land before the CTA can exit
      for (uint32_t k = (it > (uint32_t)kPfStages ? it - kPfStages : 0u); k < it; ++k)
        if (!mbar_wait(full_bar((int)(k % kPfStages)), (k / kPfStages) & 1u, abort_flag)) break;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x, ++lt) {
        const PfTile c = pf_tile(P, tile);
        const int kbs = P.p[c.pi].kblocks;
        const int b = (int)(lt & 1u);
        if (!mbar_wait(acce_bar(b), ((lt >> 1) & 1u) ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)b * kPfBN;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int s = (int)(it % kPfStages);
          const uint32_t ph = (it / kPfStages) & 1u;
          if (!mbar_wait(full_bar(s), ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + (uint32_t)s * kPfAStage, b0 = sB + (uint32_t)s * kPfBStage;
#pragma unroll
          for (int kk = 0; kk < kPfBK / 16; ++kk)
            tc_mma_bf16(d_tmem, sw128_desc(a0 + 32u * kk), sw128_desc(b0 + 32u * kk), kIdesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit(empty_bar(s));
        }
        if (ok) tc_commit(accf_bar(b));
      }
      // every issued MMA completes before the tensor memory is freed, also when
      // a wait gave up (then the epilogue may not have waited for them)
      tc_commit(done_bar);
      volatile int drain_flag = 0;
      mbar_wait(done_bar, 0, &drain_flag, 100000000ull);
    }
  } else if (warp < 2 + kPfProducerWarps) {
    // ---------------- A producers: codes -> bfloat16 {+-2, +-0} ----------------
    // Two groups of four warps fill alternate k-blocks, so two stages are
    // being expanded at any time.  Inside a group, thread (i, hf) owns code
    // plane p of output jj of every tile, steps 2 hf and 2 hf + 1: rows
    // RO*jj + 2p (real axis) and RO*jj + 2p + 1 (imaginary axis), chunks
    // 4 hf .. 4 hf + 3.  A 16-byte chunk is 8 columns 16 s + 8 h + 2 q' + e
    // (q' = 0..3): the signs come from the sign words of the four lanes
    // (g, q') of the output's lane quad, the axis flags from the flag word of
    // lane (g, h + 2 (s >> 1)).  The quad's words of two blocks are 64
    // contiguous bytes of the code stage; the next pair of blocks (of this
    // tile or the next) is read while the current one is expanded.
    const int gt = tid - 64;
    const int grp = gt / (32 * kPfGroupWarps);
    const int lt = gt - grp * 32 * kPfGroupWarps;
    const int pi = lt >> 1, hf = lt & 1;
    const int planes = 2 * T;
    const bool active = pi < J * planes;
    const int jj = active ? pi / planes : 0;
    const int p = active ? pi - jj * planes : 0;
    const uint32_t r_re = (uint32_t)(RO * jj + 2 * p);
    const uint32_t row_re = r_re * 128u, row_im = (r_re + 1u) * 128u;
    const uint32_t sw_re = r_re & 7u, sw_im = (r_re + 1u) & 7u;
    const uint32_t smask = 0x80008000u + (uint32_t)(P.M >> 30);  // register-held mask (M < 2^30)

    // loader cursor: tile, pair, and the code windows before the tile's first
    uint32_t ld_wc = 0;
    int64_t ld_tile = blockIdx.x;
    int64_t ld_c2 = 0;
    int64_t ld_fullc = 0, ld_pairs = 0;
    bool ld_live = false;  // this thread has a row of the tile (else it expands zeros)
    uint32_t ld_run = 0;   // its (row tile, plane) run in a code stage
    int ld_g = 0;
    auto set_ld_tile = [&]() {
      ld_live = false;
      if (ld_tile >= P.total_tiles) return;
      const PfTile c = pf_tile(P, ld_tile);
      const PrefillProblem& pr = P.p[c.pi];
      const int64_t KB = col_blocks(pr.m);
      ld_fullc = KB >> 1;
      ld_pairs = (KB + 1) >> 1;
      const int64_t j = c.rt * J + jj;
      const int rtl = (int)((j >> 4) - pf_first_row_tile<J>(c.rt));
      ld_run = pf_run_off(rtl * planes + p);
      ld_g = (int)(j & 7);
      ld_live = active && j < pr.n;
    };
    // the quad's words of the cursor's pair from its window's code stage
    // (false: a wait gave up)
    uint4 nxt[4];
    auto load_pair = [&](uint4 (&dst)[4]) -> bool {
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
      if (ld_tile >= P.total_tiles) return true;
      const uint32_t k = ld_wc + (uint32_t)(ld_c2 / kPfWinPairs);
      const int cs = (int)(k % kPfCStages);
      // one wait per window (its copies complete one phase of the barrier)
      if (ld_c2 % kPfWinPairs == 0 &&
          __any_sync(0xffffffffu, !mbar_wait(fullC(cs), (k / kPfCStages) & 1u, abort_flag) ? 1 : 0))
        return false;
      if (!ld_live) return true;
      const uint32_t cb = sC + (uint32_t)cs * kPfCStage + ld_run + (uint32_t)(ld_c2 % kPfWinPairs) * 512u;
      if (ld_c2 < ld_fullc) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(dst[q].x), "=r"(dst[q].y), "=r"(dst[q].z), "=r"(dst[q].w)
                       : "r"(cb + (uint32_t)(4 * ld_g + q) * 16u)
                       : "memory");
      } else {  // an odd last block: 8 bytes a lane
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                       : "=r"(dst[q].x), "=r"(dst[q].y)
                       : "r"(cb + (uint32_t)(4 * ld_g + q) * 8u)
                       : "memory");
      }
      return true;
    };
    // past the pair just read: its window's stage goes back to the code warp
    // after the window's last pair
    auto advance = [&]() {
      if (ld_tile >= P.total_tiles) return;
      if ((ld_c2 + 1) % kPfWinPairs == 0 || ld_c2 + 1 == ld_pairs) {
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyC((int)((ld_wc + (uint32_t)(ld_c2 / kPfWinPairs)) % kPfCStages)));
      }
      if (++ld_c2 == ld_pairs) {
        ld_wc += (uint32_t)((ld_pairs + kPfWinPairs - 1) / kPfWinPairs);
        ld_c2 = 0;
        ld_tile += gridDim.x;
        set_ld_tile();
      }
    };
    set_ld_tile();
    bool ld_ok = load_pair(nxt);
    advance();

    uint32_t it = 0;
    bool ok = ld_ok;
    for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
      const PfTile c = pf_tile(P, tile);
      const PrefillProblem& pr = P.p[c.pi];
      const int64_t j = c.rt * J + jj;
      const bool live = active && j < pr.n;
      const int rho = (int)((j >> 3) & 1);
      for (int kb0 = 0; ok && kb0 < pr.kblocks; kb0 += 2) {
        uint4 cur[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
        if (!load_pair(nxt)) {
          ok = false;
          break;
        }
        advance();
        const int nb = min(2, pr.kblocks - kb0);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (b >= nb) break;
          const int s = (int)(it % kPfStages);
          const uint32_t ph = (it / kPfStages) & 1u;
          const bool mine = (int)(it % kPfProducerGroups) == grp;
          ++it;
          if (!mine) continue;
          // every lane polls the stage's barrier (no divergent branch)
          if (__any_sync(0xffffffffu, !mbar_wait(empty_bar(s), ph ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          if (live) {
            const uint32_t st = sA + (uint32_t)s * kPfAStage;
            uint32_t S[4], F[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              S[q] = (b == 0 ? cur[q].x : cur[q].z) << rho;         // row rho's signs one bit up
              F[q] = ~(b == 0 ? cur[q].y : cur[q].w) >> (16 * rho);  // real-axis flags of row rho in the low half
            }
            // chunk order rotated by the plane index, so that the eight lanes of
            // a quarter-warp store to eight different 16-byte bank groups
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              const int idx = (t4 + p) & 3;
              const int ss = idx >> 1, h = idx & 1;
              const int sstep = 2 * hf + ss;                  // 16-column step of the block
              const uint32_t cc = (uint32_t)(2 * sstep + h);  // 16-byte chunk of the 128-byte row
              const uint32_t fword = F[h + 2 * hf];           // flag word of lane (g, h + 2 (s >> 1))
              const uint32_t fsh = (uint32_t)(sstep & 1);
              const uint32_t ssh = (uint32_t)(4 * sstep + 2 * h);
              uint32_t re[4], im[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                // real flags of columns (2q, 2q + 1) at bits 0 and 2, then at bits 14 and 30
                const uint32_t fr = (((fword >> (4 * q + fsh)) & 5u) * 0x10004000u) & 0x40004000u;
                re[q] = real_operand_pf(S[q] << ssh, smask, fr);  // (sign, real flag)
                im[q] = re[q] ^ 0x40004000u;                      // (sign, imaginary flag)
              }
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + row_re + ((cc ^ sw_re) << 4)),
                           "r"(re[0]), "r"(re[1]), "r"(re[2]), "r"(re[3])
                           : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + row_im + ((cc ^ sw_im) << 4)),
                           "r"(im[0]), "r"(im[1]), "r"(im[2]), "r"(im[3])
                           : "memory");
            }
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
        }
      }
    }
  } else if (warp < 6 + kPfProducerWarps) {
    // ---------------- epilogue ----------------
    const int eq = warp & 3;  // TMEM lanes 32 eq .. 32 eq + 31
    const int r = 32 * eq + lane;
    const int jj = r / RO;
    const int within = r - jj * RO;
    const int p = within >> 1, a = within & 1;
    const bool prow = p < 2 * T;
    const int X = prow ? p / T : 0;
    constexpr int V = 32 / RO;  // values per lane after the reduction
    const int off = V * (lane % RO);
    uint32_t lt = 0;
    for (int64_t tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x, ++lt) {
      const PfTile c = pf_tile(P, tile);
      const PrefillProblem& pr = P.p[c.pi];
      const int b = (int)(lt & 1u);
      const int64_t j = c.rt * J + jj;
      const bool valid = prow && j < pr.n;
      const float s = valid ? 0.5f * __ldg(pr.scales + ((int64_t)p * 2 + a) * pr.n + j) : 0.0f;
      // (Re, Im) = (cA Da + cB Db, cC Da + cD Db), Da/Db = this code row's dot with a/b
      const float sx = X == 0 ? s : -s;
      const float cA = a == 0 ? s : 0.0f, cB = a == 0 ? 0.0f : -sx;
      const float cC = a == 0 ? 0.0f : s, cD = a == 0 ? sx : 0.0f;
      bool got = true;
      if (lane == 0) got = mbar_wait(accf_bar(b), (lt >> 1) & 1u, abort_flag);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * eq) << 16) + (uint32_t)b * kPfBN;
      const int64_t ystride = 2 * pr.n;
#pragma unroll 1
      for (int cc = 0; cc < kPfBN / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tbase + 32u * cc, v);
        tmem_ld_wait();
        float w[32];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float da = __uint_as_float(v[2 * u]), db = __uint_as_float(v[2 * u + 1]);
          w[2 * u] = fmaf(cA, da, cB * db);
          w[2 * u + 1] = fmaf(cC, da, cD * db);
        }
        // sum over the RO code rows of each output (consecutive lanes)
#pragma unroll
        for (int d = RO / 2, L = 32; d >= 1; d >>= 1, L >>= 1) {
          const bool hi = (lane & d) != 0;
#pragma unroll
          for (int e = 0; e < L / 2; ++e) {
            const float keep = hi ? w[e + L / 2] : w[e];
            const float send = hi ? w[e] : w[e + L / 2];
            w[e] = keep + __shfl_xor_sync(0xffffffffu, send, d);
          }
        }
        if (j < pr.n) {
#pragma unroll
          for (int e = 0; e < V; e += 2) {
            const int idx = off + e;
            const int64_t tok = (int64_t)c.tt * kPfTokens + 16 * cc + (idx >> 1);
            if (tok < P.M) {
              float* yr = pr.y + tok * ystride;
              yr[j] = w[e];
              yr[pr.n + j] = w[e + 1];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(b));
    }
  } else if (lane == 0) {
    // ---------------- code copies: each window of the tile's codes into the code ring ----------------
    // Per (16-row tile rtl of the tile, plane p): the run of the window's
    // block pairs (512 bytes each, an odd last block 256) of layout 2, to
    // run rtl 2T + p of the stage.
    uint32_t it = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
      const PfTile c = pf_tile(P, tile);
      const PrefillProblem& pr = P.p[c.pi];
      const int64_t KB = col_blocks(pr.m), fullc = KB >> 1, pairs = (KB + 1) >> 1;
      const int64_t rt0 = pf_first_row_tile<J>(c.rt);
      const int rtiles = (int)min((int64_t)(J > 16 ? J / 16 : 1), row_tiles(pr.n) - rt0);
      const int64_t pb = plane_bytes(pr.n, pr.m);
      for (int64_t c0 = 0; c0 < pairs; c0 += kPfWinPairs, ++it) {
        const int s = (int)(it % kPfCStages);
        if (!mbar_wait(emptyC(s), ((it / kPfCStages) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const int64_t full = max((int64_t)0, min((int64_t)kPfWinPairs, fullc - c0));
        const int64_t tail = min((int64_t)kPfWinPairs, pairs - c0) > full ? 1 : 0;
        const uint32_t run = (uint32_t)(full * 512 + tail * 256);
        mbar_arrive_expect_tx(fullC(s), run * (uint32_t)(rtiles * 2 * T));
        for (int rtl = 0; rtl < rtiles; ++rtl)
          for (int p = 0; p < 2 * T; ++p)
            bulk_load(sC + (uint32_t)s * kPfCStage + pf_run_off(rtl * 2 * T + p),
                      pr.codes + (int64_t)p * pb + (rt0 + rtl) * KB * kTileBytes + c0 * 512, run, fullC(s));
      }
    }
    // no copy outlives the CTA: wait for the last stages to land
    for (uint32_t k = (it > (uint32_t)kPfCStages ? it - kPfCStages : 0u); k < it; ++k)
      if (!mbar_wait(fullC((int)(k % kPfCStages)), (k / kPfCStages) & 1u, abort_flag)) break;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kPfTmemCols);
  }
}

// Self-test of the bounded wait: one thread waits on a barrier that nothing
// arrives at, with a short limit; the wait must give up, raise the timeout
// flag and return, leaving the context usable.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns);
  }
}

}  // namespace f2i
