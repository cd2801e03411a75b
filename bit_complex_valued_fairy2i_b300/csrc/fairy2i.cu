// Host side of the C ABI declared in include/fairy2i.h: argument checks,
// launch configuration and error reporting.  All arithmetic of the layer runs
// in the kernels included below.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "../../include/fairy2i.h"
#include "layout.cuh"
#include "convert_quantize.cuh"
#include "linear_decode.cuh"
#include "linear_prefill.cuh"
#include "linear_tc_decode.cuh"
#include "linear_grad.cuh"
#include "linear_lut.cuh"
#include "linear_dq.cuh"

namespace {

// An NVTX range over one C-ABI call (a no-op unless a profiler is attached),
// so that timelines show which library call issued which kernels.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

thread_local std::string g_last_error;

fairy2i_status fail(fairy2i_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

fairy2i_status ok() {
  g_last_error.clear();
  return FAIRY2I_OK;
}

fairy2i_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

// Opt a kernel in to more than 48 KB of dynamic shared memory, once per
// (kernel, device): later calls, including calls made while a stream is being
// captured into a CUDA graph, issue no attribute call.
struct SmemAttr {
  const void* fn;
  int device;
  size_t bytes;
};
std::mutex g_attr_mu;
std::vector<SmemAttr> g_attr;

fairy2i_status ensure_smem(const void* fn, size_t smem, const char* what) {
  if (smem <= 32 * 1024) return FAIRY2I_OK;  // well inside the default limit, static smem included
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const SmemAttr& a : g_attr)
    if (a.fn == fn && a.device == dev && a.bytes >= smem) return FAIRY2I_OK;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "%s shared memory attribute: %s", what, cudaGetErrorString(e));
  g_attr.push_back({fn, dev, smem});
  return FAIRY2I_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

fairy2i_status check_packed(const fairy2i_packed* q) {
  if (!q) return fail(FAIRY2I_ERR_INVALID_ARG, "packed descriptor is NULL");
  if (q->version != FAIRY2I_LAYOUT_VERSION && q->version != FAIRY2I_LAYOUT_LUT)
    return fail(FAIRY2I_ERR_INVALID_ARG, "packed layout version %d, library reads %d and %d", q->version,
                FAIRY2I_LAYOUT_VERSION, FAIRY2I_LAYOUT_LUT);
  if (q->n < 1 || q->m < 1) return fail(FAIRY2I_ERR_SHAPE, "n=%lld m=%lld must be >= 1", (long long)q->n, (long long)q->m);
  if (q->T < 1 || q->T > FAIRY2I_MAX_T) return fail(FAIRY2I_ERR_UNSUPPORTED, "T=%d outside [1, %d]", q->T, FAIRY2I_MAX_T);
  if (q->m > FAIRY2I_MAX_M) return fail(FAIRY2I_ERR_UNSUPPORTED, "m=%lld above %d", (long long)q->m, FAIRY2I_MAX_M);
  if (!q->codes || !q->scales) return fail(FAIRY2I_ERR_INVALID_ARG, "codes or scales pointer is NULL");
  if (!aligned(q->codes, 256)) return fail(FAIRY2I_ERR_INVALID_ARG, "codes pointer not 256-byte aligned");
  if (!aligned(q->scales, 16)) return fail(FAIRY2I_ERR_INVALID_ARG, "scales pointer not 16-byte aligned");
  return FAIRY2I_OK;
}

// --- decode launch helpers --------------------------------------------------

// Resident CTAs per SM for a kernel at a given dynamic shared memory size,
// cached per (kernel, device, bytes).
struct OccEntry {
  const void* fn;
  int device;
  size_t smem;
  int blocks;
};
std::mutex g_occ_mu;
std::vector<OccEntry> g_occ;

int resident_ctas(const void* fn, int threads, size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_occ_mu);
  for (const OccEntry& e : g_occ)
    if (e.fn == fn && e.device == dev && e.smem == smem) return e.blocks;
  int nb = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess || nb < 1) nb = 1;
  g_occ.push_back({fn, dev, smem, nb});
  return nb;
}

// Decode partition: `slots` resident CTAs shared among the problems in
// proportion to their bytes; every CTA of a problem owns tiles_per_cta
// (<= tiles_max) consecutive row tiles.  Returns the number of CTAs.
int partition(f2i::LinearGroup& G, int slots, int tiles_max) {
  double total = 0.0;
  for (int i = 0; i < G.count; ++i)
    total += (double)f2i::row_tiles(G.p[i].n) * (double)f2i::col_blocks(G.p[i].m);
  int ctas = 0;
  for (int i = 0; i < G.count; ++i) {
    const int64_t RT = f2i::row_tiles(G.p[i].n);
    const double share = (double)RT * (double)f2i::col_blocks(G.p[i].m) / total;
    const int64_t want = std::max<int64_t>(1, (int64_t)(slots * share));
    const int64_t tpc = std::max<int64_t>(1, std::min<int64_t>(tiles_max, (RT + want - 1) / want));
    G.p[i].cta_begin = ctas;
    G.p[i].tiles_per_cta = (int32_t)tpc;
    ctas += (int)((RT + tpc - 1) / tpc);
  }
  return ctas;
}

template <int NPL, int TILES, int WARPS>
fairy2i_status launch_mma_t(f2i::LinearGroup& G, size_t smem, int tiles_max, cudaStream_t s) {
  auto k = f2i::linear_mma_kernel<NPL, TILES, WARPS>;
  const void* fn = reinterpret_cast<const void*>(k);
  fairy2i_status st = ensure_smem(fn, smem, "mma decode");
  if (st != FAIRY2I_OK) return st;
  const int slots = sm_count() * resident_ctas(fn, WARPS * 32, smem);
  const int ctas = partition(G, slots, tiles_max);
  k<<<ctas, WARPS * 32, smem, s>>>(G);
  return check_launch("mma decode launch");
}

// 16-warp CTAs exist only where 512 threads fit the register file without
// spills (NPL * TILES <= 8, at most 128 registers per thread).
template <int NPL>
fairy2i_status launch_mma_tiles(f2i::LinearGroup& G, int tiles, bool wide, size_t smem, int tiles_max,
                                cudaStream_t s) {
  constexpr int W = f2i::kMmaWarpsWide;
  if (wide) {
    if (tiles == 1) return launch_mma_t<NPL, 1, W>(G, smem, tiles_max, s);
    if constexpr (NPL * 2 <= 8)
      if (tiles == 2) return launch_mma_t<NPL, 2, W>(G, smem, tiles_max, s);
    if constexpr (NPL * 4 <= 8)
      if (tiles == 4) return launch_mma_t<NPL, 4, W>(G, smem, tiles_max, s);
    return fail(FAIRY2I_ERR_UNSUPPORTED, "mma decode: no 16-warp form for %d planes x %d token pairs", NPL, tiles);
  }
  constexpr int N = f2i::kMmaWarps;
  return tiles == 1   ? launch_mma_t<NPL, 1, N>(G, smem, tiles_max, s)
         : tiles == 2 ? launch_mma_t<NPL, 2, N>(G, smem, tiles_max, s)
                      : launch_mma_t<NPL, 4, N>(G, smem, tiles_max, s);
}

// One launch of the sparse mma decode for up to 8 tokens of every problem in
// G (two tokens per mma).  Shared memory: the code rings, the staged
// activations ([2M + 1][x_stride] bfloat16) and the per-warp partial outputs
// of up to tiles_max row tiles.
constexpr int kMmaTokens = 8;
constexpr size_t kMmaWideSmem = 220 * 1024;  // one CTA per SM

int mma_token_pairs(int M) { return M <= 2 ? 1 : M <= 4 ? 2 : 4; }

// Shared-memory bytes of a launch with `warps` warps: fixed part (code rings
// and staged activations) and partial outputs per row tile.
void mma_smem(int warps, int T, int M, int64_t xstr_max, size_t& fixed, size_t& per_tile) {
  const size_t ring = (size_t)warps * 2 * (2 * T) * 512;
  const size_t xbytes = (((size_t)(2 * M + 1) * xstr_max * sizeof(uint16_t)) + 15) & ~(size_t)15;
  fixed = ring + xbytes;
  per_tile = (size_t)warps * mma_token_pairs(M) * 64 * sizeof(float2);
}

// Whether a launch runs as one 16-warp CTA per SM.  Measured on the LLaMA-2-7B
// block at T = 2 against two 8-warp CTAs per SM: 24.6 against 26.65 us at M = 1,
// 55.7 against 65.8 us at M = 4 (the whole-row-tile partition balances better
// over 148 large CTAs than over 296 small ones).  Needs the 16-warp form
// (2T planes x token pairs <= 8) and room for two row tiles of partial outputs.
bool mma_wide(int T, int M, int64_t xstr_max) {
  if (2 * T * mma_token_pairs(M) > 8) return false;
  size_t fixed, per_tile;
  mma_smem(f2i::kMmaWarpsWide, T, M, xstr_max, fixed, per_tile);
  return fixed + 2 * per_tile <= kMmaWideSmem;
}

// The mma decode forms a lane's code offsets inside a layer in 32 bits (plane
// index x plane bytes + offset in the plane): all 2T planes of a layer must
// lie within 4 GB.
bool mma_offsets_fit(const fairy2i_packed& q) {
  return (uint64_t)(2 * q.T) * (uint64_t)f2i::plane_bytes(q.n, q.m) <= 0xFFFFFFFFull;
}

fairy2i_status run_mma(f2i::LinearGroup& G, int T, cudaStream_t s) {
  const int tiles = mma_token_pairs(G.M);
  int64_t xstr_max = 0;
  for (int i = 0; i < G.count; ++i) xstr_max = std::max(xstr_max, f2i::x_stride(G.p[i].m));
  const bool wide = mma_wide(T, G.M, xstr_max);
  size_t fixed, per_tile, limit;
  if (wide) {
    mma_smem(f2i::kMmaWarpsWide, T, G.M, xstr_max, fixed, per_tile);
    limit = kMmaWideSmem;
  } else {
    // Two 8-warp CTAs per SM when the buffers leave room for at least four row
    // tiles of partial outputs; otherwise one CTA with up to 200 KB.
    mma_smem(f2i::kMmaWarps, T, G.M, xstr_max, fixed, per_tile);
    limit = fixed + 4 * per_tile <= 110 * 1024 ? 110 * 1024 : 200 * 1024;
  }
  if (fixed + per_tile > limit)
    return fail(FAIRY2I_ERR_UNSUPPORTED, "mma decode: buffers need %zu bytes of shared memory", fixed + per_tile);
  const int tiles_max = (int)std::min<size_t>(f2i::kMaxTilesPerCta, (limit - fixed) / per_tile);
  const size_t smem = fixed + (size_t)tiles_max * per_tile;
  switch (T) {
    case 1: return launch_mma_tiles<2>(G, tiles, wide, smem, tiles_max, s);
    case 2: return launch_mma_tiles<4>(G, tiles, wide, smem, tiles_max, s);
    case 3: return launch_mma_tiles<6>(G, tiles, wide, smem, tiles_max, s);
    case 4: return launch_mma_tiles<8>(G, tiles, wide, smem, tiles_max, s);
    default: return fail(FAIRY2I_ERR_UNSUPPORTED, "mma decode supports T <= 4 (got %d)", T);
  }
}

// Tokens per sparse-mma launch: 8, or fewer when the staged activations of
// the widest layer of the group would not fit in shared memory.
int mma_chunk(const fairy2i_packed* qs, int count, int T) {
  int64_t xstr_max = 0;
  for (int i = 0; i < count; ++i) xstr_max = std::max(xstr_max, f2i::x_stride(qs[i].m));
  const size_t ring = (size_t)f2i::kMmaWarps * 2 * (2 * T) * 512;
  for (int mc = kMmaTokens; mc > 1; mc /= 2) {
    const size_t xbytes = (((size_t)(2 * mc + 1) * xstr_max * sizeof(uint16_t)) + 15) & ~(size_t)15;
    const int tiles = mc <= 2 ? 1 : mc <= 4 ? 2 : 4;
    if (ring + xbytes + (size_t)f2i::kMmaWarps * tiles * 64 * sizeof(float2) <= 200 * 1024) return mc;
  }
  return 1;
}

// Whether a sparse-mma launch of these layers with mc tokens keeps all 16
// warps per SM: one 16-warp CTA, or two 8-warp CTAs (the rules run_mma
// applies).  If not, the caller launches the layers per activation width.
bool mma_full_sm(const fairy2i_packed* qs, int count, int T, int mc) {
  int64_t xstr_max = 0;
  for (int i = 0; i < count; ++i) xstr_max = std::max(xstr_max, f2i::x_stride(qs[i].m));
  if (mma_wide(T, mc, xstr_max)) return true;
  size_t fixed, per_tile;
  mma_smem(f2i::kMmaWarps, T, mc, xstr_max, fixed, per_tile);
  return fixed + 4 * per_tile <= 110 * 1024;
}

fairy2i_status run_addsub(f2i::LinearGroup& G, cudaStream_t s) {
  int ctas = 0;
  int64_t m_pad_max = 0;
  for (int i = 0; i < G.count; ++i) {
    G.p[i].cta_begin = ctas;
    ctas += (int)((f2i::row_tiles(G.p[i].n) + f2i::kAddSubWarps - 1) / f2i::kAddSubWarps);
    m_pad_max = std::max(m_pad_max, f2i::col_blocks(G.p[i].m) * 64);
  }
  const size_t smem = (size_t)f2i::kAddSubTok * m_pad_max * sizeof(uint32_t);
  fairy2i_status st = ensure_smem(reinterpret_cast<const void*>(f2i::linear_addsub_kernel), smem, "addsub decode");
  if (st != FAIRY2I_OK) return st;
  f2i::linear_addsub_kernel<<<ctas, f2i::kAddSubWarps * 32, smem, s>>>(G);
  return check_launch("addsub decode launch");
}

// --- prefill (tcgen05) launch helpers ---------------------------------------

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
fairy2i_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000& out) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      return fail(FAIRY2I_ERR_CUDA, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(e));
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  out = fn;
  return FAIRY2I_OK;
}

// x [M][2m] bfloat16 seen as a [2M][m] tensor (row 2 * token + part), tiles of
// 256 rows x 64 columns, 128-byte swizzle, zero fill outside.
fairy2i_status make_x_map(CUtensorMap* map, const void* x, int64_t M, int64_t m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  fairy2i_status st = tensor_map_encoder(enc);
  if (st != FAIRY2I_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)m, (cuuint64_t)(2 * M)};
  const cuuint64_t strides[1] = {(cuuint64_t)m * 2};
  const cuuint32_t box[2] = {(cuuint32_t)f2i::kPfBK, (cuuint32_t)f2i::kPfBN};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FAIRY2I_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FAIRY2I_OK;
}

// One half of x [M][2m] bfloat16, or of its fp16 copy (half 0: Re x, columns
// 0..m-1; half 1: Im x) as a [M][m] tensor with row pitch 2m: tiles of N
// tokens x 64 columns, 128-byte swizzle, zero fill past m columns and M tokens
// (the dequantized GEMM's B operand).  The Im half starts 2m bytes in:
// 16-byte aligned for m a multiple of 8.
fairy2i_status make_x_map_half(CUtensorMap* map, const void* x, int64_t M, int64_t m, int half, int N, bool f16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  fairy2i_status st = tensor_map_encoder(enc);
  if (st != FAIRY2I_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)m, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)m * 4};
  const cuuint32_t box[2] = {(cuuint32_t)f2i::kDqBK, (cuuint32_t)N};
  const cuuint32_t estr[2] = {1, 1};
  void* base = const_cast<uint8_t*>(static_cast<const uint8_t*>(x) + (half ? 2 * m : 0));
  const CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                         strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FAIRY2I_ERR_CUDA, "cuTensorMapEncodeTiled (x half %d) failed (%d)", half, (int)r);
  return FAIRY2I_OK;
}

// Launches a kernel as a programmatic dependent of the previous work in the
// stream (it may start while that work finishes; its griddepcontrol.wait
// orders everything that depends on it).
template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Params& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, P);
}

// The fp16 form is a programmatic dependent of its conversion launch: it sets
// up and decodes codes while the conversion finishes; only the threads that
// read the fp16 copy or the tokens' factors wait for it.
template <int T, int NT, bool SMALL, bool F16>
fairy2i_status launch_dq_t(const f2i::DqParams& P, int grid, cudaStream_t s) {
  auto k = f2i::linear_dq_kernel<T, NT, SMALL, F16>;
  const size_t smem = f2i::dq_smem_bytes<NT, T, SMALL, F16>();
  fairy2i_status st = ensure_smem(reinterpret_cast<const void*>(k), smem, "dequantized prefill");
  if (st != FAIRY2I_OK) return st;
  if (F16) {
    const cudaError_t e = launch_pdl(k, dim3((unsigned)grid), dim3(f2i::kDqThreads), smem, s, P);
    if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "dequantized prefill launch: %s", cudaGetErrorString(e));
  } else {
    k<<<(unsigned)grid, f2i::kDqThreads, smem, s>>>(P);
  }
  return check_launch("dequantized prefill launch");
}

// Tiles of a launch that fits one or a few waves differ in length (a tile
// costs one decode + MMA step per 128 columns of x~, plus its epilogue), so a
// round-robin deal leaves some CTAs with far more steps than the mean. For up
// to kDqSchedMax tiles the host deals them longest first, each to the CTA
// with the least work so far; larger launches keep the round-robin deal.
void dq_schedule(f2i::DqParams& P, int grid, int nt) {
  P.sched_n = 0;
  if (P.total_tiles > f2i::kDqSchedMax || grid > f2i::kDqMaxCtas || grid < 1) return;
  std::vector<std::pair<int64_t, int>> order;  // (cost, tile)
  order.reserve((size_t)P.total_tiles);
  for (int i = 0; i < P.count; ++i) {
    const f2i::DqProblem& pr = P.p[i];
    const int64_t n_tiles = (int64_t)pr.row_tiles * pr.tok_tiles;
    for (int64_t t = 0; t < n_tiles; ++t) order.emplace_back((int64_t)pr.kpairs * nt + 1, (int)(pr.tile_begin + t));
  }
  std::stable_sort(order.begin(), order.end(),
                   [](const std::pair<int64_t, int>& a, const std::pair<int64_t, int>& b) { return a.first > b.first; });
  using Load = std::pair<int64_t, int>;  // (work so far, cta)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int b = 0; b < grid; ++b) heap.emplace(0, b);
  std::vector<std::vector<int>> lists((size_t)grid);
  for (const auto& o : order) {
    Load l = heap.top();
    heap.pop();
    lists[(size_t)l.second].push_back(o.second);
    l.first += o.first;
    heap.push(l);
  }
  int k = 0;
  for (int b = 0; b < grid; ++b) {
    P.cta_begin[b] = (uint16_t)k;
    for (int t : lists[(size_t)b]) P.sched[k++] = (uint16_t)t;
  }
  P.cta_begin[grid] = (uint16_t)k;
  P.sched_n = k;
}

constexpr size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of the fp16 form for one launch's layers: per layer the fp16 copy
// of x (M x 2m values) and the per-token factors (M floats), each 256-byte
// aligned; launches run in stream order and reuse it.
size_t dq16_launch_workspace(const fairy2i_packed* qs, int cnt, int64_t M) {
  size_t need = 0;
  for (int i = 0; i < cnt; ++i) need += round256((size_t)M * 4 * (size_t)qs[i].m) + round256((size_t)M * 4);
  return need;
}
size_t dq16_workspace(const fairy2i_packed* qs, int count, int64_t M) {
  size_t need = 0;
  for (int p0 = 0; p0 < count; p0 += f2i::kDqMaxGroup)
    need = std::max(need, dq16_launch_workspace(qs + p0, std::min(f2i::kDqMaxGroup, count - p0), M));
  return need;
}

template <int T, int NT, bool SMALL>
fairy2i_status launch_dq_form(const f2i::DqParams& P, int grid, bool f16, cudaStream_t s) {
  return f16 ? launch_dq_t<T, NT, SMALL, true>(P, grid, s) : launch_dq_t<T, NT, SMALL, false>(P, grid, s);
}

// The dense GEMM of the dequantized real matrix (layout 3, m a multiple of 8,
// T <= 4): one launch per kDqMaxGroup layers, tiles of 64 outputs x NT N tokens
// (N = min(256, M rounded up to 16); NT = 2 above 256 tokens for T <= 2).
// f16: the fp16 form, each launch preceded by the activations' conversion
// into the workspace (dq16_workspace bytes, 256-byte aligned; checked here).
fairy2i_status run_dq(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int count, int64_t M, int T,
                      cudaStream_t s, bool f16 = false, void* ws = nullptr, size_t ws_bytes = 0,
                      bool out_bf16 = false) {
  if (f16) {
    const size_t need = dq16_workspace(qs, count, M);
    if (!ws) return fail(FAIRY2I_ERR_INVALID_ARG, "the fp16 dequantized GEMM needs a workspace of %zu bytes", need);
    if (ws_bytes < need)
      return fail(FAIRY2I_ERR_INVALID_ARG, "workspace of %zu bytes, the fp16 dequantized GEMM needs %zu", ws_bytes, need);
    if (!aligned(ws, 256)) return fail(FAIRY2I_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  }
  for (int p0 = 0; p0 < count; p0 += f2i::kDqMaxGroup) {
    const int cnt = std::min(f2i::kDqMaxGroup, count - p0);
    const void* xb[f2i::kDqMaxGroup];  // the B operand of each layer: x or its fp16 copy
    const float* xf[f2i::kDqMaxGroup] = {};
    for (int i = 0; i < cnt; ++i) xb[i] = xs[p0 + i];
    if (f16) {
      f2i::DqXParams XP;
      memset(&XP, 0, sizeof(XP));
      XP.count = cnt;
      uint8_t* w = static_cast<uint8_t*>(ws);
      for (int i = 0; i < cnt; ++i) {
        XP.x[i] = static_cast<const uint16_t*>(xs[p0 + i]);
        XP.xh[i] = reinterpret_cast<uint16_t*>(w);
        w += round256((size_t)M * 4 * (size_t)qs[p0 + i].m);
        XP.xfac[i] = reinterpret_cast<float*>(w);
        w += round256((size_t)M * 4);
        XP.m[i] = (int32_t)qs[p0 + i].m;
        xb[i] = XP.xh[i];
        xf[i] = XP.xfac[i];
      }
      f2i::dq_x16_kernel<<<dim3((unsigned)M, (unsigned)cnt), f2i::kDqXThreads, 0, s>>>(XP);
      fairy2i_status st = check_launch("activation conversion launch");
      if (st != FAIRY2I_OK) return st;
    }
    f2i::DqParams P;
    memset(&P, 0, sizeof(P));
    P.count = cnt;
    P.T = T;
    P.M = (int32_t)M;
    P.N = M >= f2i::kDqBN ? f2i::kDqBN : (int32_t)((M + 15) / 16 * 16);  // the MMA's N: a multiple of 16
    // token tiles per decoded k-block pair (two need the shared memory that the
    // larger code windows of T > 2 take)
    const int nt = M > f2i::kDqBN && T <= 2 ? 2 : 1;
    int64_t tiles = 0;
    for (int i = 0; i < cnt; ++i) {
      const fairy2i_packed& q = qs[p0 + i];
      for (int half = 0; half < 2; ++half) {
        fairy2i_status st = make_x_map_half(&P.tmap[2 * i + half], xb[i], M, q.m, half, P.N, f16);
        if (st != FAIRY2I_OK) return st;
      }
      f2i::DqProblem& pr = P.p[i];
      pr.codes = static_cast<const uint8_t*>(q.codes);
      pr.scales = q.scales;
      pr.y = ys[p0 + i];
      pr.xfac = xf[i];
      pr.out_bf16 = out_bf16 ? 1 : 0;
      pr.n = (int32_t)q.n;
      pr.m = (int32_t)q.m;
      pr.row_tiles = (int32_t)((q.n + 63) / 64);
      pr.tok_tiles = (int32_t)((M + (int64_t)nt * P.N - 1) / ((int64_t)nt * P.N));
      pr.kpairs = (int32_t)((q.m + f2i::kDqBK - 1) / f2i::kDqBK);
      pr.tile_begin = tiles;
      tiles += (int64_t)pr.row_tiles * pr.tok_tiles;
    }
    P.total_tiles = tiles;
    const int grid = (int)std::min<int64_t>(tiles, sm_count());
    dq_schedule(P, grid, nt);
    const bool small = nt == 1 && P.N <= 64;  // value tables in 8 KB-B-stage room
    fairy2i_status st;
    switch (T * 2 + nt - 1) {
      case 2: st = small ? launch_dq_form<1, 1, true>(P, grid, f16, s) : launch_dq_form<1, 1, false>(P, grid, f16, s); break;
      case 3: st = launch_dq_form<1, 2, false>(P, grid, f16, s); break;
      case 4: st = small ? launch_dq_form<2, 1, true>(P, grid, f16, s) : launch_dq_form<2, 1, false>(P, grid, f16, s); break;
      case 5: st = launch_dq_form<2, 2, false>(P, grid, f16, s); break;
      case 6: st = small ? launch_dq_form<3, 1, true>(P, grid, f16, s) : launch_dq_form<3, 1, false>(P, grid, f16, s); break;
      case 8: st = small ? launch_dq_form<4, 1, true>(P, grid, f16, s) : launch_dq_form<4, 1, false>(P, grid, f16, s); break;
      default: return fail(FAIRY2I_ERR_UNSUPPORTED, "dequantized prefill supports T <= 4");
    }
    if (st != FAIRY2I_OK) return st;
  }
  return ok();
}

template <int RO>
fairy2i_status launch_tcgen05_t(const f2i::PrefillParams& P, cudaStream_t s) {
  auto k = f2i::linear_tcgen05_kernel<RO>;
  const void* fn = reinterpret_cast<const void*>(k);
  fairy2i_status st = ensure_smem(fn, f2i::kPfSmemBytes, "tcgen05 prefill");
  if (st != FAIRY2I_OK) return st;
  const int64_t grid = std::min<int64_t>(P.total_tiles, sm_count());
  k<<<(unsigned)grid, f2i::kPfThreads, f2i::kPfSmemBytes, s>>>(P);
  return check_launch("tcgen05 prefill launch");
}

// Code rows per output in a prefill tile: 4T rounded up to a power of two.
int prefill_rows_per_output(int T) { return T == 1 ? 4 : T == 2 ? 8 : 16; }

fairy2i_status run_tcgen05(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int count, int64_t M,
                           int T, cudaStream_t s) {
  const int ro = prefill_rows_per_output(T);
  const int J = f2i::kPfBM / ro;
  for (int p0 = 0; p0 < count; p0 += f2i::kPfMaxGroup) {
    const int cnt = std::min(f2i::kPfMaxGroup, count - p0);
    f2i::PrefillParams P;
    memset(&P, 0, sizeof(P));
    P.count = cnt;
    P.T = T;
    P.M = (int32_t)M;
    int64_t tiles = 0;
    for (int i = 0; i < cnt; ++i) {
      const fairy2i_packed& q = qs[p0 + i];
      fairy2i_status st = make_x_map(&P.tmap[i], xs[p0 + i], M, q.m);
      if (st != FAIRY2I_OK) return st;
      f2i::PrefillProblem& pr = P.p[i];
      pr.codes = static_cast<const uint8_t*>(q.codes);
      pr.scales = q.scales;
      pr.y = ys[p0 + i];
      pr.n = q.n;
      pr.m = q.m;
      pr.row_tiles = (q.n + J - 1) / J;
      pr.tok_tiles = (int32_t)((M + f2i::kPfTokens - 1) / f2i::kPfTokens);
      pr.kblocks = (int32_t)((q.m + f2i::kPfBK - 1) / f2i::kPfBK);
      pr.tile_begin = tiles;
      tiles += pr.row_tiles * pr.tok_tiles;
    }
    P.total_tiles = tiles;
    fairy2i_status st = ro == 4 ? launch_tcgen05_t<4>(P, s) : ro == 8 ? launch_tcgen05_t<8>(P, s)
                                                                       : launch_tcgen05_t<16>(P, s);
    if (st != FAIRY2I_OK) return st;
  }
  return ok();
}

// --- batch decode on the sparse tensor core (tcgen05.mma.sp) ---------------

// Output rows per tile: 2T planes x R rows fill at most the 128 TMEM lanes.
int tc_decode_rows(int T) { return T <= 2 ? 64 / T : 16; }

// Code planes of layer q as TMA views: full two-block chunks as (u32 of a lane
// quad, lane quad g, chunk, row tile, plane) with 64-byte swizzle, and an odd
// last block as (u32, g, row tile, plane).  Boxes cover one chunk of R rows of
// every plane.
fairy2i_status make_code_maps(CUtensorMap* cmap, CUtensorMap* tmap, const fairy2i_packed& q, int R) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  fairy2i_status st = tensor_map_encoder(enc);
  if (st != FAIRY2I_OK) return st;
  const int64_t KB = f2i::col_blocks(q.m), rt = f2i::row_tiles(q.n), full = KB / 2;
  const uint64_t plane = (uint64_t)f2i::plane_bytes(q.n, q.m);
  const cuuint64_t planes = (cuuint64_t)(2 * q.T);
  if (full > 0) {
    const cuuint64_t dims[5] = {16, 8, (cuuint64_t)full, (cuuint64_t)rt, planes};
    const cuuint64_t strides[4] = {64, 512, (cuuint64_t)(KB * 256), plane};
    const cuuint32_t box[5] = {16, 8, 1, (cuuint32_t)(R / 16), (cuuint32_t)planes};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(cmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, q.codes, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FAIRY2I_ERR_CUDA, "cuTensorMapEncodeTiled (code chunks) failed (%d)", (int)r);
  }
  if (KB & 1) {
    void* tail = static_cast<uint8_t*>(q.codes) + full * 512;
    const cuuint64_t dims[4] = {8, 8, (cuuint64_t)rt, planes};
    const cuuint64_t strides[3] = {32, (cuuint64_t)(KB * 256), plane};
    const cuuint32_t box[4] = {8, 8, (cuuint32_t)(R / 16), (cuuint32_t)planes};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, tail, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FAIRY2I_ERR_CUDA, "cuTensorMapEncodeTiled (code tail) failed (%d)", (int)r);
  }
  return FAIRY2I_OK;
}

// One launch over up to kTdMaxGroup layers: tiles of R output rows are given
// to CTAs by longest-processing-time-first (cost = MMAs + a constant for the
// epilogue), so every CTA gets nearly the same number of MMAs.
fairy2i_status launch_tc_decode(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int count,
                                int64_t M, int T, cudaStream_t s) {
  static_assert(sizeof(f2i::TdParams) <= 32000, "kernel parameters too large");
  const int R = tc_decode_rows(T);
  f2i::TdParams* Pp = new f2i::TdParams;
  std::unique_ptr<f2i::TdParams> guard(Pp);
  f2i::TdParams& P = *Pp;
  memset(&P, 0, sizeof(P));
  P.count = count;
  P.T = T;
  P.R = R;
  P.M = (int32_t)M;
  P.N = 16 * (int32_t)((M + 1) / 2);
  P.nsub = P.N <= 32 ? 4 : 2;
  P.bstage_bytes = 256 * P.N;
  struct Tile {
    int cost, prob, tile;
  };
  std::vector<Tile> tiles;
  for (int i = 0; i < count; ++i) {
    const fairy2i_packed& q = qs[i];
    fairy2i_status st = make_code_maps(&P.cmap[i], &P.tmap[i], q, R);
    if (st != FAIRY2I_OK) return st;
    f2i::TdProblem& pr = P.p[i];
    pr.scales = q.scales;
    pr.x = static_cast<const uint16_t*>(xs[i]);
    pr.y = ys[i];
    pr.n = (int32_t)q.n;
    pr.m = (int32_t)q.m;
    pr.KB = (int32_t)f2i::col_blocks(q.m);
    pr.tiles = (int32_t)((q.n + R - 1) / R);
    for (int k = 0; k < pr.tiles; ++k) tiles.push_back({2 * pr.KB + 8, i, k});
  }
  const int ctas = (int)std::min<int64_t>({(int64_t)tiles.size(), (int64_t)sm_count(), (int64_t)f2i::kTdMaxCtas});
  std::stable_sort(tiles.begin(), tiles.end(), [](const Tile& a, const Tile& b) { return a.cost > b.cost; });
  // least-loaded CTA first (ties to the lower index): a min-heap of (load, cta)
  std::vector<std::vector<uint16_t>> per(ctas);
  std::priority_queue<std::pair<int64_t, int>, std::vector<std::pair<int64_t, int>>, std::greater<>> heap;
  for (int c = 0; c < ctas; ++c) heap.push({0, c});
  for (const Tile& t : tiles) {
    auto [load, c] = heap.top();
    heap.pop();
    per[c].push_back((uint16_t)((t.prob << 13) | t.tile));
    heap.push({load + t.cost, c});
  }
  int e = 0;
  for (int c = 0; c < ctas; ++c) {
    if (per[c].size() > (size_t)f2i::kTdMaxLocal)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "sparse tensor-core decode: %zu tiles on one CTA", per[c].size());
    std::sort(per[c].begin(), per[c].end());
    P.off[c] = (uint16_t)e;
    for (uint16_t v : per[c]) P.sched[e++] = v;
  }
  P.off[ctas] = (uint16_t)e;
  const void* fn = reinterpret_cast<const void*>(f2i::linear_tc_decode_kernel);
  const size_t smem = std::max<size_t>(
      120 * 1024, 1024 + (size_t)f2i::kTdAStages * f2i::kTdAStageBytes + (size_t)f2i::kTdTStages * P.bstage_bytes +
                      f2i::kTdRedBytes + sizeof(f2i::TdSmem));
  fairy2i_status st = ensure_smem(fn, smem, "sparse tensor-core decode");
  if (st != FAIRY2I_OK) return st;
  f2i::linear_tc_decode_kernel<<<ctas, f2i::kTdThreads, smem, s>>>(P);
  return check_launch("sparse tensor-core decode launch");
}

fairy2i_status run_tc_decode(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int count,
                             int64_t M, int T, cudaStream_t s) {
  const int R = tc_decode_rows(T);
  for (int b0 = 0; b0 < count;) {
    int b1 = b0;
    int64_t t = 0;
    while (b1 < count && b1 - b0 < f2i::kTdMaxGroup) {
      const int64_t ti = (qs[b1].n + R - 1) / R;
      if (ti > 8192) return fail(FAIRY2I_ERR_UNSUPPORTED, "n=%lld too large for the sparse tensor-core decode",
                                 (long long)qs[b1].n);
      if (b1 > b0 && t + ti > f2i::kTdMaxSched) break;
      if (t + ti > f2i::kTdMaxSched) return fail(FAIRY2I_ERR_UNSUPPORTED, "layer with too many row tiles");
      t += ti;
      ++b1;
    }
    fairy2i_status st = launch_tc_decode(qs + b0, xs + b0, ys + b0, b1 - b0, M, T, s);
    if (st != FAIRY2I_OK) return st;
    b0 = b1;
  }
  return ok();
}

// Largest token count of the sparse tensor-core decode (N = 8 B columns per
// token, at most 64).
constexpr int64_t kTcDecodeMaxTokens = 8;

// Token count from which FAIRY2I_ALGO_AUTO takes the tcgen05 prefill path.
constexpr int64_t kPrefillMinTokens = 16;
// Token count from which AUTO, given a workspace, takes the fp16 dequantized
// GEMM over the table-lookup decode on layout 3.  The table lookup runs in
// launches of 2 or 3 tokens at T <= 2 (26.6 and 41 us each on a LLaMA-2-7B
// block), the fp16 GEMM takes ~128 us at any count up to 16: measured per
// block (eager / CUDA graph) at 9 tokens 123.9 / 115.3 us against 127.6 /
// 125.0, at 10 tokens 134.4 / 125.2 against 128.0 / 125.3.
constexpr int64_t kDqMinTokens = 10;

// The quantizer over U, W (FUSED = false) or straight from R (true); the
// caller has checked the arguments.  Codes are zeroed first: each row ORs its
// bits into words it shares with the other row of its lane pair.
template <int LAYOUT>
void quantize_kernels(const float2* U, const float2* W, const float* R, int64_t n, int64_t m, int32_t T, int64_t rows,
                      int wpt, int threads, uint8_t* codes, float* scales, cudaStream_t s) {
  if (R == nullptr) {
    const dim3 grid((unsigned)rows, 2);
    if (wpt == 1) f2i::quantize_words_kernel<1, false, LAYOUT><<<grid, threads, 0, s>>>(U, W, R, n, m, T, codes, scales);
    else f2i::quantize_words_kernel<2, false, LAYOUT><<<grid, threads, 0, s>>>(U, W, R, n, m, T, codes, scales);
  } else {
    const dim3 grid(2, (unsigned)rows);
    if (wpt == 1) f2i::quantize_words_kernel<1, true, LAYOUT><<<grid, threads, 0, s>>>(U, W, R, n, m, T, codes, scales);
    else f2i::quantize_words_kernel<2, true, LAYOUT><<<grid, threads, 0, s>>>(U, W, R, n, m, T, codes, scales);
  }
}

fairy2i_status launch_quantize(const float2* U, const float2* W, const float* R, int64_t n, int64_t m, int32_t T,
                               const fairy2i_packed* out, cudaStream_t s) {
  uint8_t* codes = static_cast<uint8_t*>(out->codes);
  if (out->version == FAIRY2I_LAYOUT_LUT) {
    // layout 3: every 16-byte chunk of a row is written once by the row's CTA
    // (rows past n in the last tile write zeros), so nothing is cleared first
    const int64_t words = 4 * f2i::l3_row_slots(m);
    const int wpt = words <= f2i::kQuantThreads ? 1 : 2;
    const int threads = (int)(((words + wpt - 1) / wpt + 31) / 32 * 32);
    const int64_t rows = f2i::l3_tiles(n) * 32;
    if (R != nullptr && rows > 65535) return fail(FAIRY2I_ERR_UNSUPPORTED, "n=%lld too large for the fused path", (long long)n);
    quantize_kernels<3>(U, W, R, n, m, T, rows, wpt, threads, codes, out->scales, s);
    return check_launch("quantize launch");
  }
  cudaError_t e = cudaMemsetAsync(out->codes, 0, fairy2i_codes_bytes(n, m, T), s);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "memset codes: %s", cudaGetErrorString(e));
  const int64_t words = 4 * f2i::col_blocks(m);  // packed words per row
  const int wpt = words <= f2i::kQuantThreads ? 1 : 2;
  const int threads = (int)(((words + wpt - 1) / wpt + 31) / 32 * 32);
  quantize_kernels<2>(U, W, R, n, m, T, n, wpt, threads, codes, out->scales, s);
  return check_launch("quantize launch");
}

// --- table-lookup decode (layout 3) ------------------------------------------

// Layers of one launch: consecutive runs of at most kLutMaxGroup layers.
// Workspace of a launch with mc tokens: a float2 partial output per (unit,
// token, row of the tile) of every layer with more than one window.
size_t lut_launch_workspace(const fairy2i_packed* qs, int cnt, int mc) {
  size_t parts = 0;
  for (int i = 0; i < cnt; ++i) {
    const int64_t tiles = f2i::l3_tiles(qs[i].n), windows = f2i::l3_windows(qs[i].m);
    if (windows > 1) parts += (size_t)(tiles * windows) * (size_t)mc * 32;
  }
  return parts * sizeof(float2);
}

size_t lut_workspace(const fairy2i_packed* qs, int count, int64_t M, int T) {
  const int mc = f2i::lut_launch_tokens(M, 0, T);  // the first launch is the largest
  size_t need = 0;
  for (int p0 = 0; p0 < count; p0 += f2i::kLutMaxGroup)
    need = std::max(need, lut_launch_workspace(qs + p0, std::min(f2i::kLutMaxGroup, count - p0), mc));
  return need;
}


template <int T, int M>
fairy2i_status launch_lut_t(const f2i::LutParams& P, int ctas, cudaStream_t s) {
  auto k = f2i::linear_lut_kernel<T, M>;
  fairy2i_status st = ensure_smem(reinterpret_cast<const void*>(k), f2i::kLutSmemBytes, "table-lookup decode");
  if (st != FAIRY2I_OK) return st;
  const cudaError_t e = launch_pdl(k, dim3(ctas), dim3(f2i::kLutThreads), f2i::kLutSmemBytes, s, P);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "table-lookup decode launch: %s", cudaGetErrorString(e));
  return check_launch("table-lookup decode launch");
}

fairy2i_status launch_lut(const f2i::LutParams& P, int T, int mc, int ctas, cudaStream_t s) {
  switch (T * 8 + mc) {
    case 9: return launch_lut_t<1, 1>(P, ctas, s);
    case 10: return launch_lut_t<1, 2>(P, ctas, s);
    case 11: return launch_lut_t<1, 3>(P, ctas, s);
    case 17: return launch_lut_t<2, 1>(P, ctas, s);
    case 18: return launch_lut_t<2, 2>(P, ctas, s);
    case 19: return launch_lut_t<2, 3>(P, ctas, s);
    case 25: return launch_lut_t<3, 1>(P, ctas, s);
    case 26: return launch_lut_t<3, 2>(P, ctas, s);
    case 33: return launch_lut_t<4, 1>(P, ctas, s);
    default: return fail(FAIRY2I_ERR_UNSUPPORTED, "table-lookup decode: no kernel for T=%d with %d tokens", T, mc);
  }
}

// One launch per kLutMaxGroup layers and per lut_launch_tokens tokens.  Units
// (layer, window, row tile) are split over one CTA per SM by their cost, in
// launch order: 8 per slot of codes plus 3 for the unit's epilogue.
fairy2i_status run_lut(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int count, int64_t M, int T,
                       void* ws, size_t ws_bytes, cudaStream_t s, bool out_bf16 = false) {
  const size_t need = lut_workspace(qs, count, M, T);
  if (need > 0) {
    if (!ws) return fail(FAIRY2I_ERR_INVALID_ARG, "table-lookup decode needs a workspace of %zu bytes", need);
    if (ws_bytes < need)
      return fail(FAIRY2I_ERR_INVALID_ARG, "workspace of %zu bytes, the table-lookup decode needs %zu", ws_bytes, need);
    if (!aligned(ws, 256)) return fail(FAIRY2I_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  }
  for (int i = 0; i < count; ++i)
    if (f2i::l3_tiles(qs[i].n) * f2i::l3_windows(qs[i].m) > (int64_t)1 << 30)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "layer %d too large for the table-lookup decode", i);
  std::unique_ptr<f2i::LutParams> holder(new f2i::LutParams);
  f2i::LutParams& P = *holder;
  f2i::LutReduceParams RP;
  for (int p0 = 0; p0 < count; p0 += f2i::kLutMaxGroup) {
    const int cnt = std::min(f2i::kLutMaxGroup, count - p0);
    for (int64_t t0 = 0, mc = 0; t0 < M; t0 += mc) {
      mc = f2i::lut_launch_tokens(M, t0, T);
      memset(&P, 0, sizeof(P));
      memset(&RP, 0, sizeof(RP));
      const size_t wsn = lut_launch_workspace(qs + p0, cnt, mc);
      P.count = cnt;
      P.M = mc;
      P.partials = wsn ? static_cast<float2*>(ws) : nullptr;
      RP.M = mc;
      int64_t units = 0, part = 0, rrows = 0;
      for (int i = 0; i < cnt; ++i) {
        const fairy2i_packed& q = qs[p0 + i];
        f2i::LutProblem& L = P.p[i];
        L.codes = static_cast<const uint8_t*>(q.codes);
        L.scales = q.scales;
        L.x = static_cast<const uint16_t*>(xs[p0 + i]) + t0 * 2 * q.m;
        L.y = reinterpret_cast<float*>(reinterpret_cast<char*>(ys[p0 + i]) +
                                       t0 * 2 * q.n * (out_bf16 ? 2 : (int64_t)sizeof(float)));
        L.out_bf16 = out_bf16 ? 1 : 0;
        L.n = (int32_t)q.n;
        L.m = (int32_t)q.m;
        L.tiles = (int32_t)f2i::l3_tiles(q.n);
        L.windows = (int32_t)f2i::l3_windows(q.m);
        L.unit_begin = (int32_t)units;
        L.part_begin = part;
        units += (int64_t)L.tiles * L.windows;
        if (L.windows > 1) {
          f2i::LutReduceProblem& Rp = RP.p[RP.count++];
          Rp.y = L.y;
          Rp.out_bf16 = L.out_bf16;
          Rp.part = P.partials + part;
          Rp.n = L.n;
          Rp.tiles = L.tiles;
          Rp.windows = L.windows;
          Rp.row_begin = (int32_t)rrows;
          rrows += 32 * (int64_t)L.tiles;
          part += (int64_t)L.tiles * L.windows * mc * 32;
        }
      }
      if (units > INT32_MAX / 2 || rrows > INT32_MAX / 32)
        return fail(FAIRY2I_ERR_UNSUPPORTED, "too many units for one launch");
      P.total_units = (int32_t)units;
      const int ctas = (int)std::min<int64_t>({units, (int64_t)sm_count(), (int64_t)f2i::kLutMaxCtas});
      // cost-balanced split of the units, in order: CTA c starts at the first
      // unit whose preceding cost reaches c / ctas of the total (costs are
      // constant inside a (layer, window), so each boundary is one division)
      int64_t total = 0;
      for (int i = 0; i < cnt; ++i) {
        const f2i::LutProblem& L = P.p[i];
        for (int w = 0; w < L.windows; ++w) total += (int64_t)L.tiles * (8 * f2i::l3_slots(L.m, w) + 3);
      }
      int c = 1;
      int64_t before = 0;
      P.cta_begin[0] = 0;
      for (int i = 0; i < cnt && c < ctas; ++i) {
        const f2i::LutProblem& L = P.p[i];
        for (int w = 0; w < L.windows && c < ctas; ++w) {
          const int64_t cost = 8 * f2i::l3_slots(L.m, w) + 3;
          while (c < ctas) {
            const int64_t need = total * c - before * ctas;  // k * cost * ctas >= need
            const int64_t k = need <= 0 ? 0 : (need + cost * ctas - 1) / (cost * ctas);
            if (k >= L.tiles) break;
            P.cta_begin[c++] = L.unit_begin + w * L.tiles + (int32_t)k;
          }
          before += (int64_t)L.tiles * cost;
        }
      }
      while (c < ctas) P.cta_begin[c++] = (int32_t)units;
      P.cta_begin[ctas] = (int32_t)units;
      // every CTA's first batch of segments (runs of units inside one (layer,
      // window)), as the kernel would find them: up to two for one token, one
      // otherwise (the tables of that many windows fit the shared memory)
      const int nseg_max = mc == 1 ? 2 : 1;
      for (int cc = 0; cc < ctas; ++cc) {
        int uu = P.cta_begin[cc];
        const int u_end = P.cta_begin[cc + 1];
        int k = 0;
        while (k < nseg_max && uu < u_end) {
          int i = 0;
          while (i + 1 < cnt && uu >= P.p[i + 1].unit_begin) ++i;
          const f2i::LutProblem& L = P.p[i];
          const int w = (uu - L.unit_begin) / L.tiles;
          f2i::LutSeg& g = P.first[cc][k];
          g.unit = uu;
          g.tau0 = uu - L.unit_begin - w * L.tiles;
          g.win = (uint16_t)w;
          g.prob = (uint8_t)i;
          g.nb = (uint8_t)f2i::l3_slots(L.m, w);
          uu = std::min(u_end, L.unit_begin + (w + 1) * L.tiles);
          ++k;
        }
        if (k == 0) {  // an empty range: the prefetch reads segment 0's layer and window
          P.first[cc][0] = f2i::LutSeg{u_end, 0, 0, 0, 0};
        }
        P.first_nseg[cc] = (uint8_t)k;
        P.first_end[cc] = uu;
      }
      fairy2i_status st = launch_lut(P, T, mc, ctas, s);
      if (st != FAIRY2I_OK) return st;
      if (RP.count > 0) {
        RP.total_rows = (int32_t)rrows;
        const int64_t work = rrows * mc * 4;
        const int rgrid = (int)std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, 8 * (int64_t)sm_count()));
        // an ordinary launch: the decode's CTAs hold a whole SM each, so an early
        // (programmatic) launch only parks the reduction's CTAs on the SMs the
        // decode leaves, and measured slower (about 1 us per launch pair)
        f2i::lut_reduce_kernel<<<rgrid, 256, 0, s>>>(RP);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "table-lookup reduction launch: %s", cudaGetErrorString(e));
        st = check_launch("table-lookup reduction launch");
        if (st != FAIRY2I_OK) return st;
      }
    }
  }
  return ok();
}

// with_ws: the call came through a *_ws entry point (workspace may still be
// NULL when none is needed).
// out_bf16: y holds bfloat16 elements (layout 3 only).
fairy2i_status linear_group_impl(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int32_t count,
                                 int64_t M, fairy2i_algo algo, bool with_ws, void* ws, size_t ws_bytes,
                                 cudaStream_t s, bool out_bf16 = false) {
  if (count < 1 || count > 256) return fail(FAIRY2I_ERR_INVALID_ARG, "count=%d outside [1, 256]", count);
  if (!qs || !xs || !ys) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL array argument");
  if (M < 0) return fail(FAIRY2I_ERR_SHAPE, "M=%lld is negative", (long long)M);
  if ((int)algo < 0 || (int)algo > 7) return fail(FAIRY2I_ERR_INVALID_ARG, "unknown algo %d", (int)algo);
  if (!qs) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL descriptor array");
  const int T = qs[0].T;
  for (int i = 0; i < count; ++i) {
    fairy2i_status st = check_packed(&qs[i]);
    if (st != FAIRY2I_OK) return st;
    if (qs[i].T != T) return fail(FAIRY2I_ERR_SHAPE, "all layers of a group need the same T");
    if (qs[i].version != qs[0].version) return fail(FAIRY2I_ERR_SHAPE, "all layers of a group need the same layout");
  }
  if (qs[0].version == FAIRY2I_LAYOUT_LUT) {
    if (algo != FAIRY2I_ALGO_AUTO && algo != FAIRY2I_ALGO_LUT && algo != FAIRY2I_ALGO_TCGEN05_DQ &&
        algo != FAIRY2I_ALGO_TCGEN05_DQ16)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "layout 3 is read by the table-lookup decode and the dequantized GEMM only");
    if (T > 4) return fail(FAIRY2I_ERR_UNSUPPORTED, "layout 3 kernels support T <= 4");
    bool m_mult8_3 = true;
    for (int i = 0; i < count; ++i) m_mult8_3 = m_mult8_3 && (qs[i].m % 8) == 0;
    // AUTO: with a workspace, the table lookup below kDqMinTokens tokens and the
    // fp16 dequantized GEMM from there; without one, the bfloat16 dequantized GEMM
    fairy2i_algo a3 = algo;
    if (a3 == FAIRY2I_ALGO_AUTO) {
      if (!m_mult8_3 || (with_ws && M < kDqMinTokens)) a3 = FAIRY2I_ALGO_LUT;
      else a3 = with_ws ? FAIRY2I_ALGO_TCGEN05_DQ16 : FAIRY2I_ALGO_TCGEN05_DQ;
    }
    if ((a3 == FAIRY2I_ALGO_LUT || a3 == FAIRY2I_ALGO_TCGEN05_DQ16) && !with_ws)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "the table-lookup decode and the fp16 dequantized GEMM need a workspace: "
                                           "call fairy2i_linear_ws / fairy2i_linear_group_ws");
    if ((a3 == FAIRY2I_ALGO_TCGEN05_DQ || a3 == FAIRY2I_ALGO_TCGEN05_DQ16) && !m_mult8_3)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "the dequantized GEMM needs m to be a multiple of 8");
    if (M == 0) return ok();
    for (int i = 0; i < count; ++i) {
      if (!xs[i] || !ys[i]) return fail(FAIRY2I_ERR_INVALID_ARG, "x or y of layer %d is NULL", i);
      if (!aligned(xs[i], 16) || !aligned(ys[i], 16))
        return fail(FAIRY2I_ERR_INVALID_ARG, "x and y must be 16-byte aligned (layer %d)", i);
    }
    if (M > (int64_t)1 << 30) return fail(FAIRY2I_ERR_UNSUPPORTED, "M=%lld too large", (long long)M);
    if (a3 == FAIRY2I_ALGO_TCGEN05_DQ) return run_dq(qs, xs, ys, count, M, T, s, false, nullptr, 0, out_bf16);
    if (a3 == FAIRY2I_ALGO_TCGEN05_DQ16) return run_dq(qs, xs, ys, count, M, T, s, true, ws, ws_bytes, out_bf16);
    return run_lut(qs, xs, ys, count, M, T, ws, ws_bytes, s, out_bf16);
  }
  if (out_bf16) return fail(FAIRY2I_ERR_UNSUPPORTED, "bfloat16 outputs are written by the layout-3 kernels only");
  if (algo == FAIRY2I_ALGO_LUT || algo == FAIRY2I_ALGO_TCGEN05_DQ || algo == FAIRY2I_ALGO_TCGEN05_DQ16)
    return fail(FAIRY2I_ERR_UNSUPPORTED, "the table-lookup decode and the dequantized GEMM read layout 3 only");
  (void)ws;
  (void)ws_bytes;
  if (M == 0) return ok();  // no tokens: nothing is read or written
  for (int i = 0; i < count; ++i) {
    if (!xs[i] || !ys[i]) return fail(FAIRY2I_ERR_INVALID_ARG, "x or y of layer %d is NULL", i);
    if (!aligned(xs[i], 16) || !aligned(ys[i], 16))
      return fail(FAIRY2I_ERR_INVALID_ARG, "x and y must be 16-byte aligned (layer %d)", i);
  }
  if (M > (int64_t)1 << 30) return fail(FAIRY2I_ERR_UNSUPPORTED, "M=%lld too large", (long long)M);

  bool m_mult8 = true;
  for (int i = 0; i < count; ++i) m_mult8 = m_mult8 && (qs[i].m % 8) == 0;
  bool offsets32 = true;
  for (int i = 0; i < count; ++i) offsets32 = offsets32 && mma_offsets_fit(qs[i]);
  fairy2i_algo a = algo;
  if (a == FAIRY2I_ALGO_AUTO) {
    if (T <= 4 && M >= kPrefillMinTokens && m_mult8) a = FAIRY2I_ALGO_TCGEN05;
    else a = (T <= 4 && offsets32) ? FAIRY2I_ALGO_MMA : FAIRY2I_ALGO_ADDSUB;
  }
  if (a == FAIRY2I_ALGO_MMA && !offsets32)
    return fail(FAIRY2I_ERR_UNSUPPORTED, "mma decode: a layer's code planes exceed 4 GB (32-bit offsets)");
  if (a == FAIRY2I_ALGO_TCGEN05_SP) {
    if (T > 4) return fail(FAIRY2I_ERR_UNSUPPORTED, "sparse tensor-core decode supports T <= 4");
    if (M > kTcDecodeMaxTokens) return fail(FAIRY2I_ERR_UNSUPPORTED, "sparse tensor-core decode supports M <= 8");
    return run_tc_decode(qs, xs, ys, count, M, T, s);
  }
  if (a == FAIRY2I_ALGO_MMA && T > 4) return fail(FAIRY2I_ERR_UNSUPPORTED, "mma decode supports T <= 4");
  if (a == FAIRY2I_ALGO_TCGEN05) {
    if (T > 4) return fail(FAIRY2I_ERR_UNSUPPORTED, "tcgen05 prefill supports T <= 4");
    if (!m_mult8) return fail(FAIRY2I_ERR_UNSUPPORTED, "tcgen05 prefill needs m to be a multiple of 8");
    if (M > ((int64_t)1 << 30) - 1) return fail(FAIRY2I_ERR_UNSUPPORTED, "M=%lld too large", (long long)M);
    return run_tcgen05(qs, xs, ys, count, M, T, s);
  }

  // Launch order: when the widest layer's staged activations would leave the
  // mma decode fewer than 16 warps per SM, layers are launched in groups of
  // equal activation width (the buffer of a launch is sized for its widest
  // layer), keeping the caller's order inside a width.
  std::vector<int> order(count);
  for (int i = 0; i < count; ++i) order[i] = i;
  bool split = false;
  if (a == FAIRY2I_ALGO_MMA) {
    const int mc = (int)std::min<int64_t>(M, mma_chunk(qs, count, T));
    split = !mma_full_sm(qs, count, T, mc);
    if (split)
      std::stable_sort(order.begin(), order.end(),
                       [&](int u, int v) { return f2i::x_stride(qs[u].m) < f2i::x_stride(qs[v].m); });
  }
  for (int b0 = 0; b0 < count;) {
    int b1 = b0 + 1;
    while (b1 < count && b1 - b0 < f2i::kMaxGroup &&
           (!split || f2i::x_stride(qs[order[b1]].m) == f2i::x_stride(qs[order[b0]].m)))
      ++b1;
    const int cnt = b1 - b0;
    std::vector<fairy2i_packed> sub(cnt);
    for (int i = 0; i < cnt; ++i) sub[i] = qs[order[b0 + i]];
    const int chunk = (a == FAIRY2I_ALGO_MMA) ? mma_chunk(sub.data(), cnt, T) : f2i::kAddSubTok * 1024;
    for (int64_t t0 = 0; t0 < M; t0 += chunk) {
      f2i::LinearGroup G;
      memset(&G, 0, sizeof(G));
      G.count = cnt;
      G.M = (int32_t)std::min<int64_t>(chunk, M - t0);
      for (int i = 0; i < cnt; ++i) {
        const int li = order[b0 + i];
        const fairy2i_packed& q = qs[li];
        f2i::LinearProblem& P = G.p[i];
        P.codes = static_cast<const uint8_t*>(q.codes);
        P.scales = q.scales;
        P.x = static_cast<const uint16_t*>(xs[li]) + t0 * 2 * q.m;
        P.y = ys[li] + t0 * 2 * q.n;
        P.n = q.n;
        P.m = q.m;
        P.T = q.T;
      }
      fairy2i_status st = (a == FAIRY2I_ALGO_MMA) ? run_mma(G, T, s) : run_addsub(G, s);
      if (st != FAIRY2I_OK) return st;
    }
    b0 = b1;
  }
  return ok();
}

__device__ unsigned int g_fairy2i_error_taken;

// Scratch of fairy2i_linear_group_static: a fixed block of device memory that
// is part of the loaded library (every device that loads it keeps these
// bytes until the process exits), for callers that cannot allocate.  It holds
// the table-lookup decode's partial outputs; every call overwrites what it
// reads, so nothing needs clearing between calls.
constexpr size_t kStaticScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) unsigned char g_fairy2i_static_scratch[kStaticScratchBytes];

// The device address of the scratch array, looked up once per device (with
// that device current) on the first call there.  In host code the array's
// name is only a stand-in for the symbol, never an address a kernel may use.
std::mutex g_static_mu;
std::vector<std::pair<int, void*>> g_static_addr;

fairy2i_status static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_static_mu);
  for (const auto& a : g_static_addr)
    if (a.first == dev) {
      *out = a.second;
      return FAIRY2I_OK;
    }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_fairy2i_static_scratch);
  if (e != cudaSuccess || ptr == nullptr)
    return fail(FAIRY2I_ERR_CUDA, "address of the static scratch: %s", cudaGetErrorString(e));
  g_static_addr.push_back({dev, ptr});
  *out = ptr;
  return FAIRY2I_OK;
}

__global__ void take_error_word_kernel() { g_fairy2i_error_taken = atomicExch(&g_fairy2i_error_word, 0u); }

}  // namespace

extern "C" {

int32_t fairy2i_layout_version(void) { return FAIRY2I_LAYOUT_VERSION; }

const char* fairy2i_last_error(void) { return g_last_error.c_str(); }

size_t fairy2i_codes_bytes(int64_t n, int64_t m, int32_t T) {
  if (n < 1 || m < 1 || T < 1 || T > FAIRY2I_MAX_T) return 0;
  return (size_t)(2 * T) * (size_t)f2i::plane_bytes(n, m);
}

size_t fairy2i_codes_bytes_layout(int64_t n, int64_t m, int32_t T, int32_t version) {
  if (n < 1 || m < 1 || T < 1 || T > FAIRY2I_MAX_T) return 0;
  if (version == FAIRY2I_LAYOUT_VERSION) return (size_t)(2 * T) * (size_t)f2i::plane_bytes(n, m);
  if (version == FAIRY2I_LAYOUT_LUT) return (size_t)f2i::l3_codes_bytes(n, m, T);
  return 0;
}

size_t fairy2i_scales_count(int64_t n, int32_t T) {
  if (n < 1 || T < 1 || T > FAIRY2I_MAX_T) return 0;
  return (size_t)4 * (size_t)T * (size_t)n;
}

fairy2i_status fairy2i_convert(const float* R, int64_t rows, int64_t cols, void* U, void* W, void* stream) {
  NvtxRange nvtx_range("fairy2i_convert");
  if (!R || !U || !W) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL pointer argument");
  if (rows < 2 || cols < 2 || (rows & 1) || (cols & 1))
    return fail(FAIRY2I_ERR_SHAPE, "R is %lld x %lld; both dimensions must be even and >= 2", (long long)rows,
                (long long)cols);
  if (!aligned(R, 16) || !aligned(U, 16) || !aligned(W, 16))
    return fail(FAIRY2I_ERR_INVALID_ARG, "R, U and W must be 16-byte aligned");
  const int64_t n = rows / 2, m = cols / 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = sm_count() * 8;
  if ((m & 3) == 0) {
    f2i::convert_vec4_kernel<<<blocks, 256, 0, s>>>(R, n, m, static_cast<float4*>(U), static_cast<float4*>(W));
  } else {
    f2i::convert_scalar_kernel<<<blocks, 256, 0, s>>>(R, n, m, static_cast<float2*>(U), static_cast<float2*>(W));
  }
  return check_launch("convert launch");
}

fairy2i_status fairy2i_quantize(const void* U, const void* W, int64_t n, int64_t m, int32_t T,
                                const fairy2i_packed* out, void* stream) {
  NvtxRange nvtx_range("fairy2i_quantize");
  if (!U || !W) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL weight pointer");
  if (!aligned(U, 8) || !aligned(W, 8)) return fail(FAIRY2I_ERR_INVALID_ARG, "U and W must be 8-byte aligned");
  fairy2i_status st = check_packed(out);
  if (st != FAIRY2I_OK) return st;
  if (out->n != n || out->m != m || out->T != T)
    return fail(FAIRY2I_ERR_SHAPE, "descriptor (n=%lld, m=%lld, T=%d) does not match the call (n=%lld, m=%lld, T=%d)",
                (long long)out->n, (long long)out->m, out->T, (long long)n, (long long)m, T);
  if (n > INT32_MAX) return fail(FAIRY2I_ERR_UNSUPPORTED, "n too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_quantize(static_cast<const float2*>(U), static_cast<const float2*>(W), nullptr, n, m, T, out, s);
}

fairy2i_status fairy2i_convert_quantize(const float* R, int64_t rows, int64_t cols, int32_t T,
                                        const fairy2i_packed* out, void* stream) {
  NvtxRange nvtx_range("fairy2i_convert_quantize");
  if (!R) return fail(FAIRY2I_ERR_INVALID_ARG, "R is NULL");
  if (rows < 2 || cols < 2 || (rows & 1) || (cols & 1))
    return fail(FAIRY2I_ERR_SHAPE, "R is %lld x %lld; both dimensions must be even and >= 2", (long long)rows,
                (long long)cols);
  if (!aligned(R, 8)) return fail(FAIRY2I_ERR_INVALID_ARG, "R must be 8-byte aligned");
  fairy2i_status st = check_packed(out);
  if (st != FAIRY2I_OK) return st;
  const int64_t n = rows / 2, m = cols / 2;
  if (out->n != n || out->m != m || out->T != T)
    return fail(FAIRY2I_ERR_SHAPE, "descriptor (n=%lld, m=%lld, T=%d) does not match R (n=%lld, m=%lld, T=%d)",
                (long long)out->n, (long long)out->m, out->T, (long long)n, (long long)m, T);
  if (n > 65535) return fail(FAIRY2I_ERR_UNSUPPORTED, "n=%lld above 65535 for the fused path", (long long)n);
  return launch_quantize(nullptr, nullptr, R, n, m, T, out, static_cast<cudaStream_t>(stream));
}

fairy2i_status fairy2i_linear_ex(const fairy2i_packed* q, const void* x, int64_t M, float* y, fairy2i_algo algo,
                                 void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_ex");
  if (!q) return fail(FAIRY2I_ERR_INVALID_ARG, "packed descriptor is NULL");
  const void* xs[1] = {x};
  float* ys[1] = {y};
  return linear_group_impl(q, xs, ys, 1, M, algo, false, nullptr, 0, static_cast<cudaStream_t>(stream));
}

// Layout-3 descriptors the workspace kernels accept (same T <= 4, n, m >= 1).
bool ws_layers_ok(const fairy2i_packed* qs, int32_t count, int64_t M) {
  if (!qs || count < 1 || count > 256 || M < 1) return false;
  for (int i = 0; i < count; ++i)
    if (qs[i].version != FAIRY2I_LAYOUT_LUT || qs[i].T < 1 || qs[i].T > 4 || qs[i].T != qs[0].T || qs[i].n < 1 ||
        qs[i].m < 1)
      return false;
  return true;
}

size_t fairy2i_linear_workspace_bytes(const fairy2i_packed* qs, int32_t count, int64_t M) {
  if (!ws_layers_ok(qs, count, M)) return 0;
  bool m_mult8 = true;
  for (int i = 0; i < count; ++i) m_mult8 = m_mult8 && (qs[i].m % 8) == 0;
  const size_t lut = lut_workspace(qs, count, M, qs[0].T);
  return m_mult8 ? std::max(lut, dq16_workspace(qs, count, M)) : lut;
}

fairy2i_status fairy2i_linear_ws(const fairy2i_packed* q, const void* x, int64_t M, float* y, fairy2i_algo algo,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_ws");
  if (!q) return fail(FAIRY2I_ERR_INVALID_ARG, "packed descriptor is NULL");
  const void* xs[1] = {x};
  float* ys[1] = {y};
  return linear_group_impl(q, xs, ys, 1, M, algo, true, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

fairy2i_status fairy2i_linear_group_ws(const fairy2i_packed* qs, const void* const* xs, float* const* ys,
                                       int32_t count, int64_t M, fairy2i_algo algo, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_group_ws");
  return linear_group_impl(qs, xs, ys, count, M, algo, true, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(stream));
}

fairy2i_status fairy2i_linear_group_ws_out(const fairy2i_packed* qs, const void* const* xs, void* const* ys,
                                           int32_t count, int64_t M, fairy2i_algo algo, fairy2i_out out,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_group_ws_out");
  if (out != FAIRY2I_OUT_F32 && out != FAIRY2I_OUT_BF16)
    return fail(FAIRY2I_ERR_INVALID_ARG, "unknown output type %d", (int)out);
  return linear_group_impl(qs, xs, reinterpret_cast<float* const*>(ys), count, M, algo, true, workspace,
                           workspace_bytes, static_cast<cudaStream_t>(stream), out == FAIRY2I_OUT_BF16);
}

fairy2i_status fairy2i_linear_group_static(const fairy2i_packed* qs, const void* const* xs, float* const* ys,
                                           int32_t count, int64_t M, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_group_static");
  if (!qs || count < 1 || count > 256) return fail(FAIRY2I_ERR_INVALID_ARG, "bad descriptor array or count");
  for (int i = 0; i < count; ++i)
    if (qs[i].version != FAIRY2I_LAYOUT_LUT)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "the static-scratch decode reads layout %d (layer %d is %d)",
                  FAIRY2I_LAYOUT_LUT, i, qs[i].version);
  const size_t need = ws_layers_ok(qs, count, M) ? lut_workspace(qs, count, M, qs[0].T) : 0;
  if (need > kStaticScratchBytes)
    return fail(FAIRY2I_ERR_UNSUPPORTED,
                "these layers need %zu bytes of scratch, more than the %zu bytes this entry point holds; "
                "use fairy2i_linear_group_ws with a workspace, or fewer layers or tokens per call",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  fairy2i_status st = static_scratch_address(&scratch);
  if (st != FAIRY2I_OK) return st;
  return linear_group_impl(qs, xs, ys, count, M, FAIRY2I_ALGO_LUT, true, scratch, kStaticScratchBytes,
                           static_cast<cudaStream_t>(stream));
}

fairy2i_status fairy2i_linear(const fairy2i_packed* q, const void* x, int64_t M, float* y, void* stream) {
  return fairy2i_linear_ex(q, x, M, y, FAIRY2I_ALGO_AUTO, stream);
}

fairy2i_status fairy2i_linear_group(const fairy2i_packed* qs, const void* const* xs, float* const* ys, int32_t count,
                                    int64_t M, fairy2i_algo algo, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_group");
  return linear_group_impl(qs, xs, ys, count, M, algo, false, nullptr, 0, static_cast<cudaStream_t>(stream));
}

fairy2i_status fairy2i_linear_grad_x(const fairy2i_packed* q, const float* gy, int64_t M, float* gx, void* stream) {
  return fairy2i_linear_grad_x_group(q, &gy, &gx, 1, M, stream);
}

fairy2i_status fairy2i_linear_grad_x_group(const fairy2i_packed* qs, const float* const* gys, float* const* gxs,
                                           int32_t count, int64_t M, void* stream) {
  NvtxRange nvtx_range("fairy2i_linear_grad_x_group");
  if (count < 1 || count > 256) return fail(FAIRY2I_ERR_INVALID_ARG, "count=%d outside [1, 256]", count);
  if (!qs || !gys || !gxs) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL array argument");
  for (int i = 0; i < count; ++i) {
    fairy2i_status st = check_packed(&qs[i]);
    if (st != FAIRY2I_OK) return st;
    if (qs[i].T != qs[0].T) return fail(FAIRY2I_ERR_SHAPE, "all layers of a group need the same T");
    if (qs[i].version != FAIRY2I_LAYOUT_VERSION)
      return fail(FAIRY2I_ERR_UNSUPPORTED, "the input gradient reads layout %d only", FAIRY2I_LAYOUT_VERSION);
  }
  if (M < 0) return fail(FAIRY2I_ERR_SHAPE, "M=%lld is negative", (long long)M);
  if (M == 0) return ok();
  for (int i = 0; i < count; ++i) {
    if (!gys[i] || !gxs[i]) return fail(FAIRY2I_ERR_INVALID_ARG, "NULL gradient pointer (layer %d)", i);
    if (!aligned(gys[i], 16) || !aligned(gxs[i], 16))
      return fail(FAIRY2I_ERR_INVALID_ARG, "gy and gx must be 16-byte aligned (layer %d)", i);
  }
  const int64_t pairs = (M + 1) / 2;  // tokens go two per CTA (one when M = 1)
  if (M > f2i::kGxMaxTokens) return fail(FAIRY2I_ERR_UNSUPPORTED, "M=%lld above %d", (long long)M, f2i::kGxMaxTokens);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int b0 = 0; b0 < count; b0 += f2i::kGxMaxGroup) {
    const int cnt = std::min(f2i::kGxMaxGroup, count - b0);
    f2i::GradGroup G;
    memset(&G, 0, sizeof(G));
    G.count = cnt;
    G.T = qs[0].T;
    G.M = (int32_t)M;
    int64_t blocks = 0;  // column blocks of the launch: one grid column each
    for (int i = 0; i < cnt; ++i) {
      const fairy2i_packed& q = qs[b0 + i];
      f2i::GradProblem& P = G.p[i];
      P.codes = static_cast<const uint8_t*>(q.codes);
      P.scales = q.scales;
      P.g = gys[b0 + i];
      P.gx = gxs[b0 + i];
      P.n = q.n;
      P.m = q.m;
      P.kb_begin = (int32_t)blocks;
      blocks += f2i::col_blocks(q.m);
    }
    const dim3 grid((unsigned)blocks, (unsigned)(pairs * f2i::kGxCluster));
    if (M == 1) f2i::linear_grad_x_kernel<1><<<grid, f2i::kGxWarps * 32, 0, s>>>(G);
    else f2i::linear_grad_x_kernel<2><<<grid, f2i::kGxWarps * 32, 0, s>>>(G);
    fairy2i_status st = check_launch("input-gradient launch");
    if (st != FAIRY2I_OK) return st;
  }
  return ok();
}

fairy2i_status fairy2i_unpack_codes(const fairy2i_packed* q, uint8_t* codes_out, void* stream) {
  NvtxRange nvtx_range("fairy2i_unpack_codes");
  fairy2i_status st = check_packed(q);
  if (st != FAIRY2I_OK) return st;
  if (!codes_out) return fail(FAIRY2I_ERR_INVALID_ARG, "codes_out is NULL");
  if (q->version == FAIRY2I_LAYOUT_LUT)
    f2i::unpack_codes_l3_kernel<<<sm_count() * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(q->codes), q->n, q->m, q->T, codes_out);
  else
    f2i::unpack_codes_kernel<<<sm_count() * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(q->codes), q->n, q->m, q->T, codes_out);
  return check_launch("unpack launch");
}

fairy2i_status fairy2i_selftest_bounded_wait(int32_t limit_us, void* stream) {
  NvtxRange nvtx_range("fairy2i_selftest_bounded_wait");
  if (limit_us < 1 || limit_us > 1000000) return fail(FAIRY2I_ERR_INVALID_ARG, "limit_us=%d outside [1, 1000000]", limit_us);
  f2i::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000ull);
  return check_launch("bounded-wait self-test launch");
}

fairy2i_status fairy2i_sync_status(void* stream) {
  NvtxRange nvtx_range("fairy2i_sync_status");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  // read and clear in one atomic step on the device, so that a flag raised by
  // a kernel on another stream in between is kept for the next call
  take_error_word_kernel<<<1, 1, 0, s>>>();
  unsigned word = 0;
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&word, g_fairy2i_error_taken, sizeof(word), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(FAIRY2I_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
  if (word & f2i::kErrNonFinite) return fail(FAIRY2I_ERR_NONFINITE, "non-finite weight seen by quantize");
  if (word & f2i::kErrTimeout) return fail(FAIRY2I_ERR_TIMEOUT, "a bounded device wait gave up");
  if (word & f2i::kErrConfig) return fail(FAIRY2I_ERR_CUDA, "a kernel refused its shared-memory placement");
  return ok();
}

}  // extern "C"
