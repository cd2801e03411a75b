/*
 * fairy2i.h -- C ABI of the Fairy2i widely-linear 2-bit complex linear layer
 * for NVIDIA B300 (sm_103a).
 *
 * The layer ("Fairy2i-W2" model card, section "Widely-linear transformation";
 * "Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights {±1, ±i}",
 * Step 1) is
 *
 *        y = U x + W conj(x),      U, W complex n x m,  x complex m-vector,
 *
 * the exact complex rewrite of a real PyTorch-style linear weight R of shape
 * [2n, 2m] acting on the real activation row [Re x | Im x].  U and W are each
 * stored as T recursive-residual stages (same page, Step 3) of 2-bit phase
 * codes in {+1, -1, +i, -i} (Step 2) with one real-axis and one
 * imaginary-axis scale per output row and stage.
 *
 * Conventions for every call:
 *   - Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *     allocated and owned by the caller.  The library allocates nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream: the returned status
 *     covers argument checks and the kernel launch only.
 *   - Errors a kernel detects (non-finite weights, a bounded wait that gave
 *     up) set a per-device error word that fairy2i_sync_status() reads.
 *   - On any status other than FAIRY2I_OK nothing was launched (or the launch
 *     failed) and fairy2i_last_error() returns a message for this thread.
 *   - Layouts are row-major (C order).
 */
#ifndef FAIRY2I_H
#define FAIRY2I_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FAIRY2I_OK = 0,
    FAIRY2I_ERR_INVALID_ARG = 1, /* null or misaligned pointer, negative size, bad enum */
    FAIRY2I_ERR_SHAPE = 2,       /* odd real dimension, empty matrix, size mismatch */
    FAIRY2I_ERR_NONFINITE = 3,   /* NaN or Inf among the weights given to quantize */
    FAIRY2I_ERR_UNSUPPORTED = 4, /* T outside [1, 8], m above 16384, token count too large */
    FAIRY2I_ERR_CUDA = 5,        /* a CUDA call failed; see fairy2i_last_error() */
    FAIRY2I_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} fairy2i_status;

#define FAIRY2I_LAYOUT_VERSION 2
#define FAIRY2I_LAYOUT_LUT 3
#define FAIRY2I_MAX_T 8
#define FAIRY2I_MAX_M 16384

/* Packed quantized layer (both U and W).
 *
 * codes: FAIRY2I_LAYOUT_VERSION 2 layout, fairy2i_codes_bytes(n, m, T)
 *   bytes, 256-byte aligned.  2T code planes, plane (X, t) for X = 0 (U),
 *   1 (W) at byte offset (X*T + t) * plane_bytes with plane_bytes =
 *   ceil(n/16) * ceil(m/64) * 256.  Inside a plane, rows come in tiles of 16
 *   and columns in blocks of 64; each (row tile, column block) holds 32 lanes
 *   (g, q) = 4g + q of two little-endian 32-bit words: a sign word (bit set =
 *   the code is -1 or -i) and an axis-flag word (bit set = the code is +i or
 *   -i).  Lane (g, q) carries rows g and g + 8 of the tile:
 *     sign of (row 8 rho + g, column 16 s + 8 h + 2 q + e) at bit
 *       15 + 16 e - (4 s + 2 h + rho) of the sign word of lane (g, q);
 *     flag of (row 8 rho + g, column 16 s + 8 h + 2 q' + e) at bit
 *       4 (q' + 4 rho) + (s & 1) + 2 e of the flag word of lane
 *       (g, h + 2 (s >> 1)).
 *   Blocks are stored in chunks of two so that a lane's words of two
 *   consecutive blocks are 16 contiguous bytes (an odd last block stores 8
 *   bytes per lane).  Padding rows and columns hold zero bits.  The layout is
 *   opaque to callers; fairy2i_unpack_codes() gives the canonical view.
 * scales: fairy2i_scales_count(n, T) floats, [2 (U, W)][T][2 (real axis,
 *   imaginary axis)][n], 16-byte aligned.
 *
 * codes, FAIRY2I_LAYOUT_LUT (version 3), the table-lookup decode layout:
 *   fairy2i_codes_bytes_layout(n, m, T, 3) bytes, 256-byte aligned.  Per
 *   (row, group of 8 columns) a sign byte (bit c: the code of column 8 G + c
 *   is -1 or -i) and a q byte (sign XOR imaginary-axis flag).  Rows in tiles
 *   of 32 (row 32 tau + r), columns in windows of 256; a window stores nb
 *   slots of 512 bytes (nb = 4, or 1, 2 or 4 for a last partial window; 3 is
 *   padded to 4), each 32 rows x (8 sign bytes, 8 q bytes).  Byte i of row r
 *   in slot jj holds group (r & (8 nb - 1)) ^ (8 jj + i) of the window.
 *   Order: [window][row tile][plane (X * T + t)][slot][row][16 bytes], so
 *   window w, tile tau, plane p starts at byte w * tiles * 2T * 2048 +
 *   (tau * 2T + p) * nb * 512.  Padding rows and columns hold zero bits.
 *   Scales as for version 2.  Read by the table-lookup decode
 *   (FAIRY2I_ALGO_LUT, through fairy2i_linear_ws / fairy2i_linear_group_ws)
 *   and by fairy2i_unpack_codes; written by fairy2i_quantize and
 *   fairy2i_convert_quantize when out->version is 3. */
typedef struct {
    int32_t version; /* FAIRY2I_LAYOUT_VERSION (2) or FAIRY2I_LAYOUT_LUT (3) */
    int32_t T;       /* number of residual stages, 1..FAIRY2I_MAX_T */
    int64_t n;       /* complex output rows (real rows 2n) */
    int64_t m;       /* complex input columns (real columns 2m), 1..FAIRY2I_MAX_M */
    void *codes;     /* device, caller-owned */
    float *scales;   /* device, caller-owned */
} fairy2i_packed;

/* Algorithm choice for fairy2i_linear_ex / fairy2i_linear_group. */
typedef enum {
    FAIRY2I_ALGO_AUTO = 0,    /* pick the fastest kernel for the token count */
    FAIRY2I_ALGO_ADDSUB = 1,  /* CUDA cores: adds/subtracts only, fp32 accumulation */
    FAIRY2I_ALGO_MMA = 2,     /* decode: 2:4-sparse mma.sync, signs as bf16 +-2, axis flags as metadata */
    FAIRY2I_ALGO_TCGEN05 = 3, /* prefill: codes staged in shared memory by the TMA engine, expanded
                                 there to ternary bf16 rows ({+-2, +-0}: the factor 2 leaves with
                                 the scales), tcgen05.mma, scales in the epilogue */
    FAIRY2I_ALGO_TCGEN05_SP = 4, /* decode, M <= 8, T <= 4: 2:4-sparse tcgen05.mma.sp (e4m3 signs and axis
                                   flags as metadata in tensor memory; x as two exact e4m3 terms) */
    FAIRY2I_ALGO_LUT = 5,     /* layout 3, T <= 4: per window of 256 columns and token, tables of the
                                 256 signed sums of every 8 activations (fp16 entries, each the fp32 sum
                                 rounded once, activations scaled by a power of two per window); per
                                 code byte one shared-memory lookup and two fp32 adds */
    FAIRY2I_ALGO_TCGEN05_DQ = 6, /* layout 3, T <= 4, m a multiple of 8: tcgen05 GEMM of the dequantized
                                 real matrix (Theorem 1 rebuilt from the summed stages) as two bfloat16
                                 terms hi + lo against x; codes staged in shared memory by the TMA
                                 engine; no workspace */
    FAIRY2I_ALGO_TCGEN05_DQ16 = 7 /* as TCGEN05_DQ with one fp16 term (rows scaled by powers of two)
                                 against an fp16 copy of x scaled per token by a power of two (made
                                 in the workspace by a conversion kernel): half the MMAs and A
                                 bytes; fairy2i_linear_ws / fairy2i_linear_group_ws only */
} fairy2i_algo;

/* Bytes of the code planes of an n x m layer with T stages in layout
 * version 2 (0 on bad input). */
size_t fairy2i_codes_bytes(int64_t n, int64_t m, int32_t T);

/* Bytes of the code planes in layout `version` (2 or 3); 0 on bad input. */
size_t fairy2i_codes_bytes_layout(int64_t n, int64_t m, int32_t T, int32_t version);

/* Number of fp32 scales, 4 * T * n (0 on bad input). */
size_t fairy2i_scales_count(int64_t n, int32_t T);

/* Widely-linear conversion (Theorem 1; "Fairy2i: Ultra-Low-Bit ...", Step 1):
 *   Re U = (R11 + R22)/2, Im U = (R21 - R12)/2,
 *   Re W = (R11 - R22)/2, Im W = (R12 + R21)/2,
 * R11 = R[0:n, 0:m], R12 = R[0:n, m:2m], R21 = R[n:2n, 0:m], R22 = R[n:2n, m:2m].
 *   R      : device float32 [rows][cols] = [2n][2m], 16-byte aligned
 *   U, W   : device complex64 (float32 re, im pairs) [n][m], 16-byte aligned
 * Each output is the float32 sum rounded once, then halved (exact).
 * Errors: FAIRY2I_ERR_SHAPE for odd or non-positive rows/cols; INVALID_ARG for
 * null or misaligned pointers. */
fairy2i_status fairy2i_convert(const float *R, int64_t rows, int64_t cols,
                               void *U, void *W, void *stream);

/* Phase-aware recursive residual quantization ("Fairy2i: Ultra-Low-Bit ...",
 * Step 2 and Step 3; "Fairy2i-W2" card, "Phase-aware complex quantization",
 * "Recursive residual quantization").  For each of U and W separately,
 * r^(0) = the matrix, and for t = 0..T-1:
 *   code   = argmax over s in {+1,-1,+i,-i} of Re(r conj(s)), first maximum
 *            in that order (so |Re r| >= |Im r| picks the real axis);
 *   s_re   = mean |Re r| over the row's real-coded entries, s_im = mean |Im r|
 *            over its imaginary-coded entries (0 if none), computed exactly
 *            (64-bit integer sum of |v| * 2^(48-e), e the exponent of the
 *            row-axis maximum, then one double division, rounded to float);
 *   r     <- r - (s_re b_re + i s_im b_im), float32, one rounding.
 *   U, W   : device complex64 [n][m] (e.g. from fairy2i_convert)
 *   out    : host descriptor; out->n, out->m, out->T, out->version must match
 *            the call, out->codes and out->scales receive the result.
 * Non-finite weights set FAIRY2I_ERR_NONFINITE in the device error word
 * (read it with fairy2i_sync_status); the codes are then unspecified.
 * Errors: SHAPE (n, m < 1 or descriptor mismatch), UNSUPPORTED (T outside
 * [1, 8] or m > 16384), INVALID_ARG (null/misaligned pointers). */
fairy2i_status fairy2i_quantize(const void *U, const void *W, int64_t n, int64_t m,
                                int32_t T, const fairy2i_packed *out, void *stream);

/* Conversion and quantization in one pass: the same codes and scales as
 * fairy2i_convert followed by fairy2i_quantize, bit for bit (each weight of U
 * and W is formed from R with the conversion's float32 operations), without
 * writing U and W to memory.
 *   R   : device float32 [rows][cols] = [2n][2m], 8-byte aligned
 *   out : host descriptor with out->n = rows/2, out->m = cols/2, out->T = T
 * Errors: as fairy2i_convert and fairy2i_quantize; UNSUPPORTED for n > 65535. */
fairy2i_status fairy2i_convert_quantize(const float *R, int64_t rows, int64_t cols, int32_t T,
                                        const fairy2i_packed *out, void *stream);

/* The layer on a batch of tokens ("Fairy2i-W2" card, y = Ux + W conj(x);
 * "Fairy2i: Ultra-Low-Bit ...", "Industry implications: multiplication-free
 * inference"):
 *   y = sum over stages t of  [ s_re A_re + i s_im A_im ]_U
 *                           + [ s_re conj(A_re) + i s_im conj(A_im) ]_W,
 * A_re = (signed) sum of x over real-coded columns, A_im over
 * imaginary-coded columns.
 *   x : device bfloat16 [M][2m], each token's row is [Re x | Im x] (the real
 *       activation row of the original layer), 16-byte aligned
 *   y : device float32 [M][2n], each row [Re y | Im y], 16-byte aligned
 * M = 0 is a no-op.  fairy2i_linear uses FAIRY2I_ALGO_AUTO.
 * Errors: INVALID_ARG (null/misaligned/bad version), SHAPE, UNSUPPORTED. */
fairy2i_status fairy2i_linear(const fairy2i_packed *q, const void *x, int64_t M,
                              float *y, void *stream);
fairy2i_status fairy2i_linear_ex(const fairy2i_packed *q, const void *x, int64_t M,
                                 float *y, fairy2i_algo algo, void *stream);

/* Several independent layers evaluated by one launch (same token count M,
 * each with its own x and y), e.g. the seven projections of a decoder block.
 * qs, xs, ys are HOST arrays of `count` entries (1..256). */
fairy2i_status fairy2i_linear_group(const fairy2i_packed *qs, const void *const *xs,
                                    float *const *ys, int32_t count, int64_t M,
                                    fairy2i_algo algo, void *stream);

/* Layout-3 layers through fairy2i_linear / _ex / _group (no workspace) take
 * the dequantized GEMM (FAIRY2I_ALGO_TCGEN05_DQ; "Fairy2i: Ultra-Low-Bit ...",
 * Step 3: the stages add up to one matrix, and Step 1: its real form); with a
 * workspace (the *_ws calls below) AUTO takes the table-lookup decode below 10
 * tokens and the fp16 dequantized GEMM (FAIRY2I_ALGO_TCGEN05_DQ16) from 10
 * tokens.  The dequantized GEMM needs m a multiple of 8 (x is read by TMA in
 * two halves, Re x and Im x), so other layout-3 layers return UNSUPPORTED here
 * and go through the *_ws calls.
 * Precision (TCGEN05_DQ): the summed matrix is formed in fp32 and carried as
 * two bfloat16 terms (<= 2^-18 relative per entry), products are exact and
 * sums are fp32: about 1e-5 relative (L2) against the exact sum.
 * Precision (TCGEN05_DQ16): each row of the summed matrix is scaled by a power
 * of two and rounded once to fp16 (<= 2^-11 relative per entry); each token of
 * x is scaled by a power of two into fp16, exactly for every value at or above
 * 2^-31 of the token's largest; products are exact, sums fp32, and both
 * powers of two are undone on the fp32 result: about 3e-4 relative (L2) for
 * Gaussian weights.  Precision drops for weight scales below 2^-53 or above
 * 2^75 and for tokens whose largest magnitude is below 2^-50 (the powers of
 * two are clamped to 2^+-64); a token with Inf or NaN gives non-finite outputs.
 * Tokens run in tiles of min(256, M rounded up to 16); the codes are decoded
 * once per token tile. */

/* The layer through the table-lookup decode (same y as fairy2i_linear; "Fairy2i:
 * Ultra-Low-Bit ...", "Industry implications: multiplication-free inference":
 * each code contributes a signed activation, here eight codes at a time read
 * from a table of signed sums).  For layout-3 descriptors (all layers of a
 * group the same layout and T <= 4); layout-2 descriptors are evaluated as by
 * fairy2i_linear_ex / fairy2i_linear_group and the workspace is unused.
 *   workspace : device, caller-owned scratch of at least
 *               fairy2i_linear_workspace_bytes(qs, count, M) bytes, 256-byte
 *               aligned, any contents (no initialisation needed).  The table
 *               lookup keeps one fp32 partial output per (row, window of 256
 *               columns, token) there; a second kernel sums every row's
 *               partials in window order, so results are deterministic.  The
 *               fp16 dequantized GEMM keeps the fp16 copy of x (4 m bytes per
 *               token and layer) and the tokens' powers of two there.  Calls
 *               that may run at the same time need separate workspaces.  NULL
 *               is allowed when the size query returns 0.
 * The decode kernel is launched as a programmatic dependent of the preceding
 * work in the stream (it may start while that work finishes and waits for it
 * before reading activations or writing anything); the summing kernel is an
 * ordinary launch after it.  The fp16 dequantized GEMM is an ordinary
 * conversion launch and then the GEMM as its programmatic dependent (only the
 * GEMM's reads of the converted activations wait for the conversion).
 * Tokens go in launches of 2 (T <= 2; the first of 3 when M is odd and at
 * least 3), 2 (T = 3) or 1 (T = 4); each launch streams the codes once.  Precision: each table entry is the fp32 sum
 * of 8 scaled activations rounded once to fp16 (relative error <= 2^-11 per
 * entry), accumulated in fp32; outputs agree with the exact sum to about
 * 3e-4 relative (L2) for Gaussian activations.  A token with a non-finite
 * activation gives non-finite outputs.
 * Errors: as fairy2i_linear_ex; INVALID_ARG for a missing, short or
 * misaligned workspace; UNSUPPORTED for layout 3 with another algo than AUTO,
 * LUT, TCGEN05_DQ or TCGEN05_DQ16, for T > 4, or for a dequantized GEMM with m
 * not a multiple of 8. */
fairy2i_status fairy2i_linear_ws(const fairy2i_packed *q, const void *x, int64_t M, float *y,
                                 fairy2i_algo algo, void *workspace, size_t workspace_bytes,
                                 void *stream);
fairy2i_status fairy2i_linear_group_ws(const fairy2i_packed *qs, const void *const *xs,
                                       float *const *ys, int32_t count, int64_t M,
                                       fairy2i_algo algo, void *workspace,
                                       size_t workspace_bytes, void *stream);

/* Output element type of fairy2i_linear_group_ws_out. */
typedef enum {
    FAIRY2I_OUT_F32 = 0,  /* float32, as every other linear call writes */
    FAIRY2I_OUT_BF16 = 1  /* bfloat16: the float32 result rounded once to nearest even */
} fairy2i_out;

/* fairy2i_linear_group_ws with a choice of output type, for a caller whose next
 * layer reads bfloat16 activations (the paper has no counterpart; the decoder
 * stack's activations are bfloat16 on the model card).  ys[i] is a device
 * array [M][2n] of `out` elements, 16-byte aligned.  With FAIRY2I_OUT_BF16 each
 * output is the value FAIRY2I_OUT_F32 would hold, rounded once to bfloat16
 * (relative error <= 2^-9 against it), written by the kernel that forms it:
 * no extra launch.  Layout-3 layers only.
 * Errors: as fairy2i_linear_group_ws; INVALID_ARG for an unknown `out`;
 * UNSUPPORTED for FAIRY2I_OUT_BF16 with layout-2 layers. */
fairy2i_status fairy2i_linear_group_ws_out(const fairy2i_packed *qs, const void *const *xs,
                                           void *const *ys, int32_t count, int64_t M,
                                           fairy2i_algo algo, fairy2i_out out, void *workspace,
                                           size_t workspace_bytes, void *stream);

/* Workspace bytes of fairy2i_linear_ws / fairy2i_linear_group_ws for these
 * layers and token count, enough for every algorithm those calls accept (the
 * table lookup, and for m a multiple of 8 the fp16 dequantized GEMM): 0 if
 * the descriptors are not layout 3 (or invalid). */
size_t fairy2i_linear_workspace_bytes(const fairy2i_packed *qs, int32_t count, int64_t M);

/* The table-lookup decode with no caller workspace and no allocation (the
 * paper has no counterpart: this is a deployment aid).  For callers that
 * cannot call cudaMalloc -- e.g. a plugin inside a serving process whose
 * device memory is owned by the host application's allocator, or a real-time
 * loop that forbids device allocation after start-up.  Same inputs, outputs
 * and results as fairy2i_linear_group_ws with algo LUT (layout-3 descriptors
 * only); the partial outputs go to a fixed 8 MiB array inside the library,
 * which every device that loads the library holds until the process exits.
 *   - The first call on a device looks up that array's device address (with
 *     the device current); make that first call before any stream capture.
 *   - Every call uses the same array: calls that may overlap on the GPU (other
 *     streams, other threads) race and must be serialized by the caller.
 *   - The array needs no clearing: each call writes every byte it reads.
 * Errors: as fairy2i_linear_group_ws; UNSUPPORTED for another layout or when
 * the table lookup needs more than 8 MiB of scratch for these layers (a
 * LLaMA-2-7B block needs 1.6 MB per token of a launch). */
fairy2i_status fairy2i_linear_group_static(const fairy2i_packed *qs, const void *const *xs,
                                           float *const *ys, int32_t count, int64_t M, void *stream);

/* Input gradient of the layer for training through it with the
 * straight-through estimator ("Fairy2i: Ultra-Low-Bit ...", quantization-aware
 * training; "Fairy2i-W2" card, y = Ux + W conj(x)):
 *   dL/dx = U^^H g + W^^T conj(g),   g = dL/dRe y + i dL/dIm y,
 * the transpose of the layer's real form applied to [dL/dRe y | dL/dIm y].
 * U^ and W^ are the dequantized sums of stages of q.
 *   gy : device float32 [M][2n], each row [dL/dRe y | dL/dIm y], 16-byte aligned
 *   gx : device float32 [M][2m], each row [dL/dRe x | dL/dIm x], 16-byte aligned
 * Deterministic (fixed summation order); M = 0 is a no-op.
 * Errors: INVALID_ARG (null/misaligned/bad version), SHAPE, UNSUPPORTED (M > 16382). */
fairy2i_status fairy2i_linear_grad_x(const fairy2i_packed *q, const float *gy, int64_t M, float *gx,
                                     void *stream);

/* The input gradients of several independent layers (same T and token count M,
 * each with its own gy and gx), e.g. the seven projections of a decoder block,
 * in one launch per 32 layers.  qs, gys, gxs are HOST arrays of `count`
 * entries (1..256); the per-layer arguments mean what they mean for
 * fairy2i_linear_grad_x, and each layer's gx equals that call's bit for bit.
 * Errors: as fairy2i_linear_grad_x; INVALID_ARG also for a bad count or a NULL
 * array, SHAPE for mixed T. */
fairy2i_status fairy2i_linear_grad_x_group(const fairy2i_packed *qs, const float *const *gys,
                                           float *const *gxs, int32_t count, int64_t M, void *stream);

/* Canonical view of the codes: device uint8 [2 (U, W)][T][n][m] with values
 * 0 = +1, 1 = -1, 2 = +i, 3 = -i. */
fairy2i_status fairy2i_unpack_codes(const fairy2i_packed *q, uint8_t *codes_out, void *stream);

/* Self-test of the failure-detection path: launches one thread that waits on
 * a shared-memory barrier nothing arrives at, using the same bounded wait as
 * the prefill kernel with a limit of `limit_us` microseconds (1..1000000).
 * The wait gives up, sets FAIRY2I_ERR_TIMEOUT in the device error word and
 * the kernel returns; fairy2i_sync_status() then reports FAIRY2I_ERR_TIMEOUT
 * (and clears it).  No device fault is involved.  INVALID_ARG on a bad limit. */
fairy2i_status fairy2i_selftest_bounded_wait(int32_t limit_us, void *stream);

/* Synchronize `stream`, then read and clear this device's error word.
 * Returns FAIRY2I_OK, FAIRY2I_ERR_NONFINITE, FAIRY2I_ERR_TIMEOUT or
 * FAIRY2I_ERR_CUDA. */
fairy2i_status fairy2i_sync_status(void *stream);

/* Message for the last failing call on this thread ("" if none). */
const char *fairy2i_last_error(void);

/* FAIRY2I_LAYOUT_VERSION of the library. */
int32_t fairy2i_layout_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FAIRY2I_H */
