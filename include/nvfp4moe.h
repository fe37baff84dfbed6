/*
 * nvfp4moe -- NVFP4 W4A4 mixture-of-experts expert block for GB300 (sm_103a).
 *
 * C ABI.  Every entry point takes plain pointers and sizes; no PyTorch type appears.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers; the caller owns all memory.
 *     The library never allocates or frees memory: scratch space comes from the
 *     caller's `workspace` (size from the matching *_workspace_size call).
 *   - Calls are asynchronous on `stream` (a cudaStream_t, passed as void*; NULL is the
 *     legacy default stream) and return after the kernels are enqueued.
 *   - Arguments that can be checked on the host (sizes, alignment, workspace size) are
 *     checked before anything is enqueued; a failed check returns an error code and
 *     enqueues nothing.
 *   - Errors found on the device (an expert id out of range, a device-side wait that
 *     ran out of time) are recorded in a per-device status word; nvfp4_status_check()
 *     synchronises the stream, returns and clears it.  No kernel traps.
 *   - The library resolves a few per-device addresses once (the status word, the silu
 *     table, the scratch of nvfp4_quantize_noalloc) and keeps them for the life of the
 *     device's primary context: after cudaDeviceReset the process must not call the
 *     library on that device again.
 *   - Inputs are finite; NaN or Inf inputs give unspecified (but memory-safe) results.
 *   - Results are deterministic, and a token's output bits do not depend on the other
 *     tokens of the batch (per-token activation scales, a fixed accumulation order,
 *     no split-K, no atomics on data).
 *
 * Format (pages: "The 4-bitter Lesson: Balancing Stability and Performance in NVFP4
 * RL", §Baseline): NVFP4 = 4-bit E2M1 values, one E4M3 scale per 16 consecutive
 * values along the contraction (last) dimension, one FP32 global scale per scope.
 * Storage used by this library:
 *   codes:  uint8 [rows, cols/2], two codes per byte, element 2i in the low nibble.
 *   scales: E4M3 bytes in the 128x4 tiled layout consumed by Blackwell block-scaled
 *           MMAs: tile (r/128, c/4) at byte ((r/128)*ceil(C/4) + c/4)*512, and inside a
 *           tile (r%32)*16 + ((r%128)/32)*4 + c%4, where C = cols/16 and rows are
 *           padded to a multiple of 128 (size nvfp4_sf_bytes(rows, cols)).
 *   global scale g (decode direction): DQ(x) = value(code) * decode(sf) * g.
 * Scale arithmetic, every step one float32 operation rounded to nearest even:
 *   g = amax/2688; sf = E4M3_rn_satfinite(amax_block / (6*g)); s = decode(sf)*g.
 * Element code ("The 4-bitter Lesson...", §"Improving Gradient Stability", footnote 6:
 * Q = clip(round(w/s), qmin, qmax)): round(x / s) of the exact (unrounded) quotient onto
 * the E2M1 grid, ties to the even code, saturating at +-6, or stochastic rounding of that
 * quotient; zero magnitudes encoded as +0.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,   /* null pointer, bad size or misaligned pointer */
  NVFP4_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
  NVFP4_ERR_WORKSPACE = 3,     /* workspace too small */
  NVFP4_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  NVFP4_ERR_DEVICE_STATUS = 5, /* a kernel recorded bad input (e.g. expert id out of range) */
  NVFP4_ERR_TIMEOUT = 6        /* a device-side wait ran out of time */
} nvfp4_status;

typedef enum {
  NVFP4_SCALE_PER_TENSOR = 0,  /* one g for the whole tensor (weights, standalone tensors) */
  NVFP4_SCALE_PER_ROW = 1,     /* one g per row (per token: activations) */
  NVFP4_SCALE_PER_GROUP = 2    /* one g per `group_rows` consecutive rows (stacked experts) */
} nvfp4_scale_mode;

typedef enum {
  NVFP4_ROUND_RNE = 0,         /* round to nearest, ties to even */
  NVFP4_ROUND_STOCHASTIC = 1   /* Philox4x32-10 driven stochastic rounding of the codes */
} nvfp4_rounding;

typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 } nvfp4_out_dtype;

typedef enum {
  NVFP4_SF_SWIZZLED_128x4 = 0, /* the 128x4 tiled layout the block-scaled MMAs read (above) */
  NVFP4_SF_ROWMAJOR = 1        /* plain [rows, cols/16] bytes, scale (r, c) at r*cols/16 + c */
} nvfp4_sf_layout;

/* GEMM-tiled operand layout (the layout the expert block's GEMMs read).  An NVFP4
 * operand of K columns (K % 256 == 0) is stored as blocks of R rows (R = 128 for
 * activations, 256 for weights) by 256 K-values; block (b, kb) starts at byte
 * (b * K/256 + kb) * R * 144 and holds
 *   R * 128 bytes of codes in 128-byte-swizzled K-major order: row rr of the block at
 *   rr * 128, its 16-byte chunk j at ((j ^ (rr % 8)) * 16);
 *   (R/128) * 2048 bytes of E4M3 scales: row group g = rr/128, k-group q of 64 values:
 *   a 512-byte atom at g*2048 + q*512, scale (rr, c) at (rr%32)*16 + ((rr%128)/32)*4 + c%4.
 * Each block is the exact shared-memory image of one GEMM pipeline stage, so the GEMM
 * reads it with one bulk copy.  Size: nvfp4_tiled_bytes(rows, K, R). */
size_t nvfp4_tiled_bytes(int64_t rows, int64_t K, int32_t block_rows);

/* Prepared (quantised) expert weights.  Caller-allocated device buffers, sizes from
 * moe_weights_sizes().  Both matrices are in the GEMM-tiled layout with 256-row blocks.
 * W13 rows are stored with gate and up interleaved in chunks of 64 rows ([gate 0..63,
 * up 0..63, gate 64..127, up 64..127, ...]) so that one 256-column output tile holds the
 * gate and up columns of the same 128 h columns; W2's contraction dimension is
 * zero-padded to Ip = round_up(I, 256). */
typedef struct {
  int32_t E;          /* experts */
  int64_t H;          /* hidden size (gate/up contraction, down output) */
  int64_t I;          /* intermediate size */
  uint8_t* w13;       /* device, GEMM-tiled over E*2I rows, K = H */
  float* w13_g;       /* device [E] */
  uint8_t* w2;        /* device, GEMM-tiled over E*H rows, K = Ip */
  float* w2_g;        /* device [E] */
} nvfp4_moe_weights;

/* ---------------------------------------------------------------- sizes / status */

/* Bytes of the tiled scale-factor buffer for a rows x cols NVFP4 tensor. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* Byte sizes of the four nvfp4_moe_weights buffers, in struct order
 * (w13, w13_g, w2, w2_g). */
nvfp4_status moe_weights_sizes(int32_t E, int64_t H, int64_t I, size_t sizes_out[4]);

/* Workspace bytes for each entry point (0 when none is needed).  `op` is one of: */
enum {
  NVFP4_OP_QUANTIZE = 0,        /* args: rows, cols (others 0) */
  NVFP4_OP_PREPARE_WEIGHTS = 1, /* args: E, H, I */
  NVFP4_OP_MOE_FORWARD = 2,     /* args: T, k, E, H, I */
  NVFP4_OP_MOE_PERMUTE = 3,     /* args: T, k, E */
  NVFP4_OP_QUANTIZE_T = 4,      /* args: batches * C (rows of the transpose), R */
  NVFP4_OP_MOE_BACKWARD = 5,    /* args: T, k, E, H, I */
  NVFP4_OP_PREPARE_WEIGHTS_T = 6 /* args: E */
};
size_t nvfp4_workspace_size(int op, int64_t T_or_rows, int64_t k_or_cols, int64_t E,
                            int64_t H, int64_t I);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device: NVFP4_OK, NVFP4_ERR_DEVICE_STATUS or NVFP4_ERR_TIMEOUT. */
nvfp4_status nvfp4_status_check(void* stream);

const char* nvfp4_status_string(nvfp4_status s);

/* ---------------------------------------------------------------- quantiser */

/* NVFP4 quantisation of a BF16 matrix ("The 4-bitter Lesson...", §Baseline for the
 * format; §"Why is the NVFP4 pretraining recipe not sufficient for RL?" for the
 * per-tensor weight scale, the per-token activation scale and stochastic rounding).
 *   x:            device BF16 [rows, ld_elems], the first `cols` of each row are used.
 *   rows, cols:   cols % 16 == 0, 16 <= cols <= 8192; ld_elems >= cols, ld_elems % 8 == 0.
 *   mode:         per tensor / per row / per group of `group_rows` rows.
 *   rounding:     RNE, or stochastic with (seed, rng_offset): element with row-major
 *                 index i uses 16 bits of Philox4x32-10 block rng_offset + i/8, key=seed.
 *   global_scale_in:  device, nullable.  When given, g is read from it (1, rows or
 *                 rows/group_rows floats) instead of being computed from amax.
 *   global_scale_out: device float [1 | rows | rows/group_rows], receives g.
 *   codes_out:    device uint8 [rows, cols/2] (16-byte aligned).
 *   sf_out:       device uint8, in `sf_layout`:
 *                 NVFP4_SF_SWIZZLED_128x4: [nvfp4_sf_bytes(rows, cols)] bytes, padding
 *                   rows/columns of the tile grid written as 0 (the GEMMs' input);
 *                 NVFP4_SF_ROWMAJOR: [rows, cols/16] bytes; needs cols % 64 == 0 (else
 *                   NVFP4_ERR_UNSUPPORTED).
 *   workspace:    device, nvfp4_workspace_size(NVFP4_OP_QUANTIZE, rows, cols, ...) bytes
 *                 (holds the amax of each scope for the per-tensor / per-group modes).
 */
nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_elems,
                            nvfp4_scale_mode mode, int64_t group_rows, nvfp4_rounding rounding,
                            uint64_t seed, uint64_t rng_offset, const float* global_scale_in,
                            float* global_scale_out, uint8_t* codes_out, uint8_t* sf_out,
                            nvfp4_sf_layout sf_layout, void* workspace, size_t workspace_bytes,
                            void* stream);

/* The same quantisation as nvfp4_quantize, for callers that cannot allocate device
 * memory (for example a host plug-in that is handed only the tensors it reads and
 * writes, with no allocator or memory pool it may use).  The pages have no counterpart:
 * it is a deployment convenience, not part of the method.
 *   Same arguments as nvfp4_quantize without the workspace, scales always in the
 *   NVFP4_SF_SWIZZLED_128x4 layout.  The amax scratch of the
 *   per-tensor and per-group modes lives in a fixed 16 KB device array owned by the
 *   library (at most 4096 scopes: per-group calls with more than 4096 groups and no
 *   global_scale_in return NVFP4_ERR_UNSUPPORTED).  Every GPU that loads the library
 *   holds that array until the process exits.
 *   The first call on each device resolves the array's device address (with that
 *   device current) and keeps it while the device's primary context lives (see the
 *   preamble on cudaDeviceReset); make that first call before any stream capture.
 *   All calls share the one array and each call clears the words it uses before use:
 *   calls whose kernels overlap on the GPU (different streams, no ordering) race on it.
 *   The library calls no allocator (no cudaMalloc / cudaFree) here. */
nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_elems,
                                    nvfp4_scale_mode mode, int64_t group_rows,
                                    nvfp4_rounding rounding, uint64_t seed, uint64_t rng_offset,
                                    const float* global_scale_in, float* global_scale_out,
                                    uint8_t* codes_out, uint8_t* sf_out, void* stream);

/* Transposed quantisation, the layout of the backward's W4A4 GEMMs ("The 4-bitter
 * Lesson...", §"Why is the NVFP4 pretraining recipe not sufficient for RL?": the
 * backward GEMMs quantise their operands along the contraction of each GEMM -- the
 * weights along their output dimension for dgrad, activations and gradients along
 * tokens for wgrad -- with stochastic rounding as the recipe's option for gradients).
 * x is `batches` stacked BF16 matrices [R, C] (pitch ld elements, batch b at rows b*R);
 * the result is NVFP4 of their stacked transposes [batches*C, R], blocks of 16 along R:
 * exactly nvfp4_quantize applied to that transposed BF16 matrix -- same scopes (per
 * tensor; per row of the transpose; per group of group_rows rows of the transpose, so
 * group_rows = C gives one scale per batch), same rounding modes and Philox stream
 * (element index = row-major index in the transpose).
 *   codes_out [batches*C, R/2], sf_out tiled for batches*C rows x R/16, as nvfp4_quantize.
 *   workspace: nvfp4_workspace_size(NVFP4_OP_QUANTIZE_T, batches*C, R, 0, 0, 0) bytes
 *   (the transposed BF16 copy and the amax scratch).  R % 16 == 0, R <= 8192, ld >= C,
 *   ld % 8 == 0; x 16-byte aligned. */
nvfp4_status nvfp4_quantize_transposed(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld,
                                       nvfp4_scale_mode mode, int64_t group_rows,
                                       nvfp4_rounding rounding, uint64_t seed, uint64_t rng_offset,
                                       const float* global_scale_in, float* global_scale_out,
                                       uint8_t* codes_out, uint8_t* sf_out, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Dequantisation DQ ("The 4-bitter Lesson...", §"Improving Gradient Stability",
 * footnote 6: DQ(Q(w)) = code value x block scale x global scale, the operand of the
 * dequantised backward):
 *     out[r, c] = value(code[r, c]) * decode(sf[r, c/16]) * g[scope(r)]
 * rounded once (round to nearest even) from the exact value to out_dtype.
 *   codes: device [rows, cols/2] (element 2i in the low nibble of byte i); sf: device,
 *   128x4 tiled scales for rows x cols/16 (as nvfp4_quantize writes them); g: device
 *   float, 1 (per tensor), rows (per row) or rows/group_rows (per group) values.
 *   out: device [rows, ldo] of out_dtype.  cols % 16 == 0, ldo >= cols, ldo % 8 == 0;
 *   codes, sf and out 16-byte aligned, g 4-byte aligned.  No workspace. */
nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, const float* g, int64_t rows,
                              int64_t cols, nvfp4_scale_mode mode, int64_t group_rows, void* out,
                              nvfp4_out_dtype out_dtype, int64_t ldo, void* stream);

/* ---------------------------------------------------------------- dequantised backward */

/* BF16 grouped GEMM, the GEMM of the dequantised backward ("The 4-bitter Lesson...",
 * §"Improving Gradient Stability": the backward pass multiplies by the dequantised
 * weights DQ(Q(W)) -- see nvfp4_dequantize -- so that it differentiates the forward that
 * was actually run).  For every expert e and every row r of its group:
 *     D[r, n] = sum_k A[r, k] * B_e[n, k]
 * with BF16 operands, accumulated in FP32 on the tensor cores in a fixed order (no
 * split-K), then rounded once to out_dtype.
 *   A: device BF16 [M_total, K] (rows outside the groups are read but their results are
 *      not stored).  B: device BF16 [E, N, K].
 *   group_offsets, group_rows, M_total, D, ldd: as nvfp4_grouped_gemm.
 *   N % 128 == 0, K % 64 == 0, E <= 1024.  A, B and D 16-byte aligned; the group arrays
 *   4-byte aligned.  No workspace. */
nvfp4_status bf16_grouped_gemm(const void* A, const void* B, const int32_t* group_offsets,
                               const int32_t* group_rows, int64_t M_total, int64_t N, int64_t K,
                               int32_t E, void* D, nvfp4_out_dtype out_dtype, int64_t ldd,
                               void* stream);

/* SwiGLU backward of the expert block: for h = silu(gate) * up,
 *     dgate = dh * up * silu'(gate),  silu'(g) = s * (1 + g * (1 - s)),  s = sigmoid(g),
 *     dup   = dh * silu(gate),
 * each evaluated in float32 and rounded once to BF16 (within one BF16 ulp of the float64
 * evaluation, plus float32 round-off where silu' cancels).
 *   gu:  device BF16 [rows, 2I], gate in columns [0, I), up in [I, 2I);
 *   dh:  device BF16 [rows, I];  dgu: device BF16 [rows, 2I], [dgate | dup].
 *   I % 8 == 0; all three 16-byte aligned.  No workspace. */
nvfp4_status moe_swiglu_backward(const void* gu, const void* dh, int64_t rows, int64_t I, void* dgu,
                                 void* stream);

/* Transpose of `batches` stacked BF16 matrices: out[b*C + c, r] = x[b*R + r, c] (x has
 * pitch ld >= C elements; out is [batches*C, R], dense).  It produces the K-major form of
 * a transposed operand, e.g. DQ(W)^T for a dgrad GEMM.  x and out are 4-byte aligned. */
nvfp4_status bf16_transpose(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld, void* out,
                            void* stream);

/* ---------------------------------------------------------------- MXFP8 */

/* MXFP8, the format of the recipe's validation runs ("The 4-bitter Lesson...",
 * §"Improving Gradient Stability", Results Validation with MXFP8: quantised forward and
 * backward, and quantised forward with dequantised weights in the backward).  The pages
 * name the format without defining it.  It is read as OCP MX v1.0 MXFP8:
 *   - E4M3 elements, blocks of 32 values along a row;
 *   - one E8M0 scale per block, b = max(floor(log2 amax_block) - 8 + 127, 0);
 *   - code = E4M3_rn_satfinite(x * 2^(127 - b)), zero magnitudes encoded as +0;
 *   - no global scale: DQ(x) = value(code) * 2^(b - 127).
 * Storage:
 *   codes:  uint8 [rows, cols], one E4M3 byte per element.
 *   scales: E8M0 bytes in the same 128x4 tiled layout as the NVFP4 scales, with
 *           C = cols/32 scale columns: byte ((r/128)*ceil(C/4) + c/4)*512 +
 *           (r%32)*16 + ((r%128)/32)*4 + c%4; rows padded to a multiple of 128; size
 *           mxfp8_sf_bytes(rows, cols). */
size_t mxfp8_sf_bytes(int64_t rows, int64_t cols);

/* MXFP8 quantisation of a BF16 matrix.
 *   x:         device BF16 [rows, ld_elems]; the first `cols` of each row are used.
 *   cols % 128 == 0 (else NVFP4_ERR_UNSUPPORTED); ld_elems >= cols, ld_elems % 8 == 0.
 *   codes_out: device uint8 [rows, cols].
 *   sf_out:    device uint8 [mxfp8_sf_bytes(rows, cols)], tiled layout; the scale words
 *              of the padding rows are written as 0.
 * x, codes_out and sf_out are 16-byte aligned.  No workspace; deterministic. */
nvfp4_status mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_elems,
                            uint8_t* codes_out, uint8_t* sf_out, void* stream);

/* MXFP8 DQ: out[r, c] = value(code[r, c]) * 2^(sf[r, c/32] - 127).  The product is
 * exact in float32.  For BF16 output it is rounded once, to nearest even.
 *   codes: device [rows, cols]; sf: device, tiled as mxfp8_quantize writes it.
 *   out:   device [rows, ldo] of out_dtype.  cols % 128 == 0, ldo >= cols, ldo % 8 == 0;
 *   codes, sf and out 16-byte aligned.  No workspace. */
nvfp4_status mxfp8_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols,
                              void* out, nvfp4_out_dtype out_dtype, int64_t ldo, void* stream);

/* MXFP8 x MXFP8 grouped GEMM over ragged expert groups, on the tensor cores' block-scaled
 * FP8 MMA.  For every expert e and every row r of its group:
 *     D[r, n] = sum_k DQ(A)[r, k] * DQ(B_e)[n, k]
 * This is accumulated in FP32 in a fixed order (no split-K), then rounded once to out_dtype.
 *   A, SFA: device, codes [M_total, K], tiled scales for M_total rows.
 *   B, SFB: device, codes [E, N, K], tiled scales for E*N rows.
 *   group_offsets, group_rows, M_total, D, ldd: as nvfp4_grouped_gemm.
 *   N % 128 == 0, K % 128 == 0, E <= 1024.  A, SFA, B, SFB and D are 16-byte aligned; the
 *   group arrays 4-byte aligned.  No workspace. */
nvfp4_status mxfp8_grouped_gemm(const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                                const uint8_t* SFB, const int32_t* group_offsets,
                                const int32_t* group_rows, int64_t M_total, int64_t N, int64_t K,
                                int32_t E, void* D, nvfp4_out_dtype out_dtype, int64_t ldd,
                                void* stream);

/* ---------------------------------------------------------------- grouped GEMM */

/* W4A4 grouped GEMM over ragged expert groups ("Low-Bit Precision Training Is Ready
 * for Production...", §"What W4A4 GEMM Actually Changes": both operands in 4 bits so
 * the GEMM runs on FP4 tensor cores; "miniTE identifies and closes the execution gap
 * ...", §Development: grouped GEMMs).  For every expert e and every row r of its group
 * (rows group_offsets[e] .. group_offsets[e] + group_rows[e] - 1):
 *     D[r, n] = (gA[r] * gB[e]) * sum_k DQ'(A)[r, k] * DQ'(B_e)[n, k]
 * where DQ' = value(code) * decode(sf), accumulated in FP32 on the tensor cores in a
 * fixed order (no split-K), then rounded once to the output type.
 *   A, SFA, gA:   device, codes [M_total, K/2], tiled scales for M_total rows, [M_total].
 *   B, SFB, gB:   device, codes [E, N, K/2], tiled scales for E*N rows, [E].
 *   group_offsets: device int32 [E+1], multiples of 128, non-decreasing,
 *                 group_offsets[E] <= M_total.  group_rows: device int32 [E],
 *                 group_rows[e] <= group_offsets[e+1] - group_offsets[e].
 *   M_total:      rows allocated for A (a multiple of 128).
 *   N % 128 == 0, K % 256 == 0, E <= 1024.
 *   D:            device, [M_total, ldd] of out_dtype; rows outside every group are not
 *                 written.  ldd % 8 == 0.
 * A, SFA, B, SFB and D must be 16-byte aligned; gA, gB and the group arrays 4-byte
 * aligned.  No workspace.
 */
nvfp4_status nvfp4_grouped_gemm(const uint8_t* A, const uint8_t* SFA, const float* gA,
                                const uint8_t* B, const uint8_t* SFB, const float* gB,
                                const int32_t* group_offsets, const int32_t* group_rows,
                                int64_t M_total, int64_t N, int64_t K, int32_t E, void* D,
                                nvfp4_out_dtype out_dtype, int64_t ldd, void* stream);

/* The same grouped GEMM over operands in the GEMM-tiled layout: A with 128-row blocks
 * (M_total rows, a multiple of 128), B with 256-row blocks (E*N rows), scales inside the
 * tiles.  N % 256 == 0, K % 256 == 0, E <= 512.  gA, gB, group arrays as above.
 *   epilogue NVFP4_EPILOGUE_STORE: D as nvfp4_grouped_gemm.
 *   epilogue NVFP4_EPILOGUE_SWIGLU: B holds gate/up rows interleaved in 64-row chunks
 *     (as nvfp4_moe_weights.w13); D receives BF16 h [M_total, N/2] (row pitch N/2,
 *     ldd and out_dtype ignored) with h = BF16(silu(gate) * up) from the BF16-rounded gate
 *     and up outputs: silu(gate) * up evaluated in float64 and rounded once to BF16.
 *     The first SwiGLU call on a device (this one, moe_swiglu_quantize or
 *     moe_expert_forward) builds a 512 KB table of silu over the BF16 values with one
 *     kernel on `stream` and waits for it; make that first call outside stream capture.
 * Kernel form: one CTA per 128-row x 256-column tile by default.  With the environment
 * variable NVFP4_GEMM_CTA_PAIR=1 (read at every launch) a cluster of two CTAs shares each
 * 256-row x 256-column tile of one expert (tcgen05 cta_group::2, M=256); the results are
 * identical.  The ragged-K weight-gradient GEMMs of moe_expert_backward always use one CTA
 * per tile. */
enum { NVFP4_EPILOGUE_STORE = 0, NVFP4_EPILOGUE_SWIGLU = 1 };
nvfp4_status nvfp4_grouped_gemm_tiled(const uint8_t* A_tiled, const float* gA, const uint8_t* B_tiled,
                                      const float* gB, const int32_t* group_offsets,
                                      const int32_t* group_rows, int64_t M_total, int64_t N,
                                      int64_t K, int32_t E, void* D, nvfp4_out_dtype out_dtype,
                                      int64_t ldd, int32_t epilogue, void* stream);

/* Repack row-major codes [rows, K/2] with their 128x4 tiled scales (nvfp4_quantize's
 * output) into the GEMM-tiled layout with `block_rows`-row blocks (128 or 256); rows
 * beyond `rows` up to the next block are zero.  K % 256 == 0.  out: device,
 * nvfp4_tiled_bytes(rows, K, block_rows) bytes. */
nvfp4_status nvfp4_pack_tiled(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K,
                              int32_t block_rows, uint8_t* out, void* stream);

/* ---------------------------------------------------------------- MoE helpers */

/* Top-k routing of router logits, the "token permute by router top-k" that feeds the
 * expert GEMMs ("Low-Bit Precision Training Is Ready for Production...", §"What W4A4 GEMM
 * Actually Changes": the W4A4 GEMMs are the MoE expert layers, each token running
 * through the experts its router picks).  ids[t, :] = the k experts with the largest
 * logits, in descending order, ties to the lower expert id; weights = softmax over the
 * chosen k (renormalize != 0) or the full-softmax probabilities of the chosen experts.
 * The pages do not give the weight rule; renormalising over the chosen k is this
 * library's reading (the Qwen3 MoE convention), the other the flag's alternative.
 *   logits: device float [T, E]; ids: device int32 [T, k]; weights: device float [T, k].
 *   1 <= k <= 32, k <= E <= 1024. */
nvfp4_status moe_route_topk(const float* logits, int64_t T, int32_t E, int32_t k,
                            int renormalize, int32_t* ids, float* weights, void* stream);

/* Expert grouping ("miniTE identifies and closes the execution gap...", §Development:
 * grouped GEMMs over the experts need each expert's tokens contiguous; "Low-Bit Precision
 * Training Is Ready for Production...", §"The Cross-Engine Alignment Problem": the
 * composition of a batch must not change a token's result, so the slot order is a
 * deterministic function of the ids alone).  Of the T*k (token, j) entries:
 * counts [E], offsets [E+1] (exclusive scan of counts), padded_offsets [E+1] (each group
 * starts at a multiple of 128), inv [T, k] = slot of (t, j), perm [M_cap] = token of each
 * slot, -1 for padding slots below padded_offsets[E] (entries beyond it are not
 * written).  Slots are ordered by expert, then by token.  M_cap = round_up(T*k + E*127,
 * 128) bounds padded_offsets[E].  Ids outside [0, E) set NVFP4_ERR_DEVICE_STATUS and are
 * counted nowhere. */
nvfp4_status moe_permute(const int32_t* ids, int64_t T, int32_t k, int32_t E,
                         int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                         int32_t* inv, int32_t* perm, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Router-weighted un-permute, the last step of the expert block ("Low-Bit Precision
 * Training Is Ready for Production...", §"What W4A4 GEMM Actually Changes": the expert
 * layers' outputs return to their tokens weighted by the router; §"The Cross-Engine
 * Alignment Problem": accumulation order decides the bits, so it is fixed):
 * out[t] = BF16( sum_{j=0..k-1} w[t, j] * y[inv[t, j]] ),
 * each product and each partial sum a float32 operation, in the order j = 0..k-1.
 *   y: device BF16 [*, H]; inv: device int32 [T, k]; w: device float [T, k];
 *   out: device BF16 [T, H].  H % 8 == 0. */
nvfp4_status moe_combine(const void* y, const int32_t* inv, const float* w, int64_t T,
                         int32_t k, int64_t H, void* out, void* stream);

/* SwiGLU of the interleaved gate/up output followed by per-row NVFP4 requantisation.
 * For each row r with perm[r] >= 0 and each c < I:
 *     h[r, c] = BF16( silu(gate) * up )   (evaluated in float64, rounded once)
 * where gate/up are D's columns in the 64-chunk interleave of nvfp4_moe_weights; then
 * h's row is quantised with a per-row scale into hq [rows, Ip/2] (zero-padded to
 * Ip = round_up(I, 256)), tiled scales (Ip/16 columns) and gh [rows].
 *   d: device BF16 [rows, 2I]; h_out: device BF16 [rows, I] or NULL. */
nvfp4_status moe_swiglu_quantize(const void* d, const int32_t* perm, int64_t rows, int64_t I,
                                 void* h_out, uint8_t* hq, uint8_t* hsf, float* gh,
                                 void* stream);

/* Quantise the expert weights once per weight update ("The 4-bitter Lesson...",
 * §"Why is the NVFP4 pretraining recipe not sufficient for RL?": weights use per-block
 * E4M3 scales and one FP32 global scale; each expert matrix is its own tensor).
 *   w13: device BF16 [E, 2I, H] (gate rows 0..I-1, up rows I..2I-1);
 *   w2:  device BF16 [E, H, I].  H % 256 == 0, I % 128 == 0, H <= 2048, I <= 2048,
 *   E <= 512.
 *   out: struct of caller-allocated buffers (moe_weights_sizes). */
nvfp4_status moe_prepare_weights(const void* w13, const void* w2, int32_t E, int64_t H,
                                 int64_t I, const nvfp4_moe_weights* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* The expert block forward ("Low-Bit Precision Training Is Ready for Production...",
 * §"What W4A4 GEMM Actually Changes": W4A4 on the expert layers; "The 4-bitter
 * Lesson...", per-token activation scales, fused per-token quantiser):
 *   permute -> per-token NVFP4 of x (token order, GEMM-tiled) gathered into every routed
 *   slot -> gate/up grouped GEMM with the SwiGLU epilogue (BF16 h) -> per-row NVFP4 of h
 *   (GEMM-tiled) -> down grouped GEMM (BF16 y) -> weighted combine (BF16).  The bits equal those of the
 *   unfused chain nvfp4_grouped_gemm -> moe_swiglu_quantize -> nvfp4_grouped_gemm ->
 *   moe_combine over the same operands.
 *   x: device BF16 [T, H] and out: device BF16 [T, H], 16-byte aligned;
 *   ids: device int32 [T, k] and w: device float [T, k], 4-byte aligned;
 *   weights: prepared weights (16-byte aligned buffers).
 *   workspace: nvfp4_workspace_size(NVFP4_OP_MOE_FORWARD, T, k, E, H, I) bytes; its
 *   layout (for inspection) is given by moe_forward_workspace_layout().
 *   1 <= k <= 32, T*k < 2^31; the weights' E <= 512. */
nvfp4_status moe_expert_forward(const void* x, const int32_t* ids, const float* w, int64_t T,
                                int32_t k, const nvfp4_moe_weights* weights, void* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- backward (W4A4) */

/* Transposed expert weights for the backward's dgrad GEMMs ("The 4-bitter Lesson...",
 * §"Why is the NVFP4 pretraining recipe not sufficient for RL?": the pretraining recipe
 * runs the backward GEMMs in NVFP4 too; a dgrad GEMM dX = dY W contracts over W's output
 * dimension, so W is quantised along it).  Caller-allocated device buffers, sizes from
 * moe_weights_t_sizes() in struct order; both GEMM-tiled with 256-row blocks.
 *   w13t: W13_e^T [H, 2I] per expert (rows e*H ..), K = 2I in the canonical [gate | up]
 *         order, blocks of 16 along 2I, one FP32 global scale per expert (w13t_g [E]);
 *   w2t:  W2_e^T [I, H] per expert, rows padded to Ip = round_up(I, 256) with zeros
 *         (rows e*Ip ..), K = H, one global scale per expert (w2t_g [E]). */
typedef struct {
  int32_t E;
  int64_t H;
  int64_t I;
  uint8_t* w13t;
  float* w13t_g;
  uint8_t* w2t;
  float* w2t_g;
} nvfp4_moe_weights_t;

nvfp4_status moe_weights_t_sizes(int32_t E, int64_t H, int64_t I, size_t sizes_out[4]);

/* Quantise the transposed weights once per weight update (round to nearest).
 *   w13: device BF16 [E, 2I, H]; w2: device BF16 [E, H, I] (the forward's inputs).
 *   H % 256 == 0, I % 128 == 0, E <= 512.  workspace:
 *   nvfp4_workspace_size(NVFP4_OP_PREPARE_WEIGHTS_T, E, 0, 0, 0, 0) bytes. */
nvfp4_status moe_prepare_weights_backward(const void* w13, const void* w2, int32_t E, int64_t H, int64_t I,
                                          const nvfp4_moe_weights_t* out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* The expert block's backward in W4A4 ("The 4-bitter Lesson...", §"Why is the NVFP4
 * pretraining recipe not sufficient for RL?": every backward GEMM on NVFP4 operands with
 * stochastic rounding of the gradients -- recipe (a), "quantized forward and backward", of
 * §"Improving Gradient Stability", Results Validation).  For out = moe_expert_forward(x,
 * ids, w, weights) and its upstream gradient dout:
 *   dy[slot(t,j)] = BF16(w[t,j] dout[t]);          dw[t,j] = <dout[t], y[slot(t,j)]>  (float32)
 *   dh = Q(dy) Q(W2^T)  (dgrad, BF16)              dW2_e = Q(dy_e^T) Q(h_e^T)   (wgrad, float32)
 *   [dgate | dup] = SwiGLU backward of D = gate/up output (recomputed: the fused forward
 *   keeps only h)
 *   dxs = Q(dD) Q(W13^T) (dgrad, BF16 per slot)    dW13_e = Q(dD_e^T) Q(x_e^T)  (wgrad, float32)
 *   dx[t] = BF16(sum_j dxs[slot(t,j)])
 * Quantisation: dgrad operands along the contraction -- the gradient per routed row (one
 * FP32 scale per row) with stochastic rounding, the weights from `weights_t`; wgrad
 * operands transposed per expert along the tokens (one FP32 scale per expert matrix,
 * each expert's tokens zero-padded to a multiple of 256, at least 256), the gradient
 * with stochastic rounding, h and x to nearest.  Philox key of each stochastic
 * quantisation: seed + (((stream << 10) + expert) << 40), stream 0 = dy by rows, 1 = dy^T,
 * 2 = dD by rows, 3 = dD^T (expert 0 for the row quantisations), element index = row-major
 * index in the quantised matrix (slot layout for rows, the expert's [features, tokens]
 * transpose for wgrad).
 *   dout, x: device BF16 [T, H]; w: device float [T, k] (the forward's router weights).
 *   weights / weights_t: the forward's prepared weights and the transposed ones.
 *   fwd_workspace: the workspace of the moe_expert_forward call on these inputs (its
 *     grouping, routed activations, h and y are read; nothing in it is written), with
 *     that call ordered before this one.
 *   dx: device BF16 [T, H]; dw: device float [T, k]; dw13: device float [E, 2I, H]
 *   (canonical gate/up rows); dw2: device float [E, H, I].
 *   workspace: nvfp4_workspace_size(NVFP4_OP_MOE_BACKWARD, T, k, E, H, I) bytes; its
 *   layout is given by moe_backward_workspace_layout().
 *   H % 256 == 0, H <= 2048, I % 128 == 0, I <= 1024, 1 <= k <= 32, E <= 512; the
 *   buffers 16-byte aligned (w, dw 4-byte). */
nvfp4_status moe_expert_backward(const void* dout, const void* x, const float* w, int64_t T, int32_t k,
                                 const nvfp4_moe_weights* weights, const nvfp4_moe_weights_t* weights_t,
                                 const void* fwd_workspace, size_t fwd_workspace_bytes, uint64_t seed, void* dx,
                                 float* dw, float* dw13, float* dw2, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* Byte offsets inside the backward's workspace: [0] dy BF16 [M_cap, H], [1] Q(dy)
 * GEMM-tiled (128-row blocks, K = H), [2] its per-row scales float [M_cap], [3] dh BF16
 * [M_cap, Ip], [4] D BF16 [M_cap, 2I] (gate/up interleaved as the prepared W13), [5] dD
 * BF16 [M_cap, 2I] ([dgate | dup]), [6] Q(dD) GEMM-tiled (K = 2I), [7] its scales, [8] dxs
 * BF16 [M_cap, H], [9] K-block prefix sums int32 [E+1], [10] per-expert amax bits
 * [4E], [11] per-expert global scales float [4E] (dy^T, h^T, dD^T, x^T), [12] .. [15] the
 * wgrad operands Q(dy^T) (128-row blocks), Q(h^T) (256-row blocks, Ip rows per expert),
 * Q(dD^T), Q(x^T), [16] their capacity in 256-token K-blocks (a count), [17] total bytes. */
nvfp4_status moe_backward_workspace_layout(int64_t T, int32_t k, int32_t E, int64_t H, int64_t I,
                                           int64_t layout_out[18]);

/* Byte offsets of the forward's intermediates inside its workspace, in this order:
 * [0] counts int32[E], [1] offsets int32[E+1], [2] padded_offsets int32[E+1],
 * [3] inv int32[T*k], [4] perm int32[M_cap],
 * [5] Aq: GEMM-tiled (128-row blocks) codes and scales of the routed rows, K = H,
 * [6] equal to [5] (the scales live inside the tiles), [7] gA float[M_cap],
 * [8] h BF16 [M_cap, I], [9] hq: GEMM-tiled (128-row blocks), K = Ip,
 * [10] equal to [9], [11] gh float[M_cap], [12] y BF16 [M_cap, H] (before the down
 * GEMM this region holds the token-ordered quantised x and its per-token scales),
 * [13] M_cap (a row count, not an offset), [14] total bytes.
 * Only rows below padded_offsets[E] whose perm entry is >= 0 are meaningful. */
nvfp4_status moe_forward_workspace_layout(int64_t T, int32_t k, int32_t E, int64_t H,
                                          int64_t I, int64_t layout_out[15]);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
