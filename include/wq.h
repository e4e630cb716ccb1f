/*
 * wq.h -- C ABI of the weight-only quantized GEMM library for GB300 (sm_103a).
 *
 *   out[M, N] = A[M, K] . dequant(W)[N, K]^T      fp32 accumulation, 16-bit out
 *
 * Weight formats:
 *   W4A16   INT4 codes, two per byte along K (even k in the low nibble), value
 *           (q - 8) * S[k / G, n] with fp16 group scales S[K/G][N], G in {32, 64,
 *           128, 256}.  Source: "Low Bit Triton Kernels" (GPU MODE lecture 34),
 *           §03 core pattern (the gemlite-style BLOCK_K loop: unpack two nibbles,
 *           subtract 8, multiply by s[k // GROUP_SIZE, n], dot product).
 *   FP8     e4m3 codes W[N][K] and one fp32 per-tensor scale applied to the fp32
 *           accumulator, optional bias.  Source: "FlashInfer W8A16 GEMM
 *           (mm_bf16_fp8) analysis" (PR #7495), introduction and §2 (public API:
 *           mm_bf16_fp8 / mm_fp16_fp8 take a, b, alpha, bias, out, workspace).
 *   FP4     e2m1 codes W[N][K/2] (even k in the low nibble) with one e4m3 scale
 *           per 16 values along K and a global fp32 alpha.  Source: "FlashInfer
 *           SM100 BF16 x FP4 GEMM" (PR #4466), §2 (uint8 weight of shape [N, K/2],
 *           block scale factors reordered by an offline preparation step) and §3
 *           (the kernel takes weight, weight scale, activation, alpha, output).
 *   W4A16 variants on the same packed codes: an integer zero point per group and
 *           row, (q - Z) * S (wq_gemm_w4a16_zp), and a 16-entry fp16 codebook,
 *           LUT[q] * S (NF4-style, wq_gemm_w4a16_lut).
 *   W2A16   2-bit codes, four per byte along K, (q - 2) * S (wq_gemm_w2a16).
 *
 * Conventions for every entry point:
 *   - All arrays are row-major and live in device memory unless stated.  The
 *     caller allocates and owns every buffer; the library never allocates,
 *     frees or synchronises.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and returns immediately.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-WQ_OK status means nothing was enqueued.  WQ_ERR_CUDA reports a CUDA
 *     runtime error from the launch itself (the CUDA error is left pending).
 *   - Pointers named below as "16-byte aligned" are read by TMA / bulk copies;
 *     scalars (alpha, bias) need only element alignment.
 *   - Only compute capability 10.3 (GB300) is supported: other devices give
 *     WQ_ERR_UNSUPPORTED_DEVICE.
 *   - M == 0 (with N, K > 0) is a valid empty problem: it returns WQ_OK without
 *     launching or looking at any pointer.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* wq_stream_t; /* same type as cudaStream_t */

typedef enum { WQ_F16 = 0, WQ_BF16 = 1 } wq_dtype;

typedef enum {
    WQ_OP_W4A16 = 0,
    WQ_OP_FP8 = 1,
    WQ_OP_FP4 = 2,
    WQ_OP_W4A16_ZP = 3,
    WQ_OP_W4A16_LUT = 4,
    WQ_OP_W2A16 = 5
} wq_op;

typedef enum {
    WQ_OK = 0,
    WQ_ERR_NULL = 1,                /* a required pointer is NULL */
    WQ_ERR_SHAPE = 2,               /* M < 0, N or K <= 0, or a size rule below */
    WQ_ERR_GROUP = 3,               /* G not in {32, 64, 128, 256} or K % G != 0 */
    WQ_ERR_MISALIGNED = 4,          /* a pointer misses its alignment */
    WQ_ERR_DTYPE = 5,               /* activation dtype not supported by the op */
    WQ_ERR_WORKSPACE = 6,           /* workspace missing or smaller than required */
    WQ_ERR_UNSUPPORTED_DEVICE = 7,  /* current device is not compute capability 10.3 */
    WQ_ERR_CUDA = 8,                /* a CUDA runtime call failed */
    WQ_ERR_TIMEOUT = 9              /* a kernel gave up on a bounded wait (device status) */
} wq_status;

/* Human-readable name of a status. */
const char* wq_status_string(wq_status s);

/* ------------------------------------------------------------------ INT4 */

/* Sizes of the kernel-order ("prepacked") INT4 weight and scale buffers for an
 * N x K weight with group size G.  N is padded to a multiple of 128 and K to a
 * multiple of 256 inside them.  Host only. */
wq_status wq_int4_packed_bytes(int64_t N, int64_t K, int32_t G, size_t* w_bytes, size_t* s_bytes);

/* Offline layout transform (a pure permutation; bit-exact and invertible).
 * Reorders canonical packed codes w_canon uint8 [N][K/2] and fp16 scales s_canon
 * [K/G][N] into the tile-major order the GEMM kernels stream with bulk copies:
 * for each 128-row tile and 128-value k-block, the codes of every 16-row group in
 * the register order of a 16x16 tensor-core operand fragment (each 32-bit word is
 * one lane's fragment for one 16-wide k step), so the in-kernel unpack is one
 * mask-and-or per operand register and needs no shared-memory shuffle; scales as
 * [tile][K/G][128 rows].  Padding rows and
 * columns get code 8 and scale 0 (weight 0).  Why: "Bitblas -- Mixed-Precision
 * GEMM with the Ladder Compiler" (GPU MODE lecture 33), introduction -- when the
 * weight layout does not match what the tensor-core operand wants, the layout
 * conversion on the critical path costs more than half of the performance; the
 * Ladder compiler moves it offline.
 * Requirements: N > 0, K % 32 == 0, K % G == 0; w_kernel and s_kernel 16-byte
 * aligned and of wq_int4_packed_bytes sizes; w_canon 1-byte, s_canon 2-byte
 * aligned. */
wq_status wq_pack_int4(const uint8_t* w_canon, const void* s_canon, int64_t N, int64_t K, int32_t G,
                       uint8_t* w_kernel, void* s_kernel, wq_stream_t stream);

/* Synthetic group-wise symmetric INT4 quantiser, the step upstream of
 * wq_pack_int4 ("Low Bit Triton Kernels", GPU MODE lecture 34, hands-on exercise
 * 1: fp16 weight -> group-wise quantize -> two nibbles per byte; the page fixes no
 * scale rule, the symmetric one is taken).  For each row n and group g of G
 * consecutive k:
 *     s_canon[g][n] = RN16(amax / 7),   amax = max |w[n][k]| over the group
 *     q[n][k] = clamp(rint(w[n][k] / s) + 8, 0, 15)   (half to even; 8 if s == 0)
 * decided in fp32 with IEEE division.  w: fp16 [N][K], finite, 16-byte aligned.
 * Outputs in the canonical layouts wq_pack_int4 reads: w_canon uint8 [N][K/2]
 * (even k in the low nibble, 4-byte aligned), s_canon fp16 [K/G][N] (2-byte
 * aligned).  Requirements: N > 0, K % 32 == 0, K % G == 0, G in {32, 64, 128,
 * 256}.  A group whose amax is below 7 * 2^-14 gets a subnormal fp16 scale, whose
 * coarser step can clamp codes (at most within 2^-11 of amax). */
wq_status wq_quantize_int4(const void* w, int64_t N, int64_t K, int32_t G, uint8_t* w_canon, void* s_canon,
                           wq_stream_t stream);

/* Inverse of wq_pack_int4 (tests, export). */
wq_status wq_unpack_int4(const uint8_t* w_kernel, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                         uint8_t* w_canon, void* s_canon, wq_stream_t stream);

/* Debug export: the exact dequantized weight (q - 8) * s as fp32 [N][K], read
 * from the prepacked buffers.  The fp32 value is exact (at most 15 significant
 * bits). */
wq_status wq_debug_dequant_int4(const uint8_t* w_kernel, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                                float* w_f32, wq_stream_t stream);

/* W4A16 GEMM: out[M][N] (same 16-bit type as A) = A[M][K] . ((q - 8) * S)^T.
 * A: a_dtype [M][K], 16-byte aligned.  w_kernel / s_kernel: output of
 * wq_pack_int4 for this N, K, G.  out: 16-byte aligned, N % 8 == 0.
 * ws: workspace of at least wq_workspace_bytes(WQ_OP_W4A16, ...) bytes,
 * 16-byte aligned; may be NULL when that size is 0.  Its first 16 KiB hold
 * split-K arrival counters: zero-fill them once after allocating the workspace;
 * every call leaves them zero again (a call that ends with a timeout bit in the
 * device status may not).  One workspace may serve calls of any shape, but calls
 * that share it must not overlap on the GPU.  The dequantized operand is
 * RN((q - 8) * s) in the type of A, accumulated in fp32; split-K partial sums
 * are reduced in a fixed order, so results are identical run to run.  For
 * M <= 16 with K % 64 == 0 the sum is formed as s * sum_k A (q - 8) per group in
 * fp32 (exact products, no rounding of the operand).
 * The kernel may start while the kernel before it on the stream is finishing
 * (programmatic dependent launch); it reads w_kernel and s_kernel before it waits
 * for that kernel, and A, out and ws only after.  So the kernel immediately before
 * the call on the stream must not write w_kernel or s_kernel (wq_pack_int4 ends
 * with an ordinary launch for this reason). */
wq_status wq_gemm_w4a16(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                        int64_t M, int64_t N, int64_t K, int32_t G, void* out, void* ws, size_t ws_bytes,
                        wq_stream_t stream);

/* ---------------------------------------------------------- INT4 zero point */

/* Asymmetric (zero-point) INT4: w[n][k] = (q[n][k] - Z[k/G][n]) * S[k/G][n], one
 * integer zero point 0..15 per group and row beside the scale.  "Low Bit Triton
 * Kernels" (GPU MODE lecture 34), §02, names the group-scaled 4-bit formats of
 * GPTQ, AWQ and HQQ, which carry zero points, but prints no zero-point encoding;
 * an integer zero point in the code range is the reading taken.  With Z = 8 it is
 * the symmetric format.  Codes and scales pack with wq_pack_int4 as before.
 *
 * Size of the kernel-order zero-point buffer: N padded to 128, K to 256, one byte
 * per (group, row).  Host only. */
wq_status wq_int4_packed_zeros_bytes(int64_t N, int64_t K, int32_t G, size_t* z_bytes);

/* Layout transform of the zero points: z_canon uint8 [K/G][N] (values 0..15) to
 * z_kernel [N/128][Kp/G][128], the order of the packed scales; padding gets 8.
 * z_kernel: 16-byte aligned, wq_int4_packed_zeros_bytes long.  Values above 15
 * are not checked (the kernel reads them as given). */
wq_status wq_pack_int4_zeros(const uint8_t* z_canon, int64_t N, int64_t K, int32_t G, uint8_t* z_kernel,
                             wq_stream_t stream);

/* W4A16 GEMM with zero points: out[M][N] = A[M][K] . ((q - Z) * S)^T.  Arguments as
 * for wq_gemm_w4a16 plus z_kernel (wq_pack_int4_zeros output, 16-byte aligned), the
 * workspace sized for WQ_OP_W4A16_ZP.  The operand is RN((q - Z) * s) in the type of
 * A (q - Z is exact), accumulated in fp32, on the tile kernels; for M <= 16 with
 * K % 64 == 0 the register decode kernel forms s * (sum_k A (q - 8) + (8 - Z) sum_k A)
 * per group in fp32 instead (exact products, no operand rounding).  The same rule on
 * the kernel before the call holds, now for z_kernel as well. */
wq_status wq_gemm_w4a16_zp(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                           const uint8_t* z_kernel, int64_t M, int64_t N, int64_t K, int32_t G, void* out, void* ws,
                           size_t ws_bytes, wq_stream_t stream);

/* ------------------------------------------------------------- INT4 codebook */

/* Codebook (NF4-style) INT4: w[n][k] = LUT[q[n][k]] * S[k/G][n], the 4-bit code
 * selecting one of 16 fp16 values.  "Low Bit Triton Kernels" (GPU MODE lecture 34),
 * the passage on choosing the 16 values of a 4-bit weight: a uniform grid (INT4), a
 * non-uniform one (NF4) or a floating-point one (FP4), NF4's dequant being a lookup
 * table held in registers at about twice the instructions of the INT4 shift-and-mask.
 * The page prints no table, so the table is an argument: any 16 finite fp16 values
 * (with LUT[q] = q - 8 this is the symmetric format).  Codes and scales pack with
 * wq_pack_int4 as for W4A16.
 *
 * W4A16 GEMM with a codebook: out[M][N] = A[M][K] . (LUT[q] * S)^T.  Arguments as
 * for wq_gemm_w4a16 plus lut: 16 fp16 values in device memory, 16-byte aligned (read
 * as two 16-byte vectors); the workspace is sized for WQ_OP_W4A16_LUT.  The operand
 * is RN(LUT[q] * s) in the type of A (the product of two fp16 values is exact in
 * fp32), accumulated in fp32, on the tile kernels.  With fp16 A, M <= 16 and
 * K % 64 == 0 the register decode kernel runs instead (WQ_KERNEL_DECODE): operands
 * LUT[q] exactly, the group scale on the fp32 sums, out = RN16(sum_g s_g * sum_{k in g}
 * A LUT[q]).  lut is read after the kernel waits for the kernel before it on the
 * stream, so it may be written by that kernel; w_kernel and s_kernel follow the rule
 * of wq_gemm_w4a16. */
wq_status wq_gemm_w4a16_lut(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                            const void* lut, int64_t M, int64_t N, int64_t K, int32_t G, void* out, void* ws,
                            size_t ws_bytes, wq_stream_t stream);

/* Debug export: the exact dequantized codebook weight LUT[q] * s as fp32 [N][K],
 * read from the prepacked buffers (lut: 16 fp16 values, 2-byte aligned). */
wq_status wq_debug_dequant_int4_lut(const uint8_t* w_kernel, const void* s_kernel, const void* lut, int64_t N,
                                    int64_t K, int32_t G, float* w_f32, wq_stream_t stream);

/* ------------------------------------------------------------------ INT2 */

/* W2A16: w[n][k] = (q[n][k] - 2) * S[k/G][n], 2-bit codes q in 0..3.  "Bitblas --
 * Mixed-Precision GEMM with the Ladder Compiler" (GPU MODE lecture 33), hands-on
 * sequence item 6, names the W2A16 (INT2 weight) combination without a formula; the
 * reading taken is the INT4 format one size down: four codes per byte along K with
 * code k at bits 2 (k % 4) .. 2 (k % 4) + 1 of byte k / 4 (w_canon uint8 [N][K/4]),
 * symmetric offset 2, fp16 group scales S[K/G][N].  The codes are read canonical
 * (TMA rows of K/4 bytes); only the scales are reordered.
 *
 * Size of the kernel-order scale buffer (N padded to 128, K to 256).  Requirements:
 * N > 0, K % 64 == 0 (16-byte code rows), K % G == 0, G in {32, 64, 128, 256}.
 * Host only. */
wq_status wq_int2_packed_scales_bytes(int64_t N, int64_t K, int32_t G, size_t* s_bytes);

/* Layout transform of the scales: s_canon fp16 [K/G][N] (2-byte aligned) to s_kernel
 * [N/128][Kp/G][128] (16-byte aligned, wq_int2_packed_scales_bytes long), padding
 * zero.  Ends with an ordinary launch, as wq_pack_int4. */
wq_status wq_pack_int2_scales(const void* s_canon, int64_t N, int64_t K, int32_t G, void* s_kernel,
                              wq_stream_t stream);

/* Debug export: the exact dequantized weight (q - 2) * s as fp32 [N][K] (at most 13
 * significant bits), from the canonical codes and the packed scales. */
wq_status wq_debug_dequant_int2(const uint8_t* w_canon, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                                float* w_f32, wq_stream_t stream);

/* W2A16 GEMM: out[M][N] (type of A) = A[M][K] . ((q - 2) * S)^T.  A: a_dtype [M][K],
 * 16-byte aligned.  w_canon: uint8 [N][K/4], 16-byte aligned.  s_kernel: output of
 * wq_pack_int2_scales.  out: 16-byte aligned, N % 8 == 0.  ws: workspace sized for
 * WQ_OP_W2A16 (the rules of wq_gemm_w4a16's workspace apply).  The operand is
 * RN((q - 2) * s) in the type of A, accumulated in fp32, on the tile kernels.  With
 * M <= 16, G >= 64 and K % 256 == 0 the register decode kernel runs instead
 * (WQ_KERNEL_DECODE): operands q - 2 exactly, the group scale on the fp32 sums,
 * out = RN(sum_g s_g * sum_{k in g} A (q - 2)).  Every input is read after the kernel
 * waits for the kernel before it on the stream. */
wq_status wq_gemm_w2a16(const void* A, wq_dtype a_dtype, const uint8_t* w_canon, const void* s_kernel, int64_t M,
                        int64_t N, int64_t K, int32_t G, void* out, void* ws, size_t ws_bytes, wq_stream_t stream);

/* ------------------------------------------------------------------ FP8 */

/* Debug export: e4m3 weight [N][K] decoded through the kernel's operand
 * conversion to `operand` type and widened to fp32 (exact). */
wq_status wq_debug_dequant_fp8(const uint8_t* w_e4m3, int64_t N, int64_t K, wq_dtype operand, float* w_f32,
                               wq_stream_t stream);

/* W8A16 FP8 GEMM: out[M][N] = alpha * (A . e4m3(W)^T) + bias, fp32 epilogue,
 * rounded once to the type of A (bf16: mm_bf16_fp8, fp16: mm_fp16_fp8).
 * A: a_dtype [M][K], 16-byte aligned, K % 16 == 0.  w_e4m3: uint8 [N][K],
 * 16-byte aligned.  alpha: device pointer to one float (element aligned; read
 * by the kernel, so a CUDA graph can capture the call).  bias: NULL or [N] of
 * the type of A.  out, ws: as for wq_gemm_w4a16 (op WQ_OP_FP8).  M <= 32 with
 * K % 64 == 0 runs on the decode kernel (WQ_KERNEL_DECODE: the codes read straight
 * from W, converted in registers, no workspace); other shapes on the tile kernels.
 * The e4m3 codes S.1111.111 decode as NaN on every path. */
wq_status wq_gemm_w8a16_fp8(const void* A, wq_dtype a_dtype, const uint8_t* w_e4m3, const float* alpha,
                            const void* bias, int64_t M, int64_t N, int64_t K, void* out, void* ws,
                            size_t ws_bytes, wq_stream_t stream);

/* ------------------------------------------------------------------ FP4 */

/* Size of the prepacked FP4 block-scale buffer (N padded to 128, K to 128). */
wq_status wq_fp4_packed_sf_bytes(int64_t N, int64_t K, size_t* sf_bytes);

/* Offline reorder of the e4m3 block scales sf_canon uint8 [N][K/16] into the
 * tile-major order the kernel streams with one bulk copy per k-block (for each
 * 128-row tile and each 64 values along K, 4 bytes per row).  Padding gets 0.
 * Requirements: K % 32 == 0; sf_kernel 16-byte aligned. */
wq_status wq_pack_fp4_sf(const uint8_t* sf_canon, int64_t N, int64_t K, uint8_t* sf_kernel, wq_stream_t stream);

/* Debug export: e2m1(code) * e4m3(sf) as fp32 [N][K], through the kernel's
 * operand conversion (exact). */
wq_status wq_debug_dequant_fp4(const uint8_t* w_e2m1, const uint8_t* sf_kernel, int64_t N, int64_t K,
                               float* w_f32, wq_stream_t stream);

/* BF16 x FP4 GEMM: out[M][N] bf16 = alpha * (A . (e2m1(W) * e4m3(SF))^T).
 * A: bf16 [M][K], 16-byte aligned, K % 32 == 0.  w_e2m1: uint8 [N][K/2], 16-byte
 * aligned.  sf_kernel: output of wq_pack_fp4_sf.  alpha: device pointer to one
 * float.  out, ws: as for wq_gemm_w4a16 (op WQ_OP_FP4).  M <= 16 with K % 256 == 0
 * runs on the decode kernel (WQ_KERNEL_DECODE: codes and block scales turned into
 * exact bf16 operands in registers, no workspace); other shapes on the tile kernels. */
wq_status wq_gemm_bf16_fp4(const void* A, const uint8_t* w_e2m1, const uint8_t* sf_kernel, const float* alpha,
                           int64_t M, int64_t N, int64_t K, void* out, void* ws, size_t ws_bytes,
                           wq_stream_t stream);

/* ------------------------------------------------------------------ planning */

/* The launch plan the library picks for a problem (deterministic in the
 * arguments and the current device). */
typedef struct {
    int32_t bn;           /* tokens per tile (tcgen05 MMA N) */
    int32_t bk;           /* k per pipeline stage */
    int32_t stages;       /* shared-memory pipeline depth */
    int32_t splits;       /* CTAs sharing one output tile's K range (decode: rounded up) */
    int32_t grid;         /* CTAs launched */
    int32_t threads;      /* threads per CTA */
    int32_t smem_bytes;   /* dynamic shared memory per CTA */
    int32_t n_items;      /* tiles x splits */
    int32_t walk_n_fast;  /* 1: weight-row tiles are walked fastest (when the weight is the
                             smaller operand); WQ_WALK=n / WQ_WALK=m in the environment
                             forces either order, e.g. to measure both */
    int32_t tiles_n;
    int32_t tiles_m;
    int32_t ctas_per_sm;  /* resident CTAs per SM assumed by the plan */
    int32_t kernel;       /* WQ_KERNEL_TILE, WQ_KERNEL_DECODE or WQ_KERNEL_TILE_PAIR */
    int32_t cluster_split; /* 1: the split-K slices of a tile run as one thread-block cluster and
                              are reduced through distributed shared memory (no workspace) */
    int32_t cluster_capacity; /* splits-CTA clusters of this kernel the device holds at once
                                 (0 when not applicable); cluster_split needs tiles <= it */
} wq_plan;

/* Kernels a plan can pick.  TILE: the tcgen05 kernel (weights dequantized into
 * tensor memory, any M).  DECODE: W4A16 (symmetric or zero point) with M <= 16 and
 * K % 64 == 0, the codebook format with fp16 A, M <= 16 and K % 64 == 0, INT2 with
 * M <= 16, G >= 64 and K % 256 == 0, FP8 with
 * M <= 32 and K % 64 == 0, or FP4 with M <= 16 and K % 256 == 0; MMA operands built in
 * registers (W4A16 and codebook: from the fragment-order layout, group scale applied
 * in fp32; INT2: from the canonical codes, group scale applied in fp32; FP8 / FP4:
 * from the plain codes (and the prepacked block scales), alpha applied in fp32). */
#define WQ_KERNEL_TILE 0
#define WQ_KERNEL_DECODE 1
/* TILE_PAIR: W4A16 with large M.  The tile kernel on two-CTA clusters: 256 weight
 * rows x 256 tokens per tile, each CTA dequantizes its 128 rows and copies half of
 * the token tile, one tcgen05 MMA of M = 256 spans both SMs.  tiles_n counts
 * 256-row tiles and grid counts CTAs (two per cluster). */
#define WQ_KERNEL_TILE_PAIR 2

/* Plan and workspace size for op (a_dtype is ignored for WQ_OP_FP4, G for FP8
 * and FP4).  Either output pointer may be NULL.  Host only. */
wq_status wq_get_plan(wq_op op, wq_dtype a_dtype, int64_t M, int64_t N, int64_t K, int32_t G, wq_plan* plan,
                      size_t* ws_bytes);

/* Workspace bytes an op needs: 0 when no split-K is used or when the split-K
 * slices are reduced inside a thread-block cluster (wq_plan.cluster_split; the
 * tile kernel chooses this for token tiles of 64 or more when a cost estimate
 * favours it).  In the environment, WQ_SPLITK_WORKSPACE=1 keeps the workspace
 * reduction (the last arriver sums the slices) and WQ_SPLITK_CLUSTER=1 takes the
 * cluster reduction whenever its clusters fit in one wave, e.g. to compare the two.
 * Host only. */
wq_status wq_workspace_bytes(wq_op op, wq_dtype a_dtype, int64_t M, int64_t N, int64_t K, int32_t G,
                             size_t* bytes);

/* Host-side check of the launch planner's division by a runtime constant (the tile
 * walk and the split-K item decode divide work-item indices by tile and slice
 * counts with a multiply-shift).  "FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis",
 * §3(b): a divisor-1 magic number of 2^40 overflowed int64 in that page's kernel;
 * the planner falls back to the plain division whenever the largest dividend times
 * the magic number would not fit in 63 bits.  For divisor d and largest dividend
 * x_max (the planner's bound), writes q[i] = x[i] / d computed exactly as the
 * kernels do, and *uses_multiply = 1 when the multiply-shift path is taken (0: the
 * plain division).  Requires d >= 1, every x[i] <= x_max, n >= 0.  Host only: no
 * GPU, no CUDA call.  Returns WQ_ERR_NULL / WQ_ERR_SHAPE on bad arguments. */
wq_status wq_debug_fastdiv(uint32_t d, uint32_t x_max, const uint32_t* x, int64_t n, uint32_t* q,
                           int32_t* uses_multiply);

/* ------------------------------------------------------------------ no caller workspace */

/* Bytes of split-K scratch built into the library for wq_gemm_w4a16_noalloc. */
#define WQ_NOALLOC_SCRATCH_BYTES (8u << 20)

/* W4A16 GEMM that takes no workspace.  The paper has no counterpart: this entry
 * point is for callers that cannot allocate device memory themselves -- a framework
 * that owns all device memory through its own pool, or a decode loop where a
 * cudaMalloc (which may synchronise the device) is not allowed.  Arguments and
 * results are those of wq_gemm_w4a16 without ws / ws_bytes, and it allocates
 * nothing.  Its split-K scratch is one array of WQ_NOALLOC_SCRATCH_BYTES inside the
 * library, held on every GPU that loads the library until the process exits; a
 * problem whose scratch would not fit returns WQ_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (once per device,
 * with that device current): make that first call before any stream capture.  A
 * lookup that fails returns WQ_ERR_CUDA and is tried again by the next call.  Each
 * call clears the array's 16 KiB of arrival counters on `stream`, then runs the GEMM.
 * All calls share the array and it keeps the last call's contents, so calls that
 * overlap on the GPU (unordered streams) race; order them on one stream. */
wq_status wq_gemm_w4a16_noalloc(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                                int64_t M, int64_t N, int64_t K, int32_t G, void* out, wq_stream_t stream);

/* ------------------------------------------------------------------ device status */

/* Reads the current device's status word: bit 0..3 = a bounded wait timed out in
 * the producer / MMA / transform / epilogue role, bit 4 = draining after a
 * timeout timed out, bit 5 = the wait probe timed out.  Synchronous (copies one
 * word); returns WQ_ERR_TIMEOUT when any bit is set. */
wq_status wq_device_status(uint32_t* bits);

/* Clears the current device's status word (synchronous). */
wq_status wq_clear_device_status(void);

/* Test hook: launches one CTA whose thread waits on an mbarrier that nothing
 * arrives on, with the kernels' bounded wait of `timeout_ns` nanoseconds.  The
 * wait runs out, the kernel sets bit 5 of the device status word and returns
 * normally, leaving the context usable. */
wq_status wq_debug_wait_probe(int64_t timeout_ns, wq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
