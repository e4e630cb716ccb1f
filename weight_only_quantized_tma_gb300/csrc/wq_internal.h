// wq_internal.h -- declarations shared by the host API (wq_api.cu) and the kernel
// translation units.  Not part of the public C ABI (include/wq.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace wq {

// Weight formats of the tile kernel.  FMT_LUT4 is the INT4 layout with a 16-entry
// codebook in place of q - 8; FMT_INT2 holds canonical 2-bit codes [N][K/4] with
// the INT4 group-scale layout.
enum WFmt : int { FMT_INT4 = 0, FMT_FP8 = 1, FMT_FP4 = 2, FMT_LUT4 = 3, FMT_INT2 = 4 };
constexpr int kNumFmts = 5;
// the prepacked fragment-order INT4 code layout (wq_pack_int4)
__host__ __device__ constexpr bool int4_layout(int f) { return f == FMT_INT4 || f == FMT_LUT4; }
// fp16 group scales in the prepacked [N/128][Kp/G][128] layout, applied before the MMA
__host__ __device__ constexpr bool group_scaled(int f) { return f == FMT_INT4 || f == FMT_LUT4 || f == FMT_INT2; }

// Weight rows per CTA tile (the MMA M dimension: dequantized weight rows are the
// tcgen05 A operand, tokens are the N dimension).
constexpr int TILE_N = 128;

// INT4 kernel order (output of wq_pack_int4), N padded to 128 and K to 256:
//   [N/128][K/128][2 quads of 64 k][8 groups of 16 rows][32 slots][16 bytes]
// The 16 bytes of lane l = 4g + c (g = l / 4, c = l % 4) of a 16-row group hold,
// for the four 16-wide k steps t of the quad, one 32-bit word each: exactly the
// codes of the m16n8k16 A fragment of that lane --
//   bits  0- 3 / 16-19: row g,     k = 16t + 2c / 16t + 2c + 1
//   bits  4- 7 / 20-23: row g + 8, k = 16t + 2c / 16t + 2c + 1
//   bits  8-11 / 24-27: row g,     k = 16t + 8 + 2c / +1
//   bits 12-15 / 28-31: row g + 8, k = 16t + 8 + 2c / +1
// so one LOP3 with an fp16 "magic number" turns a nibble pair into a fragment
// register.  Lane l's 16 bytes sit at slot int4_slot(l): an XOR swizzle that keeps
// both a warp reading its lanes' slots (fragment order) and 8 threads gathering one
// row each (row order, the tcgen05 operand path) free of shared-memory bank conflicts.
__host__ __device__ __forceinline__ int int4_slot(int lane) {
    const int g = lane >> 2, c = lane & 3;
    return 4 * g + (c ^ ((g >> 1) & 3));
}
// Split-K workspace of the tile kernel: a fixed region of arrival counters (8 per
// output tile, room for kMaxSplitTiles tiles) at its start, then the fp32 partials.
// The counters must read zero when a call starts; every call leaves them zero.
constexpr int kMaxSplitTiles = 512;
constexpr size_t kSplitCounterBytes = (size_t)kMaxSplitTiles * 8 * sizeof(uint32_t);

// Padding granularity of the prepacked INT4 / FP4-scale layouts along K.
constexpr int KPAD_INT4 = 256;
constexpr int KPAD_FP4SF = 128;  // covers a whole k-block of the largest BK

// Division by a runtime constant with a multiply-shift.  For x < 2^31 and
// 1 <= d < 2^31, magic = ceil(2^(31+l) / d) with l = ceil(log2 d) gives
// floor(x * magic / 2^(31+l)) == x / d.  The product is only used when the
// largest dividend times magic fits in 63 bits; otherwise magic = 0 and the
// plain division is used.  (The overflow guard is the lesson of the
// magic-number division bug in "FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis",
// §3(b): a divisor of 1 produced a 2^40 magic that overflowed int64.)
struct FastDiv {
    uint32_t d;
    uint32_t shift;
    uint64_t magic;
};

inline FastDiv make_fastdiv(uint32_t d, uint32_t x_max) {
    FastDiv f{d, 0, 0};
    if (d == 0 || d >= (1u << 31) || x_max >= (1u << 31)) return f;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    uint32_t shift = 31 + l;
    unsigned __int128 num = ((unsigned __int128)1) << shift;
    uint64_t magic = (uint64_t)((num + d - 1) / d);
    // overflow guard: x_max * magic must stay below 2^63
    if (x_max != 0 && magic > (uint64_t)INT64_MAX / x_max) return f;
    f.shift = shift;
    f.magic = magic;
    return f;
}

__host__ __device__ __forceinline__ uint32_t fastdiv(uint32_t x, const FastDiv& f) {
    return f.magic ? (uint32_t)((x * f.magic) >> f.shift) : x / f.d;
}

// Everything a GEMM launch needs.  Passed by value as a __grid_constant__ so the
// tensor maps live in parameter space.
struct GemmParams {
    CUtensorMap tmap_a;      // activations [M][K], 16-bit, box {64, BN}, 128-byte swizzle
    CUtensorMap tmap_w;      // FP8 [N][K] / FP4 [N][K/2] weights (unused for INT4)
    CUtensorMap tmap_a_half; // activations, box half as high (half tiles)
    CUtensorMap tmap_out;    // pair kernel: out [M][N], 16-bit, box {128, 128}, no swizzle
    const uint8_t* w;        // INT4 prepacked weight tiles
    const uint8_t* sc;       // INT4 prepacked group scales / FP4 prepacked block scales
    const uint8_t* zp;       // INT4 prepacked zero points (uint8, the scales' layout) or null: zero point 8
    const uint16_t* lut;     // FMT_LUT4 codebook: 16 fp16 values, value LUT[q] * s
    const float* alpha;      // FP8 / FP4 global scale (device), unused for INT4
    const void* bias;        // FP8 optional bias [N], same 16-bit type as A
    void* out;               // [M][N], 16-bit
    int csplit;              // split-K slices of a tile are one thread-block cluster (no workspace)
    float* ws_part;          // split-K partials
    uint32_t* ws_count;      // split-K arrival tickets, one per output tile
    uint32_t* status;        // device status word (WQ_DEVICE_* bits)
    int M, N, K;
    int G;                   // INT4 group size
    int g_shift;             // log2(G)
    int tiles_n, tiles_m;    // output tiles along N (pair kernel: 256-row pairs) and M
    int splits;              // split-K slices per output tile
    int nkb;                 // k-blocks
    int a_box_rows;          // activation rows per TMA box (M when one token tile covers M, else BN)
    int a_box_rows_half;     // rows per box of tmap_a_half
    int kb_base, kb_rem;     // slice s covers kb_base * s + min(s, kb_rem) .. (nkb split as evenly as possible)
    int n_items;             // work items (tile kernel: n_full whole tiles, then two half tiles per remaining tile)
    int n_full;              // tile kernel: items below this are whole tiles (or split-K slices)
    int half_bn;             // tile kernel: tokens of a half tile (BN / 2)
    int walk_n_fast;         // tile walk order: weight rows fastest
    int w_evict_first;       // weights are streamed once (decode)
    int ngroups_pad;         // INT4: padded K / G
    int nchunks_pad;         // INT4: padded K / 32 ; FP4: padded K / 64
    FastDiv div_walk;        // divides a tile index by tiles_n (or tiles_m)
    FastDiv div_splits;      // divides an item index by splits
    long long timeout_ns;    // bound on every barrier wait
};

// Device status bits (OR-ed into *status by the kernels).
constexpr uint32_t DEVICE_TIMEOUT_PRODUCER = 1u << 0;
constexpr uint32_t DEVICE_TIMEOUT_MMA = 1u << 1;
constexpr uint32_t DEVICE_TIMEOUT_TRANSFORM = 1u << 2;
constexpr uint32_t DEVICE_TIMEOUT_EPILOGUE = 1u << 3;
constexpr uint32_t DEVICE_TIMEOUT_DRAIN = 1u << 4;

// Largest split-K cluster of the decode kernel (non-portable cluster size).
constexpr int kMaxDecodeCluster = 16;

// Static description of one compiled kernel configuration.
struct KernelConfig {
    int fmt;
    int bf16;
    int bn;          // token tile (MMA N)
    int bk;          // k per pipeline stage
    int stages;
    int nwg;         // transform warpgroups
    int threads;
    int smem_bytes;  // dynamic shared memory
    int tmem_cols;
    int ctas_per_sm;  // resident CTAs per SM (registers, shared and tensor memory)
    int max_clusters[kMaxDecodeCluster + 1];  // S-CTA clusters held at once (decode: S = 2..16; pair: S = 2)
    int pair;        // tile kernel on two-CTA clusters (tcgen05 cta_group::2, 256 weight rows per tile)
    int csplit_ok;   // tile kernel: split-K slices can be reduced inside a cluster (max_clusters[S])
};

// Per-format launch entry points, defined in wq_gemm_{int4,fp8,fp4}.cu.
// `bn` selects the instantiation; returns cudaErrorInvalidValue if none matches.
cudaError_t launch_gemm_int4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st);
cudaError_t launch_gemm_fp8(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st);
cudaError_t launch_gemm_fp4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st);
// Configuration of the instantiation for (bf16, bn); `query` asks the current
// device for the resident CTAs per SM.  False if no such instantiation exists.
bool config_int4(bool bf16, int bn, bool query, KernelConfig* cfg);
// W4A16 decode kernel (M <= 16, K % 64 == 0): register-resident mma.sync with the
// group scale applied on fp32, split-K reduced inside a thread-block cluster
// (wq_gemm_mma.cuh).  The configuration is that of the
// two-column-tile instantiation; both use the same shared memory and threads.
bool config_int4_decode(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int4_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
// The same decode kernel with per-(group, row) zero points (wq_gemm_zp_decode.cu).
bool config_int4_decode_zp(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int4_decode_zp(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
// The same decode kernel for the codebook format, fp16 activations (wq_gemm_lut_decode.cu).
bool config_int4_decode_lut(bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int4_decode_lut(const GemmParams& p, int grid, cudaStream_t st);
// INT2 decode kernel (M <= 16, G >= 64, K % 256 == 0): canonical 2-bit codes read through
// TMA, turned into q - 2 in registers (wq_decode_int2.cuh); `nt` 8-token tiles (1 or 2).
bool config_int2_decode(bool bf16, int nt, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int2_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
// FP8 decode kernel (M <= 32, K % 64 == 0): the same register-resident scheme on plain
// e4m3 weights read through TMA (wq_decode_fp8.cuh); `nt` 8-token column tiles (1, 2
// or 4) select the instantiation whose configuration is returned.
bool config_fp8_decode(bool bf16, int nt, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_fp8_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
// BF16 x FP4 decode kernel (M <= 16, K % 256 == 0): e2m1 codes and block scales turned
// into bf16 operands in registers (wq_decode_fp4.cuh).
bool config_fp4_decode(int nt, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_fp4_decode(const GemmParams& p, int grid, cudaStream_t st);
// W4A16 tile kernel on two-CTA clusters (256 weight rows x 256 tokens per tile).
bool config_int4_pair(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int4_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
bool config_fp8(bool bf16, int bn, bool query, KernelConfig* cfg);
// FP8 / FP4 tile kernels on two-CTA clusters (as the W4A16 pair kernel).
bool config_fp8_pair(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_fp8_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
bool config_fp4_pair(bool query, KernelConfig* cfg);
cudaError_t launch_gemm_fp4_pair(const GemmParams& p, int grid, cudaStream_t st);
bool config_fp4(bool bf16, int bn, bool query, KernelConfig* cfg);
// Codebook INT4 (FMT_LUT4) and INT2 tile kernels, one-CTA and pair.
bool config_lut4(bool bf16, int bn, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_lut4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st);
bool config_lut4_pair(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_lut4_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st);
bool config_int2(bool bf16, int bn, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int2(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st);
bool config_int2_pair(bool bf16, bool query, KernelConfig* cfg);
cudaError_t launch_gemm_int2_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st);

// Synthetic INT4 quantiser (fp16 [N][K] -> canonical codes and scales), wq_quant.cu.
cudaError_t launch_quantize_int4(const uint16_t* w, int64_t N, int64_t K, int G, uint8_t* wq, uint16_t* s,
                                 cudaStream_t st);

// Layout transforms, defined in wq_pack.cu.
cudaError_t launch_pack_int4(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K, int G, uint8_t* wk,
                             uint16_t* sk, cudaStream_t st);
cudaError_t launch_unpack_int4(const uint8_t* wk, const uint16_t* sk, int64_t N, int64_t K, int G, uint8_t* w,
                               uint16_t* s, cudaStream_t st);
cudaError_t launch_pack_int4_zeros(const uint8_t* z, int64_t N, int64_t K, int G, uint8_t* zk, cudaStream_t st);
cudaError_t launch_pack_group_scales(const uint16_t* s, int64_t N, int64_t K, int G, uint16_t* sk, cudaStream_t st);
cudaError_t launch_dequant_int2(const uint8_t* w, const uint16_t* sk, int64_t N, int64_t K, int G, float* out,
                                cudaStream_t st);
cudaError_t launch_dequant_int4(const uint8_t* wk, const uint16_t* sk, const uint16_t* lut, int64_t N, int64_t K,
                                int G, float* out, cudaStream_t st);
cudaError_t launch_pack_fp4_sf(const uint8_t* sf, int64_t N, int64_t K, uint8_t* sfk, cudaStream_t st);
cudaError_t launch_dequant_fp4(const uint8_t* w, const uint8_t* sfk, int64_t N, int64_t K, float* out,
                               cudaStream_t st);
cudaError_t launch_dequant_fp8(const uint8_t* w, int64_t N, int64_t K, bool bf16, float* out, cudaStream_t st);
cudaError_t launch_wait_probe(uint32_t* status, long long timeout_ns, cudaStream_t st);

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace wq
