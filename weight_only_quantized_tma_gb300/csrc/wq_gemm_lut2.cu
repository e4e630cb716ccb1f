// wq_gemm_lut2.cu -- instantiations of the GEMM kernel for the codebook INT4 format
// (FMT_LUT4: the prepacked INT4 layout, value LUT[q] * s) and for INT2 (FMT_INT2:
// canonical 2-bit codes, value (q - 2) * s).  Both run on the tile kernels at every
// M, with the INT4 tile shapes: BN = 16 / 64 / 128 / 256 one-CTA tiles (fp16
// activations; 16 and 256 for bf16) and the two-CTA pair tile for large M.
#include "wq_gemm.cuh"

namespace wq {

template <int FMT, bool BF16, int BN>
struct TileShape;
template <int FMT, bool BF16> struct TileShape<FMT, BF16, 16> { using L = GemmLauncher<FMT, BF16, 16, 128, 8, 2>; };
template <int FMT, bool BF16> struct TileShape<FMT, BF16, 64> { using L = GemmLauncher<FMT, BF16, 64, 128, 4, 2>; };
template <int FMT, bool BF16> struct TileShape<FMT, BF16, 128> { using L = GemmLauncher<FMT, BF16, 128, 128, 2, 2>; };
template <int FMT, bool BF16> struct TileShape<FMT, BF16, 256> { using L = GemmLauncher<FMT, BF16, 256, 128, 3, 2>; };
template <int FMT, bool BF16>
using PairShape = GemmLauncher<FMT, BF16, 256, 128, 4, 2, true, 3>;

template <int FMT>
static bool config_fmt(bool bf16, int bn, bool query, KernelConfig* cfg) {
    if (!bf16) {
        switch (bn) {
            case 16: *cfg = TileShape<FMT, false, 16>::L::config(query); return true;
            case 64: *cfg = TileShape<FMT, false, 64>::L::config(query); return true;
            case 128: *cfg = TileShape<FMT, false, 128>::L::config(query); return true;
            case 256: *cfg = TileShape<FMT, false, 256>::L::config(query); return true;
        }
    } else {
        switch (bn) {
            case 16: *cfg = TileShape<FMT, true, 16>::L::config(query); return true;
            case 256: *cfg = TileShape<FMT, true, 256>::L::config(query); return true;
        }
    }
    return false;
}

template <int FMT>
static cudaError_t launch_fmt(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    if (!bf16) {
        switch (bn) {
            case 16: return TileShape<FMT, false, 16>::L::launch(p, grid, st);
            case 64: return TileShape<FMT, false, 64>::L::launch(p, grid, st);
            case 128: return TileShape<FMT, false, 128>::L::launch(p, grid, st);
            case 256: return TileShape<FMT, false, 256>::L::launch(p, grid, st);
        }
    } else {
        switch (bn) {
            case 16: return TileShape<FMT, true, 16>::L::launch(p, grid, st);
            case 256: return TileShape<FMT, true, 256>::L::launch(p, grid, st);
        }
    }
    return cudaErrorInvalidValue;
}

bool config_lut4(bool bf16, int bn, bool query, KernelConfig* cfg) { return config_fmt<FMT_LUT4>(bf16, bn, query, cfg); }
cudaError_t launch_gemm_lut4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    return launch_fmt<FMT_LUT4>(p, bf16, bn, grid, st);
}
bool config_lut4_pair(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? PairShape<FMT_LUT4, true>::config(query) : PairShape<FMT_LUT4, false>::config(query);
    return true;
}
cudaError_t launch_gemm_lut4_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    return bf16 ? PairShape<FMT_LUT4, true>::launch(p, grid, st) : PairShape<FMT_LUT4, false>::launch(p, grid, st);
}

bool config_int2(bool bf16, int bn, bool query, KernelConfig* cfg) { return config_fmt<FMT_INT2>(bf16, bn, query, cfg); }
cudaError_t launch_gemm_int2(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    return launch_fmt<FMT_INT2>(p, bf16, bn, grid, st);
}
bool config_int2_pair(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? PairShape<FMT_INT2, true>::config(query) : PairShape<FMT_INT2, false>::config(query);
    return true;
}
cudaError_t launch_gemm_int2_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    return bf16 ? PairShape<FMT_INT2, true>::launch(p, grid, st) : PairShape<FMT_INT2, false>::launch(p, grid, st);
}

}  // namespace wq
