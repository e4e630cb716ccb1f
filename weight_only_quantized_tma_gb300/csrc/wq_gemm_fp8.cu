// wq_gemm_fp8.cu -- W8A16 (e4m3 weight) instantiations of the GEMM kernel.
#include "wq_gemm.cuh"

namespace wq {

using F8BF16_16 = GemmLauncher<FMT_FP8, true, 16, 128, 5, 2>;
using F8BF16_64 = GemmLauncher<FMT_FP8, true, 64, 128, 3, 2>;
using F8BF16_128 = GemmLauncher<FMT_FP8, true, 128, 128, 2, 2>;
using F8BF16_256 = GemmLauncher<FMT_FP8, true, 256, 64, 5, 2>;
using F8F16_16 = GemmLauncher<FMT_FP8, false, 16, 128, 5, 2>;
using F8F16_256 = GemmLauncher<FMT_FP8, false, 256, 64, 5, 2>;
// Large M: two-CTA clusters, 256 x 256 tiles, 128-value k-blocks: four activation
// stages (half a tile each), two weight stages and the 64 KB output staging area.
using F8F16_P = GemmLauncher<FMT_FP8, false, 256, 128, 4, 2, true, 2>;
using F8BF16_P = GemmLauncher<FMT_FP8, true, 256, 128, 4, 2, true, 2>;

bool config_fp8_pair(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? F8BF16_P::config(query) : F8F16_P::config(query);
    return true;
}

cudaError_t launch_gemm_fp8_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    return bf16 ? F8BF16_P::launch(p, grid, st) : F8F16_P::launch(p, grid, st);
}

bool config_fp8(bool bf16, int bn, bool query, KernelConfig* cfg) {
    if (bf16) {
        switch (bn) {
            case 16: *cfg = F8BF16_16::config(query);  return true;
            case 64: *cfg = F8BF16_64::config(query);  return true;
            case 128: *cfg = F8BF16_128::config(query);  return true;
            case 256: *cfg = F8BF16_256::config(query);  return true;
        }
    } else {
        switch (bn) {
            case 16: *cfg = F8F16_16::config(query);  return true;
            case 256: *cfg = F8F16_256::config(query);  return true;
        }
    }
    return false;
}

cudaError_t launch_gemm_fp8(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    if (bf16) {
        switch (bn) {
            case 16: return F8BF16_16::launch(p, grid, st);
            case 64: return F8BF16_64::launch(p, grid, st);
            case 128: return F8BF16_128::launch(p, grid, st);
            case 256: return F8BF16_256::launch(p, grid, st);
        }
    } else {
        switch (bn) {
            case 16: return F8F16_16::launch(p, grid, st);
            case 256: return F8F16_256::launch(p, grid, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace wq
