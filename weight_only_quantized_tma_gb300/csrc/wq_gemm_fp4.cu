// wq_gemm_fp4.cu -- BF16 x FP4 (e2m1 weight, e4m3 block scales) instantiations.
#include "wq_gemm.cuh"

namespace wq {

using F4_16 = GemmLauncher<FMT_FP4, true, 16, 128, 8, 2>;
using F4_64 = GemmLauncher<FMT_FP4, true, 64, 128, 4, 2>;
using F4_128 = GemmLauncher<FMT_FP4, true, 128, 128, 2, 2>;
using F4_256 = GemmLauncher<FMT_FP4, true, 256, 128, 3, 2>;
// Large M: two-CTA clusters (as the W4A16 pair kernel).
using F4_P = GemmLauncher<FMT_FP4, true, 256, 128, 4, 2, true, 3>;

bool config_fp4_pair(bool query, KernelConfig* cfg) {
    *cfg = F4_P::config(query);
    return true;
}

cudaError_t launch_gemm_fp4_pair(const GemmParams& p, int grid, cudaStream_t st) { return F4_P::launch(p, grid, st); }

bool config_fp4(bool bf16, int bn, bool query, KernelConfig* cfg) {
    if (!bf16) return false;
    switch (bn) {
        case 16: *cfg = F4_16::config(query);  return true;
        case 64: *cfg = F4_64::config(query);  return true;
        case 128: *cfg = F4_128::config(query);  return true;
        case 256: *cfg = F4_256::config(query);  return true;
    }
    return false;
}

cudaError_t launch_gemm_fp4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    if (!bf16) return cudaErrorInvalidValue;
    switch (bn) {
        case 16: return F4_16::launch(p, grid, st);
        case 64: return F4_64::launch(p, grid, st);
        case 128: return F4_128::launch(p, grid, st);
        case 256: return F4_256::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace wq
