// wq_gemm_int4.cu -- W4A16 instantiations of the GEMM kernel.
#include "wq_gemm.cuh"

namespace wq {

// (BN, BK, STAGES, NWG) per activation type.  BN <= 128 configurations fit two
// CTAs per SM (decode / split-K); BN = 256 runs one persistent CTA per SM.
using I4F16_16 = GemmLauncher<FMT_INT4, false, 16, 128, 8, 2>;
using I4F16_64 = GemmLauncher<FMT_INT4, false, 64, 128, 4, 2>;
using I4F16_128 = GemmLauncher<FMT_INT4, false, 128, 128, 2, 2>;
using I4F16_256 = GemmLauncher<FMT_INT4, false, 256, 64, 5, 2>;
using I4BF16_16 = GemmLauncher<FMT_INT4, true, 16, 128, 8, 2>;
using I4BF16_256 = GemmLauncher<FMT_INT4, true, 256, 64, 5, 2>;

bool config_int4(bool bf16, int bn, bool query, KernelConfig* cfg) {
    if (!bf16) {
        switch (bn) {
            case 16: *cfg = I4F16_16::config(query);  return true;
            case 64: *cfg = I4F16_64::config(query);  return true;
            case 128: *cfg = I4F16_128::config(query);  return true;
            case 256: *cfg = I4F16_256::config(query);  return true;
        }
    } else {
        switch (bn) {
            case 16: *cfg = I4BF16_16::config(query);  return true;
            case 256: *cfg = I4BF16_256::config(query);  return true;
        }
    }
    return false;
}

cudaError_t launch_gemm_int4(const GemmParams& p, bool bf16, int bn, int grid, cudaStream_t st) {
    if (!bf16) {
        switch (bn) {
            case 16: return I4F16_16::launch(p, grid, st);
            case 64: return I4F16_64::launch(p, grid, st);
            case 128: return I4F16_128::launch(p, grid, st);
            case 256: return I4F16_256::launch(p, grid, st);
        }
    } else {
        switch (bn) {
            case 16: return I4BF16_16::launch(p, grid, st);
            case 256: return I4BF16_256::launch(p, grid, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace wq
