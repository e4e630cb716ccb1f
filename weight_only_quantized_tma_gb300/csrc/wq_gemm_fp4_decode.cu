// wq_gemm_fp4_decode.cu -- BF16 x FP4 decode instantiations (M <= 16, K % 256 == 0).
#include "wq_decode_fp4.cuh"

namespace wq {

// Three stages of 256 codes: 16 KB of codes, 2 KB of block scales and up to 8 KB of
// activations each; two CTAs per SM.
constexpr int kFp4DecodeStages = 3;

bool config_fp4_decode(bool query, KernelConfig* cfg) {
    *cfg = Fp4DecodeLauncher<2, kFp4DecodeStages>::config(query);
    return true;
}

cudaError_t launch_gemm_fp4_decode(const GemmParams& p, int grid, cudaStream_t st) {
    if (p.M <= 8) return Fp4DecodeLauncher<1, kFp4DecodeStages>::launch(p, grid, st);
    if (p.M <= 16) return Fp4DecodeLauncher<2, kFp4DecodeStages>::launch(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
