// wq_gemm_fp4_decode.cu -- BF16 x FP4 decode instantiations (M <= 16, K % 256 == 0).
#include "wq_decode_fp4.cuh"

namespace wq {

// Two stages of 256 codes (16 KB of codes, 2 KB of block scales and 4 or 8 KB of
// activations each): four CTAs per SM for M <= 8, three for M <= 16.  The operand
// conversion makes this kernel instruction-bound, and more warps per SM hide more of
// its latency (measured on GB300, in a CUDA graph: M = 1, 12800 x 5120, 17.1 us with
// three stages and two CTAs per SM, 13.3 us with two and three; M = 16 20.8 and 15.9
// us; M = 1, 6656 x 19968, 27.5 us at three CTAs per SM and 24.6 at four, while
// 12800 x 5120 stays at 13.3 us; the FP8 decode kernel, lighter per byte, loses at
// three CTAs per SM: 11.1 -> 15.7 us at M = 1).
constexpr int kFp4DecodeStages = 2;

bool config_fp4_decode(int nt, bool query, KernelConfig* cfg) {
    *cfg = nt == 1 ? Fp4DecodeLauncher<1, kFp4DecodeStages>::config(query)
                   : Fp4DecodeLauncher<2, kFp4DecodeStages>::config(query);
    return true;
}

cudaError_t launch_gemm_fp4_decode(const GemmParams& p, int grid, cudaStream_t st) {
    if (p.M <= 8) return Fp4DecodeLauncher<1, kFp4DecodeStages>::launch(p, grid, st);
    if (p.M <= 16) return Fp4DecodeLauncher<2, kFp4DecodeStages>::launch(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
