// wq_gemm_fp8_decode.cu -- FP8 (e4m3) decode instantiations (M <= 16, K % 64 == 0).
#include "wq_decode_fp8.cuh"

namespace wq {

// Four stages of 128 values: 16 KB of weights each, the same bytes in flight per CTA
// as the W4A16 decode kernel's three 256-value stages, and two CTAs per SM.
constexpr int kFp8DecodeStages = 4;
template <bool BF16, int NT>
using F8Dec = Fp8DecodeLauncher<BF16, NT, kFp8DecodeStages>;

bool config_fp8_decode(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? F8Dec<true, 2>::config(query) : F8Dec<false, 2>::config(query);
    return true;
}

cudaError_t launch_gemm_fp8_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.M <= 8) return bf16 ? F8Dec<true, 1>::launch(p, grid, st) : F8Dec<false, 1>::launch(p, grid, st);
    if (p.M <= 16) return bf16 ? F8Dec<true, 2>::launch(p, grid, st) : F8Dec<false, 2>::launch(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
