// wq_gemm_int2_decode.cu -- INT2 (W2A16) decode instantiations (M <= 16, G >= 64,
// K % 256 == 0): three stages of 256 codes (8 KB of codes, up to 1 KB of scales and
// 4 or 8 KB of activations each), three CTAs per SM.
#include "wq_decode_int2.cuh"

namespace wq {

constexpr int kInt2DecodeStages = 3;

template <bool BF16, int NT>
static KernelConfig int2_decode_config(bool query) {
    return Int2DecodeLauncher<BF16, NT, kInt2DecodeStages, 2>::config(query);
}

bool config_int2_decode(bool bf16, int nt, bool query, KernelConfig* cfg) {
    if (nt == 1)
        *cfg = bf16 ? int2_decode_config<true, 1>(query) : int2_decode_config<false, 1>(query);
    else
        *cfg = bf16 ? int2_decode_config<true, 2>(query) : int2_decode_config<false, 2>(query);
    return true;
}

template <bool BF16, int NT>
static cudaError_t launch_dec_int2_g(const GemmParams& p, int grid, cudaStream_t st) {
    switch (p.G) {
        case 64: return Int2DecodeLauncher<BF16, NT, kInt2DecodeStages, 1>::launch(p, grid, st);
        case 128: return Int2DecodeLauncher<BF16, NT, kInt2DecodeStages, 2>::launch(p, grid, st);
        case 256: return Int2DecodeLauncher<BF16, NT, kInt2DecodeStages, 4>::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_int2_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.M <= 8) return bf16 ? launch_dec_int2_g<true, 1>(p, grid, st) : launch_dec_int2_g<false, 1>(p, grid, st);
    if (p.M <= 16) return bf16 ? launch_dec_int2_g<true, 2>(p, grid, st) : launch_dec_int2_g<false, 2>(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
