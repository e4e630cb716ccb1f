// wq_gemm_zp_decode.cu -- the register-resident decode kernel (M <= 16) for zero-point
// INT4: each group's fold adds (8 - z) S_g[m] per row, with the zero points streamed
// beside the scales.  Same shapes and instantiation grid as the symmetric decode
// kernel in wq_gemm_int4.cu.
#include "wq_gemm_mma.cuh"

namespace wq {

template <bool BF16, int NT, int GSTEPS>
using I4DecZ = MmaDecodeLauncher<BF16, NT, GSTEPS, 128, 6, true>;

bool config_int4_decode_zp(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? I4DecZ<true, 2, 8>::config(query) : I4DecZ<false, 2, 8>::config(query);
    return true;
}

template <bool BF16, int NT>
static cudaError_t launch_dec_zp_g(const GemmParams& p, int grid, cudaStream_t st) {
    switch (p.G) {
        case 32: return I4DecZ<BF16, NT, 2>::launch(p, grid, st);
        case 64: return I4DecZ<BF16, NT, 4>::launch(p, grid, st);
        case 128:
        case 256: return I4DecZ<BF16, NT, 8>::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_int4_decode_zp(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.zp == nullptr) return cudaErrorInvalidValue;
    if (p.M <= 8) return bf16 ? launch_dec_zp_g<true, 1>(p, grid, st) : launch_dec_zp_g<false, 1>(p, grid, st);
    if (p.M <= 16) return bf16 ? launch_dec_zp_g<true, 2>(p, grid, st) : launch_dec_zp_g<false, 2>(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
