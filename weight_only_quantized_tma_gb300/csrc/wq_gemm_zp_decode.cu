// wq_gemm_zp_decode.cu -- the register-resident decode kernel (M <= 16) for zero-point
// INT4: the operands are q - z, with the zero points of each group and row streamed
// beside the scales.  Same shapes and instantiation grid as the symmetric decode
// kernel in wq_gemm_int4.cu.
#include "wq_gemm_mma.cuh"

namespace wq {

template <bool BF16, int NT, int GSTEPS, int BK>
using I4DecZ = MmaDecodeLauncher<BF16, NT, GSTEPS, BK, BK == 256 ? 3 : 6, true>;

bool config_int4_decode_zp(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? I4DecZ<true, 2, 8, 128>::config(query) : I4DecZ<false, 2, 8, 128>::config(query);
    return true;
}

template <bool BF16, int NT, int BK>
static cudaError_t launch_dec_zp_g(const GemmParams& p, int grid, cudaStream_t st) {
    switch (p.G) {
        case 32: return I4DecZ<BF16, NT, 2, BK>::launch(p, grid, st);
        case 64: return I4DecZ<BF16, NT, 4, BK>::launch(p, grid, st);
        case 128: return I4DecZ<BF16, NT, 8, BK>::launch(p, grid, st);
        case 256: return I4DecZ<BF16, NT, BK / 16, BK>::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

template <bool BF16, int NT>
static cudaError_t launch_dec_zp_bk(const GemmParams& p, int grid, cudaStream_t st) {
    return p.K % 256 == 0 ? launch_dec_zp_g<BF16, NT, 256>(p, grid, st) : launch_dec_zp_g<BF16, NT, 128>(p, grid, st);
}

cudaError_t launch_gemm_int4_decode_zp(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.zp == nullptr) return cudaErrorInvalidValue;
    if (p.M <= 8) return bf16 ? launch_dec_zp_bk<true, 1>(p, grid, st) : launch_dec_zp_bk<false, 1>(p, grid, st);
    if (p.M <= 16) return bf16 ? launch_dec_zp_bk<true, 2>(p, grid, st) : launch_dec_zp_bk<false, 2>(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
