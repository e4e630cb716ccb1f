// wq_gemm_lut_decode.cu -- the register-resident decode kernel (M <= 16, fp16
// activations) for the codebook INT4 format: operands LUT[q] from byte permutes over a
// 16-entry table held in registers, the group scale on the fp32 sums.  Same layouts,
// rings and split-K exchange as the symmetric decode kernel in wq_gemm_int4.cu.
#include "wq_gemm_mma.cuh"

namespace wq {

// Stages of 128 values (four): the table and the lookups raise the registers to
// 126-133 a thread, inside the three CTAs per SM the ring allows; stages of 256
// values would take 158-164 and leave two.
template <int NT, int GSTEPS, int BK>
using I4DecL = MmaDecodeLauncher<false, NT, GSTEPS, BK, 4, false, true>;

bool config_int4_decode_lut(bool query, KernelConfig* cfg) {
    *cfg = I4DecL<2, 8, 128>::config(query);
    return true;
}

template <int NT, int BK>
static cudaError_t launch_dec_lut_g(const GemmParams& p, int grid, cudaStream_t st) {
    switch (p.G) {
        case 32: return I4DecL<NT, 2, BK>::launch(p, grid, st);
        case 64: return I4DecL<NT, 4, BK>::launch(p, grid, st);
        case 128: return I4DecL<NT, 8, BK>::launch(p, grid, st);
        case 256: return I4DecL<NT, BK / 16, BK>::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_int4_decode_lut(const GemmParams& p, int grid, cudaStream_t st) {
    if (p.lut == nullptr) return cudaErrorInvalidValue;
    if (p.M <= 8) return launch_dec_lut_g<1, 128>(p, grid, st);
    if (p.M <= 16) return launch_dec_lut_g<2, 128>(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
