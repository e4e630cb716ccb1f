// wq_gemm_int4.cu -- W4A16 instantiations of the GEMM kernel.
#include "wq_gemm.cuh"
#include "wq_gemm_mma.cuh"

namespace wq {

// (BN, BK, STAGES, NWG) per activation type.  BN <= 128 configurations fit two
// CTAs per SM (decode / split-K); BN = 256 runs one persistent CTA per SM with
// 128-value k-blocks: eight MMAs per pipeline hand-off (at 64 values per k-block
// the per-k-block hand-off, not the MMAs, bounded the kernel).
using I4F16_16 = GemmLauncher<FMT_INT4, false, 16, 128, 8, 2>;
using I4F16_64 = GemmLauncher<FMT_INT4, false, 64, 128, 4, 2>;
using I4F16_128 = GemmLauncher<FMT_INT4, false, 128, 128, 2, 2>;
using I4F16_256 = GemmLauncher<FMT_INT4, false, 256, 128, 3, 2>;
using I4BF16_16 = GemmLauncher<FMT_INT4, true, 16, 128, 8, 2>;
using I4BF16_256 = GemmLauncher<FMT_INT4, true, 256, 128, 3, 2>;
// Large M: two-CTA clusters, 256 x 256 tiles, each CTA holding half the activation
// tile: four activation stages (their reload latency bounds the k-block rate), three
// weight stages and the 64 KB output staging area.
using I4F16_P = GemmLauncher<FMT_INT4, false, 256, 128, 4, 2, true, 3>;
using I4BF16_P = GemmLauncher<FMT_INT4, true, 256, 128, 4, 2, true, 3>;

bool config_int4_pair(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? I4BF16_P::config(query) : I4F16_P::config(query);
    return true;
}

cudaError_t launch_gemm_int4_pair(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    return bf16 ? I4BF16_P::launch(p, grid, st) : I4F16_P::launch(p, grid, st);
}
// Decode (M <= 16): register-resident mma.sync kernel, one 8-token column tile for
// M <= 8, two for M <= 16, and the fold position (k steps per group) fixed at compile
// time.  Stages of 256 values (two of them) when K % 256 == 0, else of 128 (four): the
// same bytes in flight, half the per-stage barrier waits and hand-offs per byte.  The
// ring leaves room for three CTAs per SM, which then split K further: measured on
// GB300, in-graph decode step 74.6 us with three stages of 256 (two CTAs per SM) and
// 70.3 us with two (the 12288 x 4096 shapes 10.6 -> 8.7 us at M = 1, the 4096 x 4096
// ones 4.9 -> 5.5 us; choosing per shape measured 72.1 us: kernels with different
// footprints overlap worse across launches).  All instantiations share threads, shared
// memory and the cluster limits.
template <bool BF16, int NT, int GSTEPS, int BK>
using I4Dec = MmaDecodeLauncher<BF16, NT, GSTEPS, BK, BK == 256 ? 2 : 4>;
// three CTAs per SM: 228 KB of shared memory per SM, 1 KB reserved per CTA
static_assert(3 * (MmaDecodeCfg<256, 2>::SMEM_BYTES + 1024) <= 228 * 1024 &&
                  3 * (MmaDecodeCfg<128, 4>::SMEM_BYTES + 1024) <= 228 * 1024,
              "decode ring no longer fits three CTAs per SM");

bool config_int4_decode(bool bf16, bool query, KernelConfig* cfg) {
    *cfg = bf16 ? I4Dec<true, 2, 8, 128>::config(query) : I4Dec<false, 2, 8, 128>::config(query);
    return true;
}

template <bool BF16, int NT, int BK>
static cudaError_t launch_dec_g(const GemmParams& p, int grid, cudaStream_t st) {
    switch (p.G) {
        case 32: return I4Dec<BF16, NT, 2, BK>::launch(p, grid, st);
        case 64: return I4Dec<BF16, NT, 4, BK>::launch(p, grid, st);
        case 128: return I4Dec<BF16, NT, 8, BK>::launch(p, grid, st);
        case 256: return I4Dec<BF16, NT, BK / 16, BK>::launch(p, grid, st);
    }
    return cudaErrorInvalidValue;
}

template <bool BF16, int NT>
static cudaError_t launch_dec_bk(const GemmParams& p, int grid, cudaStream_t st) {
    return p.K % 256 == 0 ? launch_dec_g<BF16, NT, 256>(p, grid, st) : launch_dec_g<BF16, NT, 128>(p, grid, st);
}

cudaError_t launch_gemm_int4_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.M <= 8) return bf16 ? launch_dec_bk<true, 1>(p, grid, st) : launch_dec_bk<false, 1>(p, grid, st);
    if (p.M <= 16) return bf16 ? launch_dec_bk<true, 2>(p, grid, st) : launch_dec_bk<false, 2>(p, grid, st);
    return cudaErrorInvalidValue;
}

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
