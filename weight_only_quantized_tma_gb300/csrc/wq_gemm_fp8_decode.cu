// wq_gemm_fp8_decode.cu -- FP8 (e4m3) decode instantiations (M <= 32, K % 64 == 0).
#include "wq_decode_fp8.cuh"

namespace wq {

// Stages of 128 values, 16 KB of weights each, two CTAs per SM: four stages up to 16
// tokens (the same bytes in flight per CTA as the W4A16 decode kernel), three for 17-32
// tokens, whose activation boxes and split-K inbox are twice as large.  The range ends
// at 32 tokens: measured on GB300 (bf16, in a CUDA graph, weights beyond L2), 10240 x
// 5120 takes 19.1 / 19.9 us at 24 / 32 tokens against 22.9 / 24.0 on the tile kernel,
// but an 8-tile variant for 33-64 tokens took 31.8 / 34.0 us at 48 / 64 against
// 24.6 / 25.3: at eight token tiles the mma.sync issue rate, not HBM, bounds the kernel.
template <bool BF16, int NT>
using F8Dec = Fp8DecodeLauncher<BF16, NT, NT <= 2 ? 4 : 3>;

template <int NT>
static KernelConfig fp8_decode_config(bool bf16, bool query) {
    return bf16 ? F8Dec<true, NT>::config(query) : F8Dec<false, NT>::config(query);
}

bool config_fp8_decode(bool bf16, int nt, bool query, KernelConfig* cfg) {
    switch (nt) {
        case 1: case 2: *cfg = fp8_decode_config<2>(bf16, query); return true;   // NT = 1 has NT = 2's memory
        case 4: *cfg = fp8_decode_config<4>(bf16, query); return true;
    }
    return false;
}

cudaError_t launch_gemm_fp8_decode(const GemmParams& p, bool bf16, int grid, cudaStream_t st) {
    if (p.M <= 8) return bf16 ? F8Dec<true, 1>::launch(p, grid, st) : F8Dec<false, 1>::launch(p, grid, st);
    if (p.M <= 16) return bf16 ? F8Dec<true, 2>::launch(p, grid, st) : F8Dec<false, 2>::launch(p, grid, st);
    if (p.M <= 32) return bf16 ? F8Dec<true, 4>::launch(p, grid, st) : F8Dec<false, 4>::launch(p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace wq
