// wq_quant.cu -- synthetic group-wise symmetric INT4 quantiser, the step upstream of
// wq_pack_int4 ("Low Bit Triton Kernels", GPU MODE lecture 34, hands-on exercise 1:
// fp16 weight -> group-wise quantize -> two nibbles per byte).  Per (row n, group g):
//
//   S[g, n] = RN16(amax / 7),   amax = max over the group of |W[n, k]|
//   q[n, k] = clamp(rint(W[n, k] / S) + 8, 0, 15)      (rint: half to even; q = 8 if S = 0)
//
// Both decisions equal the exact rational roundings: amax / 7 is computed with IEEE
// division (__fdiv_rn) and is never within fp32 rounding of an fp16 tie; W / S is
// rounded exactly by rint_div below (no division per weight).  Outputs are the canonical
// layouts: packed codes [N][K/2] with even k in the low nibble, fp16 scales [K/G][N].
#include <cuda_fp16.h>
#include <cstdint>

#include "wq_internal.h"

namespace wq {
namespace {

// rint(x / s) for fp16 values x and s > 0 (rounding half to even) without a division
// per weight.  q0 = rint(x * (1 / s)) is within one of the answer (the product's
// relative error is ~2^-23 and |x / s| <= 7.5); the residual e = x - q0 s is exact in
// fp32 (x and q0 s are fp16-grid values within 14 significant bits of e), so
// comparing |e| with s / 2 decides: |e| < s/2 keeps q0, |e| > s/2 moves one step
// towards x, |e| == s/2 is a tie and takes the even neighbour.
__device__ __forceinline__ int rint_div(float x, float s, float inv) {
    float q = rintf(x * inv);
    const float e = fmaf(-q, s, x);
    const float ae = fabsf(e), h = 0.5f * s;
    if (ae > h) {
        q += copysignf(1.0f, e);
    } else if (ae == h) {
        const float q1 = q + copysignf(1.0f, e);
        if (((int)q1 & 1) == 0) q = q1;
    }
    return (int)q;
}

// One thread per 8 consecutive k of a row and per row of a group of R rows: the R
// 16-byte loads are issued before any is used, so each thread keeps R loads in flight
// (one would cap an SM at ~32 KB in flight, a third of what HBM needs).  Grid: x runs
// along a row in blocks of 256 threads, y over groups of R rows (a stride loop past
// 65535), so no thread divides.  The G / 8 threads of a scale group are aligned lanes
// of one warp (the row's K / 8 threads start at a block boundary, and G / 8 divides 32),
// so they combine amax with xor shuffles.
template <int G>
__global__ void __launch_bounds__(256) quantize_int4_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                            uint8_t* __restrict__ wq, uint16_t* __restrict__ s) {
    constexpr int TPG = G / 8;
    constexpr int R = 4;
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // 8-value chunk of the row
    const bool valid = j < K / 8;
    for (int64_t n0 = (int64_t)blockIdx.y * R; n0 < N; n0 += (int64_t)gridDim.y * R) {
        uint4 raw[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            raw[r] = make_uint4(0u, 0u, 0u, 0u);
            if (valid && n0 + r < N) raw[r] = __ldcs(reinterpret_cast<const uint4*>(w + (n0 + r) * K + j * 8));
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t n = n0 + r;
            const uint32_t words[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
            float x[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&words[i]));
                x[2 * i] = f.x;
                x[2 * i + 1] = f.y;
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
            for (int off = TPG / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
            const float sv = __half2float(sh);
            const float inv = sv != 0.0f ? __frcp_rn(sv) : 0.0f;
            uint32_t packed = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int q = 8;
                if (sv != 0.0f) {
                    q = rint_div(x[i], sv, inv) + 8;
                    q = q < 0 ? 0 : (q > 15 ? 15 : q);
                }
                packed |= (uint32_t)q << (4 * i);   // k = 8j + i: byte 4j + i / 2, even k in the low nibble
            }
            if (valid && n < N) {
                *reinterpret_cast<uint32_t*>(wq + n * (K / 2) + j * 4) = packed;
                if (j % TPG == 0) s[(j / TPG) * N + n] = __half_as_ushort(sh);
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize_int4(const uint16_t* w, int64_t N, int64_t K, int G, uint8_t* wq, uint16_t* s,
                                 cudaStream_t st) {
    const int64_t row_groups = (N + 3) / 4;
    const dim3 grid((unsigned)((K / 8 + 255) / 256), (unsigned)(row_groups < 65535 ? row_groups : 65535));
    switch (G) {
        case 32: quantize_int4_kernel<32><<<grid, 256, 0, st>>>(w, N, K, wq, s); break;
        case 64: quantize_int4_kernel<64><<<grid, 256, 0, st>>>(w, N, K, wq, s); break;
        case 128: quantize_int4_kernel<128><<<grid, 256, 0, st>>>(w, N, K, wq, s); break;
        case 256: quantize_int4_kernel<256><<<grid, 256, 0, st>>>(w, N, K, wq, s); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaPeekAtLastError();
}

}  // namespace wq
