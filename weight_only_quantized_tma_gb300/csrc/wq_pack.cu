// wq_pack.cu -- offline layout transforms, debug exports and the wait probe.
//
// INT4 kernel order (output of wq_pack_int4): see wq_internal.h.  The
// permutation is the offline layout transform of "Bitblas -- Mixed-Precision GEMM
// with the Ladder Compiler" (GPU MODE lecture 33), introduction: the packed codes
// are stored in the order the tensor-core operand fragments want, so no layout
// conversion sits on the GEMM's critical path.
//   scales:  [N/128][K/G][128 rows] fp16
//
// FP4 block-scale kernel order (output of wq_pack_fp4_sf), N padded to 128 and K
// to 128:  [N/128][K/64][128 rows][4 bytes], byte b of (tile, quad, row) is the
// e4m3 scale of k in [64*quad + 16b, +16).
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "wq_gemm.cuh"
#include "wq_internal.h"

namespace wq {

namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t work) {
    int64_t g = (work + kThreads - 1) / kThreads;
    if (g > 65535LL * 32) g = 65535LL * 32;
    return (int)(g < 1 ? 1 : g);
}

__device__ __forceinline__ uint32_t canon_code(const uint8_t* w, int64_t N, int64_t K, int64_t n, int64_t k) {
    if (n >= N || k >= K) return 8u;
    const uint8_t b = w[n * (K / 2) + k / 2];
    return (k & 1) ? (uint32_t)(b >> 4) : (uint32_t)(b & 0xF);
}

// One thread per 16-byte unit: (tile, k-block, quad, group, lane).
__global__ void pack_int4_w_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K, int64_t nkb,
                                   int64_t units, uint8_t* __restrict__ wk) {
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int lane = (int)(u % 32);
        const int64_t t1 = u / 32;
        const int gr = (int)(t1 % 8);
        const int64_t t2 = t1 / 8;
        const int tq = (int)(t2 % 2);
        const int64_t t3 = t2 / 2;
        const int64_t kb = t3 % nkb;
        const int64_t tile = t3 / nkb;
        const int g = lane >> 2, c = lane & 3;
        const int64_t n_lo = tile * TILE_N + gr * 16 + g, n_hi = n_lo + 8;
        uint32_t words[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int64_t k0 = kb * 128 + 16 * (4 * tq + t) + 2 * c, k2 = k0 + 8;
            words[t] = canon_code(w, N, K, n_lo, k0) | (canon_code(w, N, K, n_lo, k0 + 1) << 16) |
                       (canon_code(w, N, K, n_hi, k0) << 4) | (canon_code(w, N, K, n_hi, k0 + 1) << 20) |
                       (canon_code(w, N, K, n_lo, k2) << 8) | (canon_code(w, N, K, n_lo, k2 + 1) << 24) |
                       (canon_code(w, N, K, n_hi, k2) << 12) | (canon_code(w, N, K, n_hi, k2 + 1) << 28);
        }
        const int64_t dst = (u - lane) + int4_slot(lane);
        reinterpret_cast<uint4*>(wk)[dst] = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

__global__ void pack_int4_s_kernel(const uint16_t* __restrict__ s, int64_t N, int64_t groups, int64_t groups_pad,
                                   int64_t total, uint16_t* __restrict__ sk) {
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = u % TILE_N;
        const int64_t t = u / TILE_N;
        const int64_t g = t % groups_pad;
        const int64_t nt = t / groups_pad;
        const int64_t n = nt * TILE_N + r;
        sk[u] = (n < N && g < groups) ? s[g * N + n] : (uint16_t)0;
    }
}

// Code of weight (n, k) read back from the kernel-order layout.
__device__ __forceinline__ uint32_t packed_code(const uint8_t* wk, int64_t nkb, int64_t n, int64_t k) {
    const int64_t tile = n / TILE_N;
    const int r = (int)(n % TILE_N);
    const int gr = r / 16, h = (r % 16) / 8, g = r % 8;
    const int64_t kb = k / 128;
    const int kl = (int)(k % 128);
    const int tabs = kl / 16, kk = kl % 16;
    const int hi8 = kk / 8, c = (kk % 8) / 2, odd = kk & 1;
    const int tq = tabs / 4, t = tabs % 4;
    const int lane = 4 * g + c;
    const int64_t unit = (((tile * nkb + kb) * 2 + tq) * 8 + gr) * 32 + int4_slot(lane);
    const uint32_t word = reinterpret_cast<const uint32_t*>(wk + unit * 16)[t];
    return (word >> (4 * (h + 2 * hi8) + 16 * odd)) & 0xFu;
}

__global__ void unpack_int4_w_kernel(const uint8_t* __restrict__ wk, int64_t N, int64_t K, int64_t nkb,
                                     uint8_t* __restrict__ w) {
    const int64_t total = N * (K / 2);
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = u / (K / 2), j = u % (K / 2);
        const uint32_t lo = packed_code(wk, nkb, n, 2 * j);
        const uint32_t hi = packed_code(wk, nkb, n, 2 * j + 1);
        w[u] = (uint8_t)(lo | (hi << 4));
    }
}

__global__ void unpack_int4_s_kernel(const uint16_t* __restrict__ sk, int64_t N, int64_t groups, int64_t groups_pad,
                                     uint16_t* __restrict__ s) {
    const int64_t total = groups * N;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = u / N, n = u % N;
        s[u] = sk[((n / TILE_N) * groups_pad + g) * TILE_N + (n % TILE_N)];
    }
}

// (q - 8) * s, or LUT[q] * s with a codebook; both products are exact in fp32.
__global__ void dequant_int4_kernel(const uint8_t* __restrict__ wk, const uint16_t* __restrict__ sk,
                                    const uint16_t* __restrict__ lut, int64_t N, int64_t K, int G, int64_t nkb,
                                    int64_t groups_pad, float* __restrict__ out) {
    const int64_t total = N * K;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = u / K, k = u % K;
        const int q = (int)packed_code(wk, nkb, n, k);
        const uint16_t sb = sk[((n / TILE_N) * groups_pad + k / G) * TILE_N + (n % TILE_N)];
        const float v = lut ? __half2float(__ushort_as_half(lut[q])) : (float)(q - 8);
        out[u] = v * __half2float(__ushort_as_half(sb));
    }
}

__global__ void pack_fp4_sf_kernel(const uint8_t* __restrict__ sf, int64_t N, int64_t K16, int64_t quads,
                                   int64_t total, uint8_t* __restrict__ sfk) {
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = u % 4;
        const int64_t r = (u / 4) % TILE_N;
        const int64_t t = u / (4 * TILE_N);
        const int64_t qd = t % quads;
        const int64_t nt = t / quads;
        const int64_t n = nt * TILE_N + r;
        const int64_t k16 = qd * 4 + b;
        sfk[u] = (n < N && k16 < K16) ? sf[n * K16 + k16] : (uint8_t)0;
    }
}

// One thread per (row, 32-code chunk): the GEMM transform's FP4 conversion.
__global__ void dequant_fp4_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ sfk, int64_t N,
                                   int64_t K, int64_t quads, float* __restrict__ out) {
    const int64_t chunks = K / 32;
    const int64_t total = N * chunks;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = u / chunks, c = u % chunks;
        const uint8_t* src = w + n * (K / 2) + c * 16;
        uint32_t wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            wv[j] = (uint32_t)src[4 * j] | ((uint32_t)src[4 * j + 1] << 8) | ((uint32_t)src[4 * j + 2] << 16) |
                    ((uint32_t)src[4 * j + 3] << 24);
        const uint4 q = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        const uint8_t* sfp = sfk + (((n / TILE_N) * quads + c / 2) * TILE_N + (n % TILE_N)) * 4 + (c & 1) * 2;
        const uint16_t pair = (uint16_t)(sfp[0] | (sfp[1] << 8));
        uint32_t o[16];
        fp4_to_bf16(q, pair, o);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            out[n * K + c * 32 + 2 * t] = __uint_as_float(o[t] << 16);
            out[n * K + c * 32 + 2 * t + 1] = __uint_as_float(o[t] & 0xFFFF0000u);
        }
    }
}

// One thread per (row, 16-code chunk): the GEMM transform's FP8 conversion.
template <bool BF16>
__global__ void dequant_fp8_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K, float* __restrict__ out) {
    const int64_t chunks = K / 16;
    const int64_t total = N * chunks;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = u / chunks, c = u % chunks;
        const uint8_t* src = w + n * K + c * 16;
        uint32_t wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            wv[j] = (uint32_t)src[4 * j] | ((uint32_t)src[4 * j + 1] << 8) | ((uint32_t)src[4 * j + 2] << 16) |
                    ((uint32_t)src[4 * j + 3] << 24);
        uint32_t o[8];
        fp8_to_operand<BF16>(make_uint4(wv[0], wv[1], wv[2], wv[3]), o);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float lo, hi;
            if (BF16) {
                lo = __uint_as_float(o[t] << 16);
                hi = __uint_as_float(o[t] & 0xFFFF0000u);
            } else {
                lo = __half2float(__ushort_as_half((uint16_t)(o[t] & 0xFFFFu)));
                hi = __half2float(__ushort_as_half((uint16_t)(o[t] >> 16)));
            }
            out[n * K + c * 16 + 2 * t] = lo;
            out[n * K + c * 16 + 2 * t + 1] = hi;
        }
    }
}

// Waits on a barrier nothing ever arrives on; the bounded wait must give up.
__global__ void wait_probe_kernel(uint32_t* status, long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = bounded_wait(ptx::smem_u32(&bar), 0, &abort_flag, status, 1u << 5, timeout_ns);
        (void)ok;
    }
    __syncthreads();
}

}  // namespace

__global__ void stream_fence_kernel() {}

cudaError_t launch_pack_int4(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K, int G, uint8_t* wk,
                             uint16_t* sk, cudaStream_t st) {
    const int64_t Np = round_up(N, TILE_N), Kp = round_up(K, KPAD_INT4);
    const int64_t nkb = Kp / 128, units = (Np / TILE_N) * nkb * 2 * 8 * 32;
    pack_int4_w_kernel<<<grid_for(units), kThreads, 0, st>>>(w, N, K, nkb, units, wk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t groups_pad = Kp / G, total = (Np / TILE_N) * groups_pad * TILE_N;
    pack_int4_s_kernel<<<grid_for(total), kThreads, 0, st>>>(s, N, K / G, groups_pad, total, sk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The decode GEMM may start while the kernel before it on the stream is still
    // finishing and reads the packed weights before it waits for that kernel.  An
    // ordinary (non-overlapping) launch after the pack kernels makes sure that kernel
    // is never one that wrote them.
    stream_fence_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

// Group scales alone (INT2: the codes stay canonical), in the INT4 scale layout;
// ends with an ordinary launch for the same reason as launch_pack_int4.
cudaError_t launch_pack_group_scales(const uint16_t* s, int64_t N, int64_t K, int G, uint16_t* sk, cudaStream_t st) {
    const int64_t Np = round_up(N, TILE_N), Kp = round_up(K, KPAD_INT4);
    const int64_t groups_pad = Kp / G, total = (Np / TILE_N) * groups_pad * TILE_N;
    pack_int4_s_kernel<<<grid_for(total), kThreads, 0, st>>>(s, N, K / G, groups_pad, total, sk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    stream_fence_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

// INT2 debug export: (q - 2) * s from canonical codes [N][K/4] and packed scales.
__global__ void dequant_int2_kernel(const uint8_t* __restrict__ w, const uint16_t* __restrict__ sk, int64_t N,
                                    int64_t K, int G, int64_t groups_pad, float* __restrict__ out) {
    const int64_t total = N * K;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = u / K, k = u % K;
        const int q = (w[n * (K / 4) + k / 4] >> (2 * (k % 4))) & 0x3;
        const uint16_t sb = sk[((n / TILE_N) * groups_pad + k / G) * TILE_N + (n % TILE_N)];
        out[u] = (float)(q - 2) * __half2float(__ushort_as_half(sb));
    }
}

cudaError_t launch_dequant_int2(const uint8_t* w, const uint16_t* sk, int64_t N, int64_t K, int G, float* out,
                                cudaStream_t st) {
    const int64_t Kp = round_up(K, KPAD_INT4);
    dequant_int2_kernel<<<grid_for(N * K), kThreads, 0, st>>>(w, sk, N, K, G, Kp / G, out);
    return cudaGetLastError();
}

// Zero points: canonical uint8 [K/G][N] -> [N/128][Kp/G][128], the layout of the packed
// scales; padding gets 8 (with scale 0 the weight is 0 either way).
__global__ void pack_int4_z_kernel(const uint8_t* __restrict__ z, int64_t N, int64_t groups, int64_t groups_pad,
                                   int64_t total, uint8_t* __restrict__ zk) {
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = u % TILE_N;
        const int64_t t = u / TILE_N;
        const int64_t g = t % groups_pad;
        const int64_t nt = t / groups_pad;
        const int64_t n = nt * TILE_N + r;
        zk[u] = (n < N && g < groups) ? z[g * N + n] : (uint8_t)8;
    }
}

cudaError_t launch_pack_int4_zeros(const uint8_t* z, int64_t N, int64_t K, int G, uint8_t* zk, cudaStream_t st) {
    const int64_t Np = round_up(N, TILE_N), Kp = round_up(K, KPAD_INT4);
    const int64_t groups_pad = Kp / G, total = (Np / TILE_N) * groups_pad * TILE_N;
    pack_int4_z_kernel<<<grid_for(total), kThreads, 0, st>>>(z, N, K / G, groups_pad, total, zk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    stream_fence_kernel<<<1, 32, 0, st>>>();   // as after the weight packing
    return cudaGetLastError();
}

cudaError_t launch_unpack_int4(const uint8_t* wk, const uint16_t* sk, int64_t N, int64_t K, int G, uint8_t* w,
                               uint16_t* s, cudaStream_t st) {
    const int64_t Kp = round_up(K, KPAD_INT4);
    unpack_int4_w_kernel<<<grid_for(N * (K / 2)), kThreads, 0, st>>>(wk, N, K, Kp / 128, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    unpack_int4_s_kernel<<<grid_for((K / G) * N), kThreads, 0, st>>>(sk, N, K / G, Kp / G, s);
    return cudaGetLastError();
}

cudaError_t launch_dequant_int4(const uint8_t* wk, const uint16_t* sk, const uint16_t* lut, int64_t N, int64_t K,
                                int G, float* out, cudaStream_t st) {
    const int64_t Kp = round_up(K, KPAD_INT4);
    dequant_int4_kernel<<<grid_for(N * K), kThreads, 0, st>>>(wk, sk, lut, N, K, G, Kp / 128, Kp / G, out);
    return cudaGetLastError();
}

cudaError_t launch_pack_fp4_sf(const uint8_t* sf, int64_t N, int64_t K, uint8_t* sfk, cudaStream_t st) {
    const int64_t Np = round_up(N, TILE_N), quads = round_up(K, KPAD_FP4SF) / 64;
    const int64_t total = (Np / TILE_N) * quads * TILE_N * 4;
    pack_fp4_sf_kernel<<<grid_for(total), kThreads, 0, st>>>(sf, N, K / 16, quads, total, sfk);
    return cudaGetLastError();
}

cudaError_t launch_dequant_fp4(const uint8_t* w, const uint8_t* sfk, int64_t N, int64_t K, float* out,
                               cudaStream_t st) {
    const int64_t quads = round_up(K, KPAD_FP4SF) / 64;
    dequant_fp4_kernel<<<grid_for(N * (K / 32)), kThreads, 0, st>>>(w, sfk, N, K, quads, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_fp8(const uint8_t* w, int64_t N, int64_t K, bool bf16, float* out, cudaStream_t st) {
    if (bf16)
        dequant_fp8_kernel<true><<<grid_for(N * (K / 16)), kThreads, 0, st>>>(w, N, K, out);
    else
        dequant_fp8_kernel<false><<<grid_for(N * (K / 16)), kThreads, 0, st>>>(w, N, K, out);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint32_t* status, long long timeout_ns, cudaStream_t st) {
    wait_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace wq
