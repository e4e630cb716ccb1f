// wq_decode_fp4.cuh -- BF16 x FP4 decode kernel (M <= 16 tokens).
//
// The register-resident scheme of the FP8 decode kernel (wq_decode_fp8.cuh) on e2m1
// codes W[N][K/2] with one e4m3 scale per 16 codes along K and a global alpha
// ("FlashInfer SM100 BF16 x FP4 GEMM", §2: uint8 weight [N, K/2], block scales per
// 16 values, alpha on the accumulator).  Per 256-code stage: one 2-D TMA box of 128
// weight rows x 128 bytes (128-byte swizzle, straight from W), one bulk copy of the
// stage's block scales (prepacked by wq_pack_fp4_sf: [K/64][128 rows][4 scales] per
// tile) and one 3-D TMA of the activations.
//
// Operand order.  ldmatrix gives lane (g, c) bytes 4c .. 4c + 3 of a 16-byte chunk of
// its rows g and g + 8: codes 8c .. 8c + 7 of a 32-code chunk (even k in the low
// nibble).  The chunk is two 16-wide k steps: in the first the lane's fragment
// positions 2c, 2c + 1, 2c + 8, 2c + 9 stand for codes 8c .. 8c + 3, in the second for
// 8c + 4 .. 8c + 7, so the lane's activation operand for both steps is the eight
// consecutive values k = 8c .. 8c + 7 of its token (one 16-byte load), and all eight
// codes of the lane share one block scale (block 2 chunk + c / 2).  The operand value
// e2m1 * e4m3 is exact: both convert exactly to fp16, their product has at most 5
// significant bits inside fp16's normal range, and it widens exactly to bf16.
#pragma once

#include "wq_decode_fp8.cuh"

namespace wq {

// NT: 8-token MMA column tiles; the activation stages and the split-K inbox hold 8 NT
// tokens, so the one-tile kernel (M <= 8) fits four CTAs per SM.
template <int STAGES, int NT = 2>
struct Fp4DecodeCfg {
    static constexpr int BK = 256;                       // codes per weight row per stage
    static constexpr int NCW = 4;                        // compute warps, 32 rows each
    static constexpr int RGW = TILE_N / 16 / NCW;        // 16-row groups per compute warp
    static constexpr int P_WARP = NCW;                   // producer warp
    static constexpr int NTHREADS = 32 * (NCW + 1);
    static constexpr int NZ = BK / 64;                   // 64-wide activation boxes per stage
    static constexpr int W_STAGE = TILE_N * BK / 2;      // one 128 x 128-byte box
    static constexpr int SF_STAGE = TILE_N * BK / 16;    // [BK / 64 quads][128 rows][4 scales]
    static constexpr int A_STAGE = 8 * NT * 128 * NZ;    // up to 8 NT token rows of 128 bytes per box
    static constexpr int SF_BASE = STAGES * W_STAGE;
    static constexpr int A_BASE = SF_BASE + STAGES * SF_STAGE;
    static constexpr int INBOX = A_BASE + STAGES * A_STAGE;
    static constexpr int INBOX_BYTES = inbox_row_pitch(NT) * (TILE_N + 16) * 4;   // fp32 [S][R][pitch], S * R <= 128 + 15
    static constexpr int OFF_BAR = INBOX + INBOX_BYTES;
    // barriers: full and empty per stage; then the abort flag (4 B, padded to 8) and the
    // inbox barrier (split-K)
    static constexpr int OFF_INBOX_BAR = OFF_BAR + 2 * STAGES * 8 + 8;
    static constexpr int SMEM_USED = OFF_INBOX_BAR + 8;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(W_STAGE % 1024 == 0 && A_BASE % 1024 == 0 && A_STAGE % 1024 == 0, "swizzle alignment");
};

// One lane's eight codes of a row (byte i: codes 2i, 2i + 1) times the block scale
// (s2 = {s, s} in fp16) -> four bf16 pairs, exact.
__device__ __forceinline__ void e2m1x8_scaled_to_bf16(uint32_t q, uint32_t s2, uint32_t (&o)[4]) {
    uint32_t h[4];
    ptx::e2m1x8_to_f16x2x4(q, h);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = ptx::f16x2_to_bf16x2_exact(ptx::hmul2_u32(h[i], s2));
}

// NT: 8-token MMA column tiles (1 for M <= 8, 2 for M <= 16).  One CTA per item
// (tile, K slice): gridDim.x == n_items, the slices of a tile form one cluster.
template <int NT, int STAGES>
__global__ void __launch_bounds__(Fp4DecodeCfg<STAGES, NT>::NTHREADS, NT == 1 ? 4 : 3)
    wq_decode_fp4_kernel(const __grid_constant__ GemmParams p) {
    using C = Fp4DecodeCfg<STAGES, NT>;
    constexpr int NCW = C::NCW;
    constexpr int RGW = C::RGW;
    constexpr int NZ = C::NZ;
    constexpr int CHUNKS = C::BK / 32;      // 32-code chunks per stage, two k steps each
    constexpr int SETS = NT == 1 ? 2 : 1;   // accumulator chains per row group (even / odd k steps)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + 2 * STAGES * 8);
    const uint32_t inbox_bar = sbase + C::OFF_INBOX_BAR;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Item it = decode_item(p, (int)blockIdx.x);
    const int nunits = it.kb_end - it.kb_begin;
    const int tile = it.n_tile;
    const int S = p.splits;
    const int R = (TILE_N + S - 1) / S;   // inbox rows per slice: an owner's rows, at most
    const int rank = S > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int row0 = rank * TILE_N / S;     // this CTA's rows of the tile: [row0, row0 + rows_own)
    const int rows_own = (rank + 1) * TILE_N / S - row0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), NCW);
        }
        ptx::mbar_init(inbox_bar, 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
        if (S > 1) ptx::mbar_arrive_expect_tx(inbox_bar, (uint32_t)(S * rows_own * NT * 32));
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::P_WARP && lane == 0) {
        ptx::prefetch_tmap(&p.tmap_w);
        ptx::prefetch_tmap(&p.tmap_a);
    }
    __syncthreads();
    if (S > 1) ptx::cluster_arrive_relaxed();
    if (threadIdx.x == 0) ptx::grid_launch_dependents();

    float acc[RGW][SETS][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int h = 0; h < SETS; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][h][nt][e] = 0.0f;

    if (warp == C::P_WARP) {
        // ------------------------------------------------------------ producer
        // As in the FP8 decode kernel: the first STAGES weight and scale copies go out
        // before the grid dependency wait (constant inputs), activations after it; every
        // armed barrier gets all of its bytes before the loop can stop at a wait.
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint32_t a_bytes = (uint32_t)NZ * (uint32_t)p.a_box_rows * 128u;
            const int pre = nunits < STAGES ? nunits : STAGES;
            auto load_w = [&](int s, int kb) {
                ptx::mbar_arrive_expect_tx(full_bar(s), (uint32_t)(C::W_STAGE + C::SF_STAGE) + a_bytes);
                ptx::tma_load_2d(sbase + s * C::W_STAGE, &p.tmap_w, kb * (C::BK / 2), tile * TILE_N, full_bar(s),
                                 pol_w);
                const uint8_t* sf = p.sc + ((size_t)tile * p.nchunks_pad + (size_t)kb * (C::BK / 64)) * (TILE_N * 4);
                ptx::bulk_load(sbase + C::SF_BASE + s * C::SF_STAGE, sf, C::SF_STAGE, full_bar(s), pol_w);
            };
            // activation box {64 k, M tokens, NZ}: k-block kb starts at z = kb * NZ
            auto load_a = [&](int s, int kb) {
                ptx::tma_load_3d(sbase + C::A_BASE + s * C::A_STAGE, &p.tmap_a, 0, 0, kb * NZ, full_bar(s), pol_a);
            };
            for (int i = 0; i < pre; ++i) load_w(i, it.kb_begin + i);
            ptx::grid_dependency_wait();
            for (int i = 0; i < pre; ++i) load_a(i, it.kb_begin + i);
            int s = pre % STAGES;
            uint32_t ph = pre == STAGES ? 1u : 0u;
            int issued = pre;
            for (int i = pre; i < nunits; ++i) {
                if (!bounded_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_PRODUCER,
                                  p.timeout_ns))
                    break;
                load_w(s, it.kb_begin + i);
                load_a(s, it.kb_begin + i);
                ++issued;
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                const int first = issued > STAGES ? issued - STAGES : 0;
                for (int j = first; j < issued; ++j)
                    if (!drain_wait(full_bar(j % STAGES), (uint32_t)((j / STAGES) & 1), p.timeout_ns))
                        atomicOr(p.status, DEVICE_TIMEOUT_DRAIN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute warps
        const int g = lane >> 2, c = lane & 3;
        // ldmatrix.x4 per pair of chunks (2h, 2h + 1) and 16-row group: lane l addresses
        // row l % 8 of matrix l / 8 = (rows 0-7, chunk 2h), (rows 8-15, chunk 2h),
        // (rows 0-7, chunk 2h + 1), (rows 8-15, chunk 2h + 1); a chunk is one 16-byte
        // piece of the 128-byte row, at index ^ (row % 8) after the swizzle
        const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t w_row = (uint32_t)(warp * RGW * 16 + lrow) * 128u;
        uint32_t w_chunk[CHUNKS / 2];
#pragma unroll
        for (int h = 0; h < CHUNKS / 2; ++h) w_chunk[h] = (uint32_t)(((2 * h + (lane >> 4)) ^ (lane & 7)) << 4);
        // activation operand of chunk jc, token 8 nt + g: k = 32 jc + 8c .. + 7, i.e.
        // box jc / 2, 16-byte piece 4 (jc % 2) + c of the token's 128-byte row
        uint32_t a_off[CHUNKS][NT];
#pragma unroll
        for (int jc = 0; jc < CHUNKS; ++jc)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int row = (jc >> 1) * p.a_box_rows + nt * 8 + g;
                const int piece = 4 * (jc & 1) + c;
                a_off[jc][nt] = (uint32_t)(row * 128 + ((piece ^ (row & 7)) << 4));
            }
        // block scales of rows g and g + 8 of row group j: byte 4 row + (block % 4) of
        // quad block / 4, block = 2 jc + c / 2
        const int sf_row = (warp * RGW) * 16 + g;
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nunits; ++i) {
            const bool ok = bounded_wait(full_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM,
                                         p.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t sw = sbase + s * C::W_STAGE + w_row;
            const uint8_t* sfs = smem + C::SF_BASE + s * C::SF_STAGE;
            const uint32_t sa = sbase + C::A_BASE + s * C::A_STAGE;
#pragma unroll
            for (int h = 0; h < CHUNKS / 2; ++h) {
                uint32_t q[RGW][4];
#pragma unroll
                for (int j = 0; j < RGW; ++j)
                    ldmatrix_x4(sw + j * 16 * 128 + w_chunk[h], q[j][0], q[j][1], q[j][2], q[j][3]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int jc = 2 * h + u;
                    uint4 b[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) b[nt] = ld_shared_v4(sa + a_off[jc][nt]);
                    const uint8_t* sfq = sfs + (jc >> 1) * (TILE_N * 4) + 2 * (jc & 1) + (c >> 1);
#pragma unroll
                    for (int j = 0; j < RGW; ++j) {
                        const uint32_t b_lo = sfq[(sf_row + j * 16) * 4], b_hi = sfq[(sf_row + j * 16 + 8) * 4];
                        const uint32_t s_lo = ptx::e4m3x2_to_f16x2((uint16_t)(b_lo | (b_lo << 8)));
                        const uint32_t s_hi = ptx::e4m3x2_to_f16x2((uint16_t)(b_hi | (b_hi << 8)));
                        uint32_t lo[4], hi[4];
                        e2m1x8_scaled_to_bf16(q[j][2 * u], s_lo, lo);       // rows g
                        e2m1x8_scaled_to_bf16(q[j][2 * u + 1], s_hi, hi);   // rows g + 8
                        const uint32_t a0[4] = {lo[0], hi[0], lo[1], hi[1]};   // codes 8c .. 8c + 3
                        const uint32_t a1[4] = {lo[2], hi[2], lo[3], hi[3]};   // codes 8c + 4 .. 8c + 7
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_16816(acc[j][0][nt], a0, b[nt].x, b[nt].y, true);
                            mma_16816(acc[j][SETS - 1][nt], a1, b[nt].z, b[nt].w, true);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty_bar(s));
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
    // Every stage was consumed, or drained after an abort.  From here on every thread
    // of the CTA runs the same sequence (no early exit before the cluster wait).
    __syncthreads();
    ptx::grid_dependency_wait();   // alpha is an input; out may still be read upstream
    float sum[RGW][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sum[j][nt][e] = SETS == 2 ? acc[j][0][nt][e] + acc[j][SETS - 1][nt][e] : acc[j][0][nt][e];
    const float alpha = __ldg(p.alpha);
    if (p.splits == 1) {
        if (warp < NCW) {
            const int g = lane >> 2, c = lane & 3;
#pragma unroll
            for (int j = 0; j < RGW; ++j)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int n = tile * TILE_N + (warp * RGW + j) * 16 + g + 8 * (e >> 1);
                        const int m = nt * 8 + 2 * c + (e & 1);
                        if (n < p.N && m < p.M) store_out<true>(p.out, (size_t)m * p.N + n, alpha * sum[j][nt][e]);
                    }
        }
    } else {
        ptx::cluster_wait();   // every CTA of the cluster has initialised its barriers
        if (warp < NCW) decode_send_partials<NT, RGW>(sum, warp, lane, rank, S, R, sbase + C::INBOX, inbox_bar);
        if (!bounded_wait<true>(inbox_bar, 0u, abort_flag, p.status, DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns)) return;
        decode_reduce_rows<NT>(reinterpret_cast<const float*>(smem + C::INBOX), S, R, rows_own, p.M,
                           [&](int m, int r, float v) {
                               const int n = tile * TILE_N + row0 + r;
                               if (n < p.N) store_out<true>(p.out, (size_t)m * p.N + n, alpha * v);
                           });
    }
}

template <int NT, int STAGES>
struct Fp4DecodeLauncher {
    using C = Fp4DecodeCfg<STAGES, NT>;
    static constexpr auto kernel = wq_decode_fp4_kernel<NT, STAGES>;
    static cudaError_t prepare() {
        static int attr_set[64] = {0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 64 && attr_set[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess && dev < 64) attr_set[dev] = 1;
        return e;
    }
    static KernelConfig config(bool query_device) {
        KernelConfig k{FMT_FP4, 1, 16, C::BK, STAGES, 0, C::NTHREADS, C::SMEM_BYTES, 0, 1};
        if (!query_device || prepare() != cudaSuccess) return k;
        decode_residency(kernel, C::NTHREADS, C::SMEM_BYTES, &k);
        return k;
    }
    static cudaError_t launch(const GemmParams& p, int grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        if (p.splits > kMaxDecodeCluster || grid != p.n_items || p.M > 8 * NT || p.M < 1) return cudaErrorInvalidValue;
        return launch_decode_grid(kernel, p, grid, C::NTHREADS, C::SMEM_BYTES, st);
    }
};

}  // namespace wq
