// wq_decode_int2.cuh -- INT2 (W2A16) decode kernel (M <= 16 tokens, G >= 64, K % 256 == 0).
//
// The register-resident scheme of the FP8 decode kernel (wq_decode_fp8.cuh) on the
// canonical INT2 codes W[N][K/4] (code k at bits 2 (k % 4) of byte k / 4; "Bitblas",
// hands-on item 6: W2A16, value (q - 2) * s[k / G, n]): per 256-code stage one 2-D TMA
// box of 128 weight rows x 64 bytes (64-byte swizzle) straight from W, one bulk copy of
// the stage's group scales (prepacked by wq_pack_int2_scales, the INT4 scale order) and
// one 3-D TMA of the activations.  The group scale multiplies the fp32 sums of each
// group (as in the W4A16 decode kernel), so an output is the sum over groups of
// s_g * sum_{k in g} A (q - 2), rounded once.
//
// Operand order.  ldmatrix gives lane (g, c) bytes 4c .. 4c + 3 of a 16-byte chunk of
// its rows g and g + 8: codes 16c .. 16c + 15 of a 64-code chunk, byte t holding codes
// 16c + 4t .. 16c + 4t + 3.  The chunk is four 16-wide k steps: in step t the lane's
// fragment positions 2c, 2c + 1, 2c + 8, 2c + 9 stand for codes 16c + 4t .. 16c + 4t + 3
// (an MMA sums over k in any order as long as both operands agree), so the lane's
// activation operands for steps 2tp and 2tp + 1 are one 16-byte load of those eight
// values of its token.  A step mixes codes from the whole 64-code chunk, which lies
// inside one group for G >= 64 (G = 32 stays on the tile kernel).
//
// Conversion: byte t copied into both 16-bit halves of a word (one byte permute); an
// AND-OR with a magic number per half turns the two codes of each half into b + q
// exactly (the code sits at bit 0 / 2 / 4 / 6 of its half, under an exponent whose
// mantissa unit there is 1: fp16 1024 / 256 / 64 / 16; bf16, with 7 mantissa bits, takes
// the codes at bits 0 / 2 only, 128 / 32, the upper pair after a shift by 4), and one
// subtraction of b + 2 gives q - 2.
//
// Every input is read after the kernel waits for the kernel before it on the stream
// (programmatic dependent launch): the weights and scales too, unlike the W4A16 decode
// kernel, as the INT2 entry point documents.
#pragma once

#include "wq_decode_fp8.cuh"

namespace wq {

// NT: 8-token MMA column tiles (1 for M <= 8, 2 for M <= 16).
template <int STAGES, int NT = 2>
struct Int2DecodeCfg {
    static constexpr int BK = 256;                        // codes per weight row per stage
    static constexpr int NCW = 4;                         // compute warps, 32 rows each
    static constexpr int RGW = TILE_N / 16 / NCW;         // 16-row groups per compute warp
    static constexpr int P_WARP = NCW;                    // producer warp
    static constexpr int NTHREADS = 32 * (NCW + 1);
    static constexpr int NZ = BK / 64;                    // 64-wide activation boxes per stage
    static constexpr int W_STAGE = TILE_N * BK / 4;       // one 128 x 64-byte box
    static constexpr int SC_STAGE = (BK / 64) * TILE_N * 2;   // up to 4 groups (G = 64) x 128 rows, fp16
    static constexpr int A_STAGE = 8 * NT * 128 * NZ;     // up to 8 NT token rows of 128 bytes per box
    static constexpr int SC_BASE = STAGES * W_STAGE;
    static constexpr int A_BASE = SC_BASE + STAGES * SC_STAGE;
    static constexpr int INBOX = A_BASE + STAGES * A_STAGE;
    static constexpr int INBOX_BYTES = inbox_row_pitch(NT) * (TILE_N + 16) * 4;   // fp32 [S][R][pitch], S * R <= 143
    static constexpr int OFF_BAR = INBOX + INBOX_BYTES;
    // barriers: full and empty per stage; then the abort flag (4 B, padded to 8) and the
    // inbox barrier (split-K)
    static constexpr int OFF_INBOX_BAR = OFF_BAR + 2 * STAGES * 8 + 8;
    static constexpr int SMEM_USED = OFF_INBOX_BAR + 8;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(W_STAGE % 1024 == 0 && SC_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "swizzle alignment");
};

// Byte t of w (codes q0 .. q3 at bits 8t, 8t + 2, 8t + 4, 8t + 6) -> lo = {q0, q1} - 2,
// hi = {q2, q3} - 2 as pairs of 16-bit values, exact.
template <bool BF16, int T>
__device__ __forceinline__ void int2_byte_to_operand(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = ptx::prmt(w, 0u, 0x4040u | (uint32_t)T | ((uint32_t)T << 8));   // byte t in bytes 0 and 2
    if (BF16) {
        // bf16 has 7 mantissa bits: a code at bits 6-7 of a half would reach the exponent,
        // so the upper pair is shifted down to the lower pair's positions first
        lo = sub_16x2(ptx::lop3_and_or(x, 0x000C0003u, 0x42004300u), 0x42084302u, true);          // 128 + q0, 32 + q1
        hi = sub_16x2(ptx::lop3_and_or(x >> 4, 0x000C0003u, 0x42004300u), 0x42084302u, true);     // 128 + q2, 32 + q3
    } else {
        lo = sub_16x2(ptx::lop3_and_or(x, 0x000C0003u, 0x5C006400u), 0x5C086402u, false);  // 1024 + q0, 256 + q1
        hi = sub_16x2(ptx::lop3_and_or(x, 0x00C00030u, 0x4C005400u), 0x4C805420u, false);  // 64 + q2, 16 + q3
    }
}

// GCH: 64-code chunks per scale group (G / 64: 1, 2 or 4).  One CTA per item (tile,
// K slice): gridDim.x == n_items, the slices of a tile form one cluster.
template <bool BF16, int NT, int STAGES, int GCH>
__global__ void __launch_bounds__(Int2DecodeCfg<STAGES, NT>::NTHREADS, 3)
    wq_decode_int2_kernel(const __grid_constant__ GemmParams p) {
    using C = Int2DecodeCfg<STAGES, NT>;
    constexpr int NCW = C::NCW;
    constexpr int RGW = C::RGW;
    constexpr int NZ = C::NZ;
    constexpr int CHUNKS = C::BK / 64;      // 64-code chunks per stage, four k steps each
    constexpr int SETS = NT == 1 ? 2 : 1;   // accumulator chains per row group (even / odd k steps)
    static_assert(GCH == 1 || GCH == 2 || GCH == 4, "G / 64");
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

    float acc[RGW][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.0f;

    if (warp == C::P_WARP) {
        // ------------------------------------------------------------ producer
        // Every copy waits for the preceding kernel (all inputs of this entry point may
        // be written by it).  A stage's phase cannot complete before the arrive-expect-tx
        // that counts all of its bytes.  The loop stops early only at a wait, and only
        // after issuing every copy of the stages armed so far.
        if (lane == 0) {
            ptx::grid_dependency_wait();
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint32_t a_bytes = (uint32_t)NZ * (uint32_t)p.a_box_rows * 128u;
            const uint32_t sc_bytes = (uint32_t)(CHUNKS / GCH) * TILE_N * 2;
            auto load = [&](int s, int kb) {
                const uint32_t fb = full_bar(s);
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)C::W_STAGE + sc_bytes + a_bytes);
                ptx::tma_load_2d(sbase + s * C::W_STAGE, &p.tmap_w, kb * (C::BK / 4), tile * TILE_N, fb, pol_w);
                const int g0 = (kb * C::BK) >> p.g_shift;
                ptx::bulk_load(sbase + C::SC_BASE + s * C::SC_STAGE,
                               p.sc + ((size_t)tile * p.ngroups_pad + g0) * (TILE_N * 2), sc_bytes, fb, pol_w);
                // activation box {64 k, M tokens, NZ}: k-block kb starts at z = kb * NZ
                ptx::tma_load_3d(sbase + C::A_BASE + s * C::A_STAGE, &p.tmap_a, 0, 0, kb * NZ, fb, pol_a);
            };
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int i = 0; i < nunits; ++i) {
                if (i >= STAGES &&
                    !bounded_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_PRODUCER, p.timeout_ns))
                    break;
                load(s, it.kb_begin + i);
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
        // ldmatrix.x4 per pair of chunks (2hp, 2hp + 1) and 16-row group: lane l addresses
        // row l % 8 of matrix l / 8 = (rows 0-7, chunk 2hp), (rows 8-15, chunk 2hp),
        // (rows 0-7, chunk 2hp + 1), (rows 8-15, chunk 2hp + 1); 64-byte rows, 64-byte
        // swizzle: 16-byte chunk index XOR address bits 7-8, i.e. (row / 2) % 4.
        const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1);
        uint32_t w_off[RGW][CHUNKS / 2];
#pragma unroll
        for (int j = 0; j < RGW; ++j) {
            const int row = (warp * RGW + j) * 16 + lrow;
#pragma unroll
            for (int hp = 0; hp < CHUNKS / 2; ++hp)
                w_off[j][hp] = (uint32_t)(row * 64 + (((2 * hp + (lane >> 4)) ^ ((row >> 1) & 3)) << 4));
        }
        // activation operands of chunk h, steps 2tp and 2tp + 1, MMA column g of tile nt
        // (token 8 nt + g): k = 64h + 16c + 8tp .. + 7, i.e. box h, bytes 32c + 16tp of the
        // token's 128-byte row, the 16-byte chunk 2c + tp (XOR the row's swizzle), one
        // 16-byte load for both steps.  A half-warp reads rows of four consecutive tokens,
        // two even and two odd: with the swizzle its 16 chunks fall on 8 chunk positions
        // twice, the two wavefronts 256 bytes need.
        uint32_t a_off[CHUNKS][NT];
#pragma unroll
        for (int h = 0; h < CHUNKS; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int row = h * p.a_box_rows + nt * 8 + g;
                a_off[h][nt] = (uint32_t)(row * 128 + (((2 * c) ^ (row & 7)) << 4));
            }
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nunits; ++i) {
            const bool ok = bounded_wait(full_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM,
                                         p.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t sw = sbase + s * C::W_STAGE;
            const uint32_t sa = sbase + C::A_BASE + s * C::A_STAGE;
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(smem + C::SC_BASE + s * C::SC_STAGE);
            float tmp[RGW][SETS][NT][4];
#pragma unroll
            for (int hp = 0; hp < CHUNKS / 2; ++hp) {
                uint32_t q[RGW][4];
#pragma unroll
                for (int j = 0; j < RGW; ++j) ldmatrix_x4(sw + w_off[j][hp], q[j][0], q[j][1], q[j][2], q[j][3]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int h = 2 * hp + u;
                    if (h % GCH == 0) {
#pragma unroll
                        for (int j = 0; j < RGW; ++j)
#pragma unroll
                            for (int x = 0; x < SETS; ++x)
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                    for (int e = 0; e < 4; ++e) tmp[j][x][nt][e] = 0.0f;
                    }
                    uint4 bv[2][NT];
#pragma unroll
                    for (int tp = 0; tp < 2; ++tp)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) bv[tp][nt] = ld_shared_v4(sa + (a_off[h][nt] ^ (uint32_t)(tp << 4)));
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        uint32_t b[NT][2];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4& v = bv[t >> 1][nt];
                            b[nt][0] = (t & 1) ? v.z : v.x;
                            b[nt][1] = (t & 1) ? v.w : v.y;
                        }
#pragma unroll
                        for (int j = 0; j < RGW; ++j) {
                            uint32_t a[4];
                            if (t == 0) {
                                int2_byte_to_operand<BF16, 0>(q[j][2 * u], a[0], a[2]);       // rows g
                                int2_byte_to_operand<BF16, 0>(q[j][2 * u + 1], a[1], a[3]);   // rows g + 8
                            } else if (t == 1) {
                                int2_byte_to_operand<BF16, 1>(q[j][2 * u], a[0], a[2]);
                                int2_byte_to_operand<BF16, 1>(q[j][2 * u + 1], a[1], a[3]);
                            } else if (t == 2) {
                                int2_byte_to_operand<BF16, 2>(q[j][2 * u], a[0], a[2]);
                                int2_byte_to_operand<BF16, 2>(q[j][2 * u + 1], a[1], a[3]);
                            } else {
                                int2_byte_to_operand<BF16, 3>(q[j][2 * u], a[0], a[2]);
                                int2_byte_to_operand<BF16, 3>(q[j][2 * u + 1], a[1], a[3]);
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma_16816(tmp[j][t % SETS][nt], a, b[nt][0], b[nt][1], BF16);
                        }
                    }
                    if (h % GCH == GCH - 1) {
                        // acc += s * sum_{k in group} A (q - 2)
                        const int gi = h / GCH;
#pragma unroll
                        for (int j = 0; j < RGW; ++j) {
                            const uint16_t* sp = sc + gi * TILE_N + (warp * RGW + j) * 16 + g;
                            const float s_lo = __half2float(__ushort_as_half(sp[0]));
                            const float s_hi = __half2float(__ushort_as_half(sp[8]));
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    float d = tmp[j][0][nt][e];
                                    if constexpr (SETS == 2) d += tmp[j][1][nt][e];
                                    acc[j][nt][e] = fmaf((e < 2) ? s_lo : s_hi, d, acc[j][nt][e]);
                                }
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
    ptx::grid_dependency_wait();   // out may still be read upstream
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
                        if (n < p.N && m < p.M) store_out<BF16>(p.out, (size_t)m * p.N + n, acc[j][nt][e]);
                    }
        }
    } else {
        ptx::cluster_wait();   // every CTA of the cluster has initialised its barriers
        if (warp < NCW) decode_send_partials<NT, RGW>(acc, warp, lane, rank, S, R, sbase + C::INBOX, inbox_bar);
        if (!bounded_wait<true>(inbox_bar, 0u, abort_flag, p.status, DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns)) return;
        decode_reduce_rows<NT, false>(reinterpret_cast<const float*>(smem + C::INBOX), S, R, rows_own, p.M,
                                     [&](int m, int r, float v) {
                                         const int n = tile * TILE_N + row0 + r;
                                         if (n < p.N) store_out<BF16>(p.out, (size_t)m * p.N + n, v);
                                     });
    }
}

template <bool BF16, int NT, int STAGES, int GCH>
struct Int2DecodeLauncher {
    using C = Int2DecodeCfg<STAGES, NT>;
    static constexpr auto kernel = wq_decode_int2_kernel<BF16, NT, STAGES, GCH>;
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
        KernelConfig k{FMT_INT2, BF16 ? 1 : 0, 8 * NT, C::BK, STAGES, 0, C::NTHREADS, C::SMEM_BYTES, 0, 1};
        if (!query_device || prepare() != cudaSuccess) return k;
        decode_residency(kernel, C::NTHREADS, C::SMEM_BYTES, &k);
        return k;
    }
    static cudaError_t launch(const GemmParams& p, int grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        if (p.splits > kMaxDecodeCluster || grid != p.n_items || p.M > 8 * NT || p.M < 1 || p.G < 64 ||
            p.G != 64 * GCH)
            return cudaErrorInvalidValue;
        return launch_decode_grid(kernel, p, grid, C::NTHREADS, C::SMEM_BYTES, st);
    }
};

}  // namespace wq
