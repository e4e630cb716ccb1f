// wq_decode_fp8.cuh -- FP8 (e4m3) decode kernel (M <= 32 tokens).
//
// The register-resident scheme of the W4A16 decode kernel (wq_gemm_mma.cuh) on plain
// e4m3 weights W[N][K]: TMA copies 128-row x 128-byte weight boxes (128-byte swizzle)
// and the matching activation boxes into a ring of stages; each compute warp reads
// its rows with ldmatrix, converts the codes to the 16-bit MMA operand type (exact:
// every e4m3 value is an fp16 and a bf16 value) and accumulates with mma.sync in fp32.
// The per-tensor scale alpha and the optional bias are applied once, in the epilogue:
// the scale multiplies the fp32 accumulator ("FlashInfer W8A16 GEMM (mm_bf16_fp8)
// analysis", introduction, and §2 for the bias argument of mm_bf16_fp8).
//
// Operand order.  ldmatrix gives lane (g, c) the four consecutive codes 4c .. 4c + 3
// of a 16-wide k step of its rows g and g + 8.  An MMA sums over its k index in any
// order as long as the weight and the activation operands agree, so the lane's
// fragment positions 2c, 2c + 1, 2c + 8, 2c + 9 stand for k = 4c, 4c + 1, 4c + 2,
// 4c + 3 of the step, and the lane's activation operand is the four consecutive values
// k = 4c .. 4c + 3 of its token: one 8-byte shared-memory load.  No layout transform
// of the weights is needed, offline or in the kernel.  MMA column n of an 8-token
// tile holds token 2 (n % 4) + n / 4, so that the 8-byte loads of a half-warp read
// even (or odd) token rows, which the 128-byte swizzle puts on distinct banks.
//
// Work split, pipeline and split-K are those of the W4A16 decode kernel: one CTA per
// (128-row tile, K slice), warps 0-3 compute 32 rows each, warp 4 is the producer, the
// K slices of a tile are one thread-block cluster reducing through st.async.
#pragma once

#include "wq_gemm_mma.cuh"

namespace wq {

// NT: 8-token MMA column tiles per row group (1, 2 or 4: M up to 32).
template <int STAGES, int NT = 2>
struct Fp8DecodeCfg {
    static constexpr int BK = 128;                       // k values (= weight bytes per row) per stage
    static constexpr int NCW = 4;                        // compute warps, 32 rows each
    static constexpr int RGW = TILE_N / 16 / NCW;        // 16-row groups per compute warp
    static constexpr int P_WARP = NCW;                   // producer warp
    static constexpr int NTHREADS = 32 * (NCW + 1);
    static constexpr int NZ = BK / 64;                   // 64-wide activation boxes per stage
    static constexpr int W_STAGE = TILE_N * BK;          // one 128 x 128-byte box, 1024-byte aligned
    static constexpr int NTA = NT < 2 ? 2 : NT;
    static constexpr int A_STAGE = 8 * NTA * 128 * NZ;   // up to 8 NTA token rows of 128 bytes per box
    static constexpr int A_BASE = STAGES * W_STAGE;
    static constexpr int INBOX = A_BASE + STAGES * A_STAGE;
    static constexpr int INBOX_BYTES = inbox_row_pitch(NT) * (TILE_N + 16) * 4;   // fp32 [S][R][row], S * R <= 143
    static constexpr int OFF_BAR = INBOX + INBOX_BYTES;
    // barriers: full and empty per stage; then the abort flag (4 B, padded to 8) and the
    // inbox barrier (split-K)
    static constexpr int OFF_INBOX_BAR = OFF_BAR + 2 * STAGES * 8 + 8;
    static constexpr int SMEM_USED = OFF_INBOX_BAR + 8;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(W_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "swizzle alignment");
};

// Four e4m3 codes (byte i = k 4c + i) -> the operand registers of their fragment
// positions: lo = {k 4c, 4c + 1}, hi = {k 4c + 2, 4c + 3}, exact.
template <bool BF16>
__device__ __forceinline__ void e4m3x4_to_operand(uint32_t q, uint32_t& lo, uint32_t& hi) {
    lo = ptx::e4m3x2_to_f16x2((uint16_t)(q & 0xFFFFu));
    hi = ptx::e4m3x2_to_f16x2((uint16_t)(q >> 16));
    if (BF16) {
        lo = ptx::f16x2_to_bf16x2_exact(lo);
        hi = ptx::f16x2_to_bf16x2_exact(hi);
    }
}

__device__ __forceinline__ void ld_shared_v2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// NT: 8-token MMA column tiles (1 for M <= 8, 2 for M <= 16, 4 for M <= 32).  One CTA per item (tile, K slice): gridDim.x == n_items, the slices of a
// tile form one cluster.
template <bool BF16, int NT, int STAGES>
__global__ void __launch_bounds__(Fp8DecodeCfg<STAGES, NT>::NTHREADS, 2)
    wq_decode_fp8_kernel(const __grid_constant__ GemmParams p) {
    using C = Fp8DecodeCfg<STAGES, NT>;
    constexpr int NCW = C::NCW;
    constexpr int RGW = C::RGW;
    constexpr int NZ = C::NZ;
    constexpr int KSTEPS = C::BK / 16;
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
        // The first STAGES weight boxes go out before the grid dependency wait (constant
        // input); activations only after it.  A stage's phase cannot complete before the
        // arrive-expect-tx that counts all of its bytes, so the order in which they land
        // does not matter.  The loop stops early only at a wait, and only after issuing
        // every copy of the stages armed so far, so every armed barrier gets its bytes.
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint32_t a_bytes = (uint32_t)NZ * (uint32_t)p.a_box_rows * 128u;
            const int pre = nunits < STAGES ? nunits : STAGES;
            auto load_w = [&](int s, int kb) {
                ptx::mbar_arrive_expect_tx(full_bar(s), (uint32_t)C::W_STAGE + a_bytes);
                ptx::tma_load_2d(sbase + s * C::W_STAGE, &p.tmap_w, kb * C::BK, tile * TILE_N, full_bar(s), pol_w);
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
        // ldmatrix.x4 per pair of k steps (2h, 2h + 1) and 16-row group: lane l addresses
        // row l % 8 of matrix l / 8 = (rows 0-7, step 2h), (rows 8-15, step 2h),
        // (rows 0-7, step 2h + 1), (rows 8-15, step 2h + 1); a step is one 16-byte chunk
        // of the 128-byte row, at chunk ^ (row % 8) after the swizzle.
        const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t w_row = (uint32_t)(warp * RGW * 16 + lrow) * 128u;
        uint32_t w_chunk[KSTEPS / 2];
#pragma unroll
        for (int h = 0; h < KSTEPS / 2; ++h) w_chunk[h] = (uint32_t)(((2 * h + (lane >> 4)) ^ (lane & 7)) << 4);
        // activation operand of step t, MMA column g of tile nt (token 8 nt + 2 (g % 4) +
        // g / 4, spread over the banks): k = 16 t + 4c .. + 3, i.e. box t / 4, byte
        // 32 (t % 4) + 8c of the token's 128-byte row
        uint32_t a_off[KSTEPS][NT];
#pragma unroll
        for (int t = 0; t < KSTEPS; ++t)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int row = (t >> 2) * p.a_box_rows + nt * 8 + token_of_column<true>(g);
                const int chunk = 2 * (t & 3) + (c >> 1);
                a_off[t][nt] = (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4) + 8 * (c & 1));
            }
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nunits; ++i) {
            const bool ok = bounded_wait(full_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM,
                                         p.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t sw = sbase + s * C::W_STAGE + w_row;
            const uint32_t sa = sbase + C::A_BASE + s * C::A_STAGE;
#pragma unroll
            for (int h = 0; h < KSTEPS / 2; ++h) {
                uint32_t q[RGW][4];
#pragma unroll
                for (int j = 0; j < RGW; ++j) ldmatrix_x4(sw + j * 16 * 128 + w_chunk[h], q[j][0], q[j][1], q[j][2], q[j][3]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = 2 * h + u;
                    uint32_t b[NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) ld_shared_v2(sa + a_off[t][nt], b[nt][0], b[nt][1]);
#pragma unroll
                    for (int j = 0; j < RGW; ++j) {
                        uint32_t a[4];
                        e4m3x4_to_operand<BF16>(q[j][2 * u], a[0], a[2]);       // rows g
                        e4m3x4_to_operand<BF16>(q[j][2 * u + 1], a[1], a[3]);   // rows g + 8
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_16816(acc[j][t % SETS][nt], a, b[nt][0], b[nt][1], BF16);
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
    ptx::grid_dependency_wait();   // alpha and bias are inputs; out may still be read upstream
    float sum[RGW][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sum[j][nt][e] = SETS == 2 ? acc[j][0][nt][e] + acc[j][SETS - 1][nt][e] : acc[j][0][nt][e];
    const float alpha = __ldg(p.alpha);
    auto finish = [&](int m, int n, float v) {
        float b = 0.0f;
        if (p.bias != nullptr) b = load_16bit<BF16>(p.bias, (size_t)n);
        store_out<BF16>(p.out, (size_t)m * p.N + n, alpha * v + b);
    };
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
                        const int m = nt * 8 + token_of_column<true>(2 * c + (e & 1));
                        if (n < p.N && m < p.M) finish(m, n, sum[j][nt][e]);
                    }
        }
    } else {
        ptx::cluster_wait();   // every CTA of the cluster has initialised its barriers
        if (warp < NCW) decode_send_partials<NT, RGW>(sum, warp, lane, rank, S, R, sbase + C::INBOX, inbox_bar);
        if (!bounded_wait<true>(inbox_bar, 0u, abort_flag, p.status, DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns)) return;
        decode_reduce_rows<NT, true>(reinterpret_cast<const float*>(smem + C::INBOX), S, R, rows_own, p.M,
                           [&](int m, int r, float v) {
                               const int n = tile * TILE_N + row0 + r;
                               if (n < p.N) finish(m, n, v);
                           });
    }
}

template <bool BF16, int NT, int STAGES>
struct Fp8DecodeLauncher {
    using C = Fp8DecodeCfg<STAGES, NT>;
    static constexpr auto kernel = wq_decode_fp8_kernel<BF16, NT, STAGES>;
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
        KernelConfig k{FMT_FP8, BF16 ? 1 : 0, 8 * C::NTA, C::BK, STAGES, 0, C::NTHREADS, C::SMEM_BYTES, 0, 1};
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
