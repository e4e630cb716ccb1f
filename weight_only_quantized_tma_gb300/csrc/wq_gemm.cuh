// wq_gemm.cuh -- the weight-only quantized GEMM kernel for sm_103a.
//
//   out[m, n] = alpha * sum_k A[m, k] * dequant(W)[n, k]   (+ bias[n] for FP8)
//
// Orientation: dequantized weight rows are the tcgen05 A operand (MMA M = 128
// weight rows per CTA tile), activation rows (tokens) are the B operand (MMA N =
// BN tokens).  A lives in tensor memory: the transform warpgroup writes it there
// with tcgen05.st, so the 16-bit weight copy never touches shared memory or HBM.
// ("FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis", §1: on sm_100a/sm_103a a
// dedicated transform warpgroup converts the weights into TMEM.)
//
// Warp roles (128 * (1 + NWG) threads):
//   warp 0      TMA producer of the activation tiles, one per k-block, through a
//               STAGES-deep mbarrier ring released by the MMA commits;
//   warp 3      TMA producer of the packed weight tiles and their scales, through
//               a second, WSTAGES-deep ring released by the transform warps as
//               soon as they hold the codes in registers;
//   warp 1      MMA issuer: tcgen05.mma kind::f16, accumulator in TMEM, commits
//               free the activation stage and the TMEM operand stage;
//   warp 2      TMEM allocator;
// The two rings are separate so that the transform of a k-block waits only for
// its weight bytes: the chain from an MMA completing to the next copy into its
// activation stage no longer runs through the weight transform.
//
// PAIR variant (a cluster of two CTAs on the two SMs of a pair, tcgen05
// cta_group::2): one output tile is 256 weight rows x BN tokens.  Each CTA
// dequantizes its own 128 weight rows into its own TMEM and copies only its half
// of the activation tile (BN / 2 tokens); the even CTA issues MMAs of M = 256 that
// read both halves, so every SM moves half the activation bytes per MMA.  The odd
// CTA's MMA warp forwards its activation-landed barrier to the even CTA, its
// transform warps arrive on the even CTA's operand-full barrier, and the even
// CTA's commits arrive on the barriers of both CTAs.  No copy is multicast.
//   warps 4..   transform: unpack / decode + scale into 16-bit operands, then the
//               epilogue (TMEM -> registers -> alpha/bias -> 16-bit -> global),
//               including the deterministic split-K reduction: through a workspace
//               (each slice writes fp32 partials, the last arriver of a warp's strip
//               sums them), or, when the slices of a tile are one thread-block
//               cluster (p.csplit), through the other slices' shared memory after
//               the main loop (all warps of the cluster meet at two cluster barriers).
//
// Dequantization per format (all exact until the final rounding to the operand
// type, see the conversion helpers below):
//   INT4  w = RN((q - 8) * s[k / G, n])           ("Low Bit Triton Kernels", §03)
//   LUT4  w = RN(LUT[q] * s[k / G, n])            (the same page: NF4's 16 non-uniform
//                                                  values as a lookup table)
//   INT2  w = RN((q - 2) * s[k / G, n])           ("Bitblas", hands-on item 6: W2A16)
//   FP8   w = e4m3(code)       (scale on the fp32 accumulator, PR #7495 intro)
//   FP4   w = e2m1(code) * e4m3(sf[n, k / 16])    (alpha on the accumulator, PR #4466 §2)
//
// Every barrier wait is bounded; on a timeout the kernel records a status bit,
// stops issuing work, waits (bounded) for its own copies and MMAs in flight,
// releases its tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {

template <int FMT, bool BF16, int BN, int BK, int STAGES, int NWG, bool PAIR = false, int WSTAGES = STAGES>
struct GemmCfg {
    static constexpr int NT = 128 * (1 + NWG);
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;                 // tokens this CTA copies per k-block
    static constexpr int B_STAGE = B_ROWS * BK * 2;                   // activation tile bytes
    static constexpr int W_STAGE = (FMT == FMT_FP8) ? TILE_N * BK : (FMT == FMT_INT2) ? TILE_N * BK / 4 : TILE_N * BK / 2;
    static constexpr int SC_STAGE = group_scaled(FMT) ? (BK / 32) * TILE_N * 2
                                  : (FMT == FMT_FP4)  ? TILE_N * BK / 16 : 0;
    static constexpr int TMEM_COLS = (BN <= 128) ? 256 : 512;
    static constexpr int A_BASE = (BN < 64) ? 64 : BN;                // first TMEM column of operand stages
    static constexpr int A_COLS = BK / 2;                             // 16-bit operand: 2 per column
    static constexpr int A_ST_RAW = (TMEM_COLS - A_BASE) / A_COLS;
    static constexpr int A_ST = A_ST_RAW > 4 ? 4 : A_ST_RAW;          // TMEM operand stages
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_B = 0;
    static constexpr int OFF_W = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SC = OFF_W + WSTAGES * W_STAGE;
    // pair: the epilogue stages the 16-bit output tile [token][weight row] here and
    // copies it out with TMA, so the accumulator is released before the stores
    static constexpr bool STAGE_OUT = PAIR;
    static constexpr int OUT_BOX_M = 128;                             // tokens per output copy
    // INT4 zero points of the stage's groups (uint8, up to BK / 32 groups of 128 rows)
    static constexpr int ZP_STAGE = (FMT == FMT_INT4) ? (BK / 32) * TILE_N : 0;
    static constexpr int OFF_ZP = OFF_SC + WSTAGES * SC_STAGE;
    static constexpr int OFF_STG = (OFF_ZP + WSTAGES * ZP_STAGE + 1023) / 1024 * 1024;
    static constexpr int STG_BYTES = STAGE_OUT ? BN * TILE_N * 2 : 0;
    static constexpr int OFF_BAR = (OFF_STG + STG_BYTES + 127) / 128 * 128;
    static constexpr int NBARS = 2 * STAGES + 2 * WSTAGES + 2 * A_ST + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;               // alignment slack
    // FP8 / FP4 weight tiles arrive through TMA with a row pitch of W_PITCH bytes
    // and the matching swizzle; the XOR mask applies to 16-byte chunk indices.
    static constexpr int W_PITCH = W_STAGE / TILE_N;
    static constexpr uint32_t W_SWZ = (W_PITCH == 128) ? 7u : (W_PITCH == 64) ? 3u : 1u;
    // Split-K inside a cluster: after the main loop the stage memory [0, OFF_STG) of
    // every CTA is an inbox for the fp32 partial rows the other slices send it,
    // [slice][row][BN + 4] (16-byte rows for vector stores and loads; a warp's 32
    // rows then fall on 8 bank quads, the minimum for 16-byte accesses); at most
    // S * ceil(128 / S) <= 143 rows for S <= 16.
    static constexpr int CS_PITCH = BN + 4;
    static constexpr int CS_INBOX = (TILE_N + 15) * CS_PITCH * 4;
    static constexpr bool CSPLIT_OK = !PAIR && CS_INBOX <= OFF_STG;
    // two CTAs per SM when shared and tensor memory allow it (decode, split-K)
    static constexpr int MIN_BLOCKS = (!PAIR && 2 * (SMEM_BYTES + 1024) <= 228 * 1024 && TMEM_COLS <= 256) ? 2 : 1;
    static_assert(BK == 64 || BK == 128, "BK");
    static_assert(FMT != FMT_INT2 || (BK == 128 && NWG == 2), "INT2 transform: two 32-code units per warpgroup");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "BN");
    static_assert(!PAIR || BN == 256, "pair tiles are 256 x 256");
    static_assert(A_ST >= 2, "need at least two TMEM operand stages");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(B_STAGE % 1024 == 0 && W_STAGE % 1024 == 0, "1024-byte stage alignment");
};

// ---------------------------------------------------------------- conversions

// INT4 operands of one weight row for 32 values of K, gathered from the
// fragment-order layout (wq_internal.h): four lanes' 8-byte halves (c = 0..3), two
// words each (k steps t = 0, 1 of the unit).  The row is the lower (h = 0) or the
// upper (h = 1) half of its 16-row group, so its codes sit at bits 0-3/16-19 and
// 8-11/24-27 of each word (h = 0) or at bits 4-7/20-23 and 12-15/28-31 (h = 1).
// The fp16 "magic number" trick turns a nibble into 1024 + q (bits 0-3, exponent
// 2^10) or 64 + q (bits 4-7, exponent 2^6 where the mantissa unit is 1/16);
// subtracting 1032 or 72 gives q - 8 exactly, and one multiply by the group scale
// rounds once: RN16((q - 8) * s).  Output o[8t + c] holds the pair
// (k = 16t + 2c, +1), o[8t + 4 + c] the pair (k = 16t + 8 + 2c, +1).
struct Int4RowConsts {
    uint32_t mask, magic, bias;   // per row half
};
__device__ __forceinline__ Int4RowConsts int4_row_consts(int h) {
    return h ? Int4RowConsts{0x00F000F0u, 0x54005400u, 0x54805480u}   // 64 + q, minus 72
             : Int4RowConsts{0x000F000Fu, 0x64006400u, 0x64086408u};  // 1024 + q, minus 1032
}

__device__ __forceinline__ void int4_row_to_f16(const uint2 (&w)[4], const Int4RowConsts& k, uint32_t s2,
                                                uint32_t (&o)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t wt[2] = {w[c].x, w[c].y};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t lo = ptx::lop3_and_or(wt[t], k.mask, k.magic);
            const uint32_t hi = ptx::lop3_and_or(wt[t] >> 8, k.mask, k.magic);
            o[8 * t + c] = ptx::hmul2_u32(ptx::hsub2_u32(lo, k.bias), s2);
            o[8 * t + 4 + c] = ptx::hmul2_u32(ptx::hsub2_u32(hi, k.bias), s2);
        }
    }
}

// Same gather for bf16 operands: q - 8 is exact in fp16, (q - 8) * s is exact in
// fp32 (4 + 11 significant bits), one rounding to bf16.
__device__ __forceinline__ void int4_row_to_bf16(const uint2 (&w)[4], const Int4RowConsts& k, float s,
                                                 uint32_t (&o)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t wt[2] = {w[c].x, w[c].y};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t lo = ptx::hsub2_u32(ptx::lop3_and_or(wt[t], k.mask, k.magic), k.bias);
            const uint32_t hi = ptx::hsub2_u32(ptx::lop3_and_or(wt[t] >> 8, k.mask, k.magic), k.bias);
            const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            o[8 * t + c] = ptx::f32x2_to_bf16x2(fl.x * s, fl.y * s);
            o[8 * t + 4 + c] = ptx::f32x2_to_bf16x2(fh.x * s, fh.y * s);
        }
    }
}

// A row's 32 values of one unit (the gather of int4_row_to_f16) through the
// codebook, times the group scale: RN16(LUT[q] * s) (the fp16 product of two fp16
// values is one rounding of the exact product).
__device__ __forceinline__ void lut16_row_to_f16(const uint2 (&w)[4], uint32_t hshift, const Lut16& t, uint32_t s2,
                                                 uint32_t (&o)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t wt[2] = {w[c].x, w[c].y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t lo, hi;
            lut16_word(wt[k], hshift, t, lo, hi);
            o[8 * k + c] = ptx::hmul2_u32(lo, s2);
            o[8 * k + 4 + c] = ptx::hmul2_u32(hi, s2);
        }
    }
}

// bf16 operands: LUT[q] * s is exact in fp32 (11 + 11 significant bits), one
// rounding to bf16.
__device__ __forceinline__ void lut16_row_to_bf16(const uint2 (&w)[4], uint32_t hshift, const Lut16& t, float s,
                                                  uint32_t (&o)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t wt[2] = {w[c].x, w[c].y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t lo, hi;
            lut16_word(wt[k], hshift, t, lo, hi);
            const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            o[8 * k + c] = ptx::f32x2_to_bf16x2(fl.x * s, fl.y * s);
            o[8 * k + 4 + c] = ptx::f32x2_to_bf16x2(fh.x * s, fh.y * s);
        }
    }
}

// INT2 (W2A16): 32 codes of a row, two canonical words (code k at bits 2 (k % 16)
// of word k / 16) -> 16 pairs (k = 2p, 2p + 1) in o[p].  Per word, the even and the
// odd codes are separated into the low and the high halves (AND, shift-AND, two byte
// permutes), so that code pair p sits at bits 4p' / 16 + 4p' of a word; the fp16
// "magic number" for that position (exponent 2^10, 2^6, 2^2: mantissa unit 1, 1/16,
// 1/256 shifted by 0, 4, 8 bits) turns it into b + q with one AND-OR, and the fourth
// pair of each half is shifted down first.  Subtracting b + 2 gives q - 2 exactly;
// one multiply by the group scale rounds once: RN16((q - 2) * s).
__device__ __forceinline__ void int2_word_to_pairs(uint32_t w, uint32_t (&h)[8]) {
    const uint32_t ev = w & 0x33333333u;            // codes 2p at bits 4p
    const uint32_t od = (w >> 2) & 0x33333333u;     // codes 2p + 1 at bits 4p
    const uint32_t x = ptx::prmt(ev, od, 0x5410u);  // pairs 0-3: even in the low half, odd in the high
    const uint32_t y = ptx::prmt(ev, od, 0x7632u);  // pairs 4-7
    const uint32_t src[2] = {x, y};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t v = src[j];
        h[4 * j + 0] = ptx::hsub2_u32(ptx::lop3_and_or(v, 0x00030003u, 0x64006400u), 0x64026402u);   // 1024 + q
        h[4 * j + 1] = ptx::hsub2_u32(ptx::lop3_and_or(v, 0x00300030u, 0x54005400u), 0x54205420u);   // 64 + q
        h[4 * j + 2] = ptx::hsub2_u32(ptx::lop3_and_or(v, 0x03000300u, 0x44004400u), 0x46004600u);   // 4 + q
        h[4 * j + 3] = ptx::hsub2_u32(ptx::lop3_and_or(v >> 12, 0x00030003u, 0x64006400u), 0x64026402u);
    }
}

__device__ __forceinline__ void int2_row_to_f16(const uint2& w, uint32_t s2, uint32_t (&o)[16]) {
    uint32_t h[8];
    int2_word_to_pairs(w.x, h);
#pragma unroll
    for (int p = 0; p < 8; ++p) o[p] = ptx::hmul2_u32(h[p], s2);
    int2_word_to_pairs(w.y, h);
#pragma unroll
    for (int p = 0; p < 8; ++p) o[8 + p] = ptx::hmul2_u32(h[p], s2);
}

// bf16 operands: (q - 2) * s is exact in fp32, one rounding to bf16.
__device__ __forceinline__ void int2_row_to_bf16(const uint2& w, float s, uint32_t (&o)[16]) {
    const uint32_t wv[2] = {w.x, w.y};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint32_t h[8];
        int2_word_to_pairs(wv[j], h);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[p]));
            o[8 * j + p] = ptx::f32x2_to_bf16x2(f.x * s, f.y * s);
        }
    }
}

// FP8: 16 e4m3 codes (one 16-byte chunk, k ascending) -> 8 operand words.
template <bool BF16>
__device__ __forceinline__ void fp8_to_operand(const uint4& q, uint32_t (&o)[8]) {
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t lo = ptx::e4m3x2_to_f16x2((uint16_t)(wv[j] & 0xFFFFu));
        uint32_t hi = ptx::e4m3x2_to_f16x2((uint16_t)(wv[j] >> 16));
        if (BF16) {
            lo = ptx::f16x2_to_bf16x2_exact(lo);
            hi = ptx::f16x2_to_bf16x2_exact(hi);
        }
        o[2 * j] = lo;
        o[2 * j + 1] = hi;
    }
}

// FP4: 32 e2m1 codes (one 16-byte chunk, byte b holds k = 2b (low nibble) and
// 2b + 1) times the two e4m3 block scales of the chunk -> 16 bf16x2 words.
// e2m1 * e4m3 has at most 5 significant bits and stays inside the normal fp16
// range, so the f16 product and its bf16 copy are exact.
__device__ __forceinline__ void fp4_to_bf16(const uint4& q, uint16_t sf_pair, uint32_t (&o)[16]) {
    const uint32_t sf2 = ptx::e4m3x2_to_f16x2(sf_pair);
    const uint32_t s_lo = __byte_perm(sf2, 0, 0x1010);   // {sf0, sf0}
    const uint32_t s_hi = __byte_perm(sf2, 0, 0x3232);   // {sf1, sf1}
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t h[4];
        ptx::e2m1x8_to_f16x2x4(wv[j], h);
        const uint32_t s2 = (j < 2) ? s_lo : s_hi;
#pragma unroll
        for (int i = 0; i < 4; ++i) o[4 * j + i] = ptx::f16x2_to_bf16x2_exact(ptx::hmul2_u32(h[i], s2));
    }
}

template <int FMT, bool BF16, int BN, int BK, int STAGES, int NWG, bool PAIR, int WSTAGES>
__global__ void __launch_bounds__(128 * (1 + NWG), (GemmCfg<FMT, BF16, BN, BK, STAGES, NWG, PAIR, WSTAGES>::MIN_BLOCKS))
    wq_gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = GemmCfg<FMT, BF16, BN, BK, STAGES, NWG, PAIR, WSTAGES>;
    constexpr int CG = PAIR ? 2 : 1;   // tcgen05 CTA group of every tcgen05 instruction here
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };                 // activation stage landed
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };     // activation stage free
    auto wfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };            // weight stage landed
    auto wempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + WSTAGES + s); }; // weight stage free
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 * WSTAGES + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 * WSTAGES + C::A_ST + a); };
    const uint32_t accfull_bar = bar0 + 8u * (2 * STAGES + 2 * WSTAGES + 2 * C::A_ST);
    const uint32_t accempty_bar = accfull_bar + 8u;
    const uint32_t final_bar = accfull_bar + 16u;
    const uint32_t epi_bar = accfull_bar + 24u;   // staged epilogue: sync of the transform warps
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* tmem_slot = misc + 0;
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_epi = 128 * NWG;
    // pair: rank 0 issues the MMAs; barriers it waits on count the other CTA too
    const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
    const bool issuer = (rank == 0);
    const int ctas = PAIR ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // pair, rank 0: its own copies plus the forwarded arrival of rank 1's
            ptx::mbar_init(full_bar(s), (PAIR && issuer) ? 2 : 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < WSTAGES; ++s) {
            ptx::mbar_init(wfull_bar(s), 1);
            ptx::mbar_init(wempty_bar(s), n_epi / 32);
        }
        // weight-empty, operand-full and accumulator-empty take one arrival per
        // transform warp (of both CTAs of a pair)
        for (int a = 0; a < C::A_ST; ++a) {
            ptx::mbar_init(afull_bar(a), ctas * n_epi / 32);
            ptx::mbar_init(aempty_bar(a), 1);
        }
        ptx::mbar_init(accfull_bar, 1);
        ptx::mbar_init(accempty_bar, ctas * n_epi / 32);
        ptx::mbar_init(final_bar, 1);
        ptx::mbar_init(epi_bar, n_epi / 32);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&p.tmap_a);
        if (!int4_layout(FMT)) ptx::prefetch_tmap(&p.tmap_w);
    }
    if (warp == 2) {
        ptx::tmem_alloc<CG>(sbase + C::OFF_MISC, C::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // pair: both CTAs' barriers are initialised before either CTA signals the other
    if (PAIR) ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a barrier of the issuing CTA / of the other CTA, as a shared::cluster address
    auto at_issuer = [&](uint32_t bar) { return PAIR ? ptx::mapa_shared(bar, 0) : bar; };
    auto at_other = [&](uint32_t bar) { return ptx::mapa_shared(bar, (uint32_t)(rank ^ 1)); };
    // this CTA's 128-row weight tile of an item (pair: two per item)
    auto w_tile = [&](const Item& it) { return PAIR ? 2 * it.n_tile + rank : it.n_tile; };
    const int tiles_w = (p.N + TILE_N - 1) / TILE_N;
    // persistent walk: a pair takes items as one
    const int item0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int istride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    // The next kernel on the stream may start its own set-up now (programmatic
    // dependent launch); it waits for this grid before touching shared data.
    if (threadIdx.x == 0) ptx::grid_launch_dependents();

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------------------ producers
        // warp 0: activation tiles (freed by the MMA commits); warp 3: weight
        // tiles and scales (freed by the transform warps)
        if (lane == 0) {
            const bool act = (warp == 0);
            const int NS = act ? STAGES : WSTAGES;   // depth of this producer's ring
            const uint64_t pol = act ? ptx::policy_evict_last()
                                     : (p.w_evict_first ? ptx::policy_evict_first() : ptx::policy_evict_last());
            int s = 0;
            uint32_t ph = 0;
            long long issued = 0;
            bool ok = true;
            // every global input may have been written by the previous kernel on the
            // stream: wait for it (programmatic dependent launch) before the first copy
            ptx::grid_dependency_wait();
            for (int item = item0; item < p.n_items && ok; item += istride) {
                const Item it = decode_item(p, item);
                for (int kb = it.kb_begin; kb < it.kb_end; ++kb) {
                    if (!bounded_wait(act ? empty_bar(s) : wempty_bar(s), ph ^ 1u, abort_flag, p.status,
                                            DEVICE_TIMEOUT_PRODUCER, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (act) {
                        // activation rows >= M are not loaded: they only feed accumulator
                        // columns that are never stored, and out-of-range rows would cost
                        // the copy engine a zero fill
                        // a half tile copies only its own rows (a box half as high)
                        const uint32_t fb = full_bar(s);
                        const void* tmap = it.half ? &p.tmap_a_half : &p.tmap_a;
                        const int rows = it.half ? p.a_box_rows_half : p.a_box_rows;
                        ptx::mbar_arrive_expect_tx(fb, (uint32_t)((BK / 64) * rows * 128));
                        const uint32_t b_dst = sbase + C::OFF_B + s * C::B_STAGE;
                        // pair: this CTA's half of the tokens (of a half tile: its quarter)
                        const int row0 = it.m_tile * BN + it.m_sub +
                                         (PAIR ? rank * (it.half ? BN / 4 : C::B_ROWS) : 0);
#pragma unroll
                        for (int j = 0; j < BK / 64; ++j)
                            ptx::tma_load_2d(b_dst + j * (C::B_ROWS * 128), tmap, kb * BK + j * 64, row0, fb, pol);
                    } else if (PAIR && w_tile(it) >= tiles_w) {
                        // the odd CTA of a pair past the last weight tile (N / 128 odd):
                        // nothing to copy; its operand rows only reach output rows >= N
                        ptx::mbar_arrive(wfull_bar(s));
                    } else {
                        const uint32_t fb = wfull_bar(s);
                        const uint32_t w_dst = sbase + C::OFF_W + s * C::W_STAGE;
                        const uint32_t sc_dst = sbase + C::OFF_SC + s * C::SC_STAGE;
                        if (int4_layout(FMT)) {
                            const int gcnt = (p.G >= BK) ? 1 : (BK >> p.g_shift);
                            const uint32_t sc_bytes = (uint32_t)gcnt * TILE_N * 2;
                            const uint32_t zp_bytes = (FMT == FMT_INT4 && p.zp) ? (uint32_t)gcnt * TILE_N : 0u;
                            ptx::mbar_arrive_expect_tx(fb, C::W_STAGE + sc_bytes + zp_bytes);
                            const uint8_t* wsrc =
                                p.w + ((size_t)w_tile(it) * p.nchunks_pad + (size_t)kb * (BK / 32)) * (TILE_N * 16);
                            ptx::bulk_load(w_dst, wsrc, C::W_STAGE, fb, pol);
                            const int g0 = (kb * BK) >> p.g_shift;
                            const uint8_t* ssrc = p.sc + ((size_t)w_tile(it) * p.ngroups_pad + g0) * (TILE_N * 2);
                            ptx::bulk_load(sc_dst, ssrc, sc_bytes, fb, pol);
                            if (FMT == FMT_INT4 && p.zp)
                                ptx::bulk_load(sbase + C::OFF_ZP + s * C::ZP_STAGE,
                                               p.zp + ((size_t)w_tile(it) * p.ngroups_pad + g0) * TILE_N, zp_bytes, fb,
                                               pol);
                        } else if (FMT == FMT_INT2) {
                            // canonical 2-bit rows through TMA (BK / 4 bytes per row), group
                            // scales as for INT4
                            const int gcnt = (p.G >= BK) ? 1 : (BK >> p.g_shift);
                            const uint32_t sc_bytes = (uint32_t)gcnt * TILE_N * 2;
                            ptx::mbar_arrive_expect_tx(fb, C::W_STAGE + sc_bytes);
                            ptx::tma_load_2d(w_dst, &p.tmap_w, kb * (BK / 4), w_tile(it) * TILE_N, fb, pol);
                            const int g0 = (kb * BK) >> p.g_shift;
                            const uint8_t* ssrc = p.sc + ((size_t)w_tile(it) * p.ngroups_pad + g0) * (TILE_N * 2);
                            ptx::bulk_load(sc_dst, ssrc, sc_bytes, fb, pol);
                        } else if (FMT == FMT_FP4) {
                            ptx::mbar_arrive_expect_tx(fb, C::W_STAGE + C::SC_STAGE);
                            ptx::tma_load_2d(w_dst, &p.tmap_w, kb * (BK / 2), w_tile(it) * TILE_N, fb, pol);
                            const uint8_t* ssrc =
                                p.sc + ((size_t)w_tile(it) * p.nchunks_pad + (size_t)kb * (BK / 64)) * (TILE_N * 4);
                            ptx::bulk_load(sc_dst, ssrc, C::SC_STAGE, fb, pol);
                        } else {
                            ptx::mbar_arrive_expect_tx(fb, C::W_STAGE);
                            ptx::tma_load_2d(w_dst, &p.tmap_w, kb * BK, w_tile(it) * TILE_N, fb, pol);
                        }
                    }
                    ++issued;
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (ok && act) {
                // tail: every stage released, i.e. every MMA commit aimed at this
                // CTA's activation ring has landed before the CTA can exit
                for (int j = 0; j < STAGES && ok; ++j) {
                    ok = bounded_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_PRODUCER,
                                            p.timeout_ns);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // wait for this thread's own copies in flight before the CTA can exit
                const long long first = issued > NS ? issued - NS : 0;
                for (long long j = first; j < issued; ++j) {
                    const int sj = (int)(j % NS);
                    if (!drain_wait(act ? full_bar(sj) : wfull_bar(sj), (uint32_t)((j / NS) & 1), p.timeout_ns))
                        atomicOr(p.status, DEVICE_TIMEOUT_DRAIN);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1 && PAIR && !issuer) {
        // ------------------------------------------------------------ pair, odd CTA: forwarder
        // The even CTA's MMAs read this CTA's activation half: pass each stage's
        // landing on to the even CTA's full barrier.
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int item = item0; item < p.n_items && ok; item += istride) {
                const Item it = decode_item(p, item);
                for (int kb = it.kb_begin; kb < it.kb_end; ++kb) {
                    if (!bounded_wait(full_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_MMA, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_cluster(at_issuer(full_bar(s)));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_full = ptx::make_idesc_f16(BF16, PAIR ? 256 : 128, BN);
            constexpr uint32_t idesc_half = ptx::make_idesc_f16(BF16, PAIR ? 256 : 128, BN >= 32 ? BN / 2 : BN);
            // every commit arrives on this CTA's barrier and, in a pair, on the other's
            auto commit = [&](uint32_t bar) {
                ptx::mma_commit<CG>(bar);
                if (PAIR) ptx::mma_commit<CG>(at_other(bar));
            };
            // The issuing thread runs at most about one MMA ahead of the tensor pipe,
            // so every instruction between two MMAs is pipe time unless it overlaps an
            // MMA in flight.  Hence: the next k-block's barriers are probed (without
            // blocking) before its last MMA is issued, and a k-block's commits go out
            // after the next k-block's first MMA (they then also cover that MMA, which
            // frees the stages one MMA later).
            const uint32_t empty0_o = PAIR ? at_other(empty_bar(0)) : 0u;   // barriers are contiguous
            const uint32_t aempty0_o = PAIR ? at_other(aempty_bar(0)) : 0u;
            auto commit_stage = [&](int cs, int ca) {
                ptx::mma_commit<CG>(empty_bar(cs));
                ptx::mma_commit<CG>(aempty_bar(ca));
                if (PAIR) {
                    ptx::mma_commit<CG>(empty0_o + 8u * cs);
                    ptx::mma_commit<CG>(aempty0_o + 8u * ca);
                }
            };
            int s = 0, a = 0;
            uint32_t ph = 0, aph = 0, accph = 0;
            bool ok = true;
            for (int item = item0; item < p.n_items && ok; item += istride) {
                const Item it = decode_item(p, item);
                if (!bounded_wait(accempty_bar, accph ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_MMA,
                                  p.timeout_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t idesc = it.half ? idesc_half : idesc_full;   // half tile: MMA N = BN / 2
                int pend_s = -1, pend_a = 0;   // commits owed for the previous k-block
                bool ready = false;            // this k-block's operands already seen landed
                for (int kb = it.kb_begin; kb < it.kb_end; ++kb) {
                    if (!ready && (!bounded_wait(afull_bar(a), aph, abort_flag, p.status, DEVICE_TIMEOUT_MMA,
                                                 p.timeout_ns) ||
                                   !bounded_wait(full_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_MMA,
                                                 p.timeout_ns))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t b_base = sbase + C::OFF_B + s * C::B_STAGE;
                    const uint32_t a_tmem = tmem + C::A_BASE + a * C::A_COLS;
                    const int s_n = (s + 1 == STAGES) ? 0 : s + 1;
                    const uint32_t ph_n = (s + 1 == STAGES) ? (ph ^ 1u) : ph;
                    const int a_n = (a + 1 == C::A_ST) ? 0 : a + 1;
                    const uint32_t aph_n = (a + 1 == C::A_ST) ? (aph ^ 1u) : aph;
                    ready = false;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t b_addr = b_base + (kk / 4) * (C::B_ROWS * 128) + (kk % 4) * 32;
                        ptx::mma_f16_ts<CG>(tmem, a_tmem + kk * 8, ptx::make_sdesc_sw128(b_addr), idesc,
                                            (kb > it.kb_begin || kk > 0) ? 1u : 0u);
                        if (kk == 0 && pend_s >= 0) commit_stage(pend_s, pend_a);
                        if (kk == BK / 16 - 2 && kb + 1 < it.kb_end)
                            ready = ptx::mbar_test_wait(afull_bar(a_n), aph_n) && ptx::mbar_test_wait(full_bar(s_n), ph_n);
                    }
                    pend_s = s;
                    pend_a = a;
                    s = s_n;
                    ph = ph_n;
                    a = a_n;
                    aph = aph_n;
                }
                if (!ok) break;
                if (pend_s >= 0) commit_stage(pend_s, pend_a);
                commit(accfull_bar);
                accph ^= 1u;
            }
            // pair: the last epilogue of both CTAs has arrived here before the CTA exits
            if (PAIR && ok && !*abort_flag)
                bounded_wait(accempty_bar, accph ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_MMA, p.timeout_ns);
            if (*abort_flag) {
                ptx::mma_commit<CG>(final_bar);
                if (!drain_wait(final_bar, 0, p.timeout_ns)) atomicOr(p.status, DEVICE_TIMEOUT_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ transform + epilogue
        const int ew = warp - 4;            // 0 .. 4*NWG-1
        const int wg = ew >> 2;             // transform warpgroup
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;  // weight row inside the tile == TMEM lane
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        int s = 0, a = 0;
        uint32_t ph = 0, aph = 0, accph = 0, eph = 0;
        bool ok = true;
        // all transform warps meet here (bounded, so an aborting warp cannot strand
        // the others the way a hardware barrier would)
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(epi_bar);
            const bool w = __all_sync(0xffffffffu, bounded_wait(epi_bar, eph, abort_flag, p.status,
                                                                DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns));
            eph ^= 1u;
            return w;
        };
        ptx::grid_dependency_wait();   // alpha / bias are global inputs too
        const float alpha = group_scaled(FMT) ? 1.0f : __ldg(p.alpha);
        // One k-block of the transform: waits for its codes and a free TMEM operand
        // stage, writes the 16-bit operand there and hands it to the MMA issuer.
        auto transform_one = [&]() -> bool {
            bool w1 = bounded_wait(wfull_bar(s), ph, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM, p.timeout_ns);
            bool w2 = w1 && bounded_wait(aempty_bar(a), aph ^ 1u, abort_flag, p.status,
                                               DEVICE_TIMEOUT_TRANSFORM, p.timeout_ns);
            if (!__all_sync(0xffffffffu, w2)) {
                return false;
            }
            ptx::tc_fence_after();
            const uint8_t* wt = smem + C::OFF_W + s * C::W_STAGE;
            const uint8_t* sct = smem + C::OFF_SC + s * C::SC_STAGE;
            const uint32_t a_col = tmem + lane_addr + C::A_BASE + a * C::A_COLS;
            if (FMT == FMT_FP8) {
                constexpr int CH = BK / 16;  // 16-byte chunks (16 codes, 8 columns) per row
#pragma unroll
                for (int c = wg * (CH / NWG); c < (wg + 1) * (CH / NWG); ++c) {
                    const uint4 q = *reinterpret_cast<const uint4*>(wt + swz(r * C::W_PITCH + c * 16, C::W_SWZ));
                    uint32_t o[8];
                    fp8_to_operand<BF16>(q, o);
                    ptx::tmem_st8(a_col + c * 8, o);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(wempty_bar(s));   // codes consumed
            } else {
                constexpr int CH = BK / 32;  // 16-byte chunks (32 codes, 16 columns) per row
                constexpr int CPW = CH / NWG;  // chunks per transform warpgroup
                const int c0 = wg * CPW;
                // all shared-memory loads first, then the conversions, then the TMEM
                // stores, so the units overlap instead of running back to back
                uint2 qi[CPW][4];     // INT4: four lanes' halves per 32-k unit
                uint4 q[CPW];         // FP4: one 16-byte chunk per 32-k unit
                uint16_t sv[CPW];
                const int gr = r >> 4, g8 = r & 7;
#pragma unroll
                for (int i = 0; i < CPW; ++i) {
                    const int c = c0 + i;
                    if (int4_layout(FMT) && CPW % 2 == 0) {
                        // units c, c + 1 (c even) are the two 8-byte halves of the same
                        // 16-byte slots of quad c / 2: one 16-byte load per slot serves both
                        if (i % 2 == 0) {
                            const uint8_t* ub = wt + (c >> 1) * 4096 + gr * 512;
#pragma unroll
                            for (int l = 0; l < 4; ++l) {
                                const uint4 v = *reinterpret_cast<const uint4*>(ub + int4_slot(4 * g8 + l) * 16);
                                qi[i][l] = make_uint2(v.x, v.y);
                                qi[i + 1][l] = make_uint2(v.z, v.w);
                            }
                            sv[i] = *reinterpret_cast<const uint16_t*>(sct + (((c * 32) >> p.g_shift) * TILE_N + r) * 2);
                            sv[i + 1] = (p.g_shift >= 6) ? sv[i]   // both units in one group (G >= 64)
                                      : *reinterpret_cast<const uint16_t*>(sct + ((((c + 1) * 32) >> p.g_shift) * TILE_N + r) * 2);
                        }
                    } else if (int4_layout(FMT)) {
                        // unit c: quad c / 2 of the stage, k steps 2 (c % 2) and 2 (c % 2) + 1
                        const uint8_t* ub = wt + (c >> 1) * 4096 + gr * 512 + (c & 1) * 8;
#pragma unroll
                        for (int l = 0; l < 4; ++l)
                            qi[i][l] = *reinterpret_cast<const uint2*>(ub + int4_slot(4 * g8 + l) * 16);
                        sv[i] = *reinterpret_cast<const uint16_t*>(sct + (((c * 32) >> p.g_shift) * TILE_N + r) * 2);
                    } else if (FMT == FMT_INT2) {
                        // unit c: bytes 8c .. 8c + 7 of the row (32 codes); units c, c + 1
                        // (c even) share one 16-byte chunk
                        if (i % 2 == 0) {
                            const uint4 v = *reinterpret_cast<const uint4*>(wt + swz(r * C::W_PITCH + (c >> 1) * 16, C::W_SWZ));
                            qi[i][0] = make_uint2(v.x, v.y);
                            qi[i + 1][0] = make_uint2(v.z, v.w);
                            sv[i] = *reinterpret_cast<const uint16_t*>(sct + (((c * 32) >> p.g_shift) * TILE_N + r) * 2);
                            sv[i + 1] = (p.g_shift >= 6) ? sv[i]
                                      : *reinterpret_cast<const uint16_t*>(sct + ((((c + 1) * 32) >> p.g_shift) * TILE_N + r) * 2);
                        }
                    } else {
                        q[i] = *reinterpret_cast<const uint4*>(wt + swz(r * C::W_PITCH + c * 16, C::W_SWZ));
                        sv[i] = *reinterpret_cast<const uint16_t*>(sct + (c >> 1) * (TILE_N * 4) + r * 4 + (c & 1) * 2);
                    }
                }
                uint32_t o[CPW][16];
                if (FMT == FMT_LUT4) {
                    // codebook: LUT[q] * s
                    const Lut16 tab = lut16_load(p.lut);
                    const uint32_t hshift = (uint32_t)((r >> 3) & 1) * 4u;
#pragma unroll
                    for (int i = 0; i < CPW; ++i) {
                        if (BF16)
                            lut16_row_to_bf16(qi[i], hshift, tab, __half2float(__ushort_as_half(sv[i])), o[i]);
                        else
                            lut16_row_to_f16(qi[i], hshift, tab, (uint32_t)sv[i] | ((uint32_t)sv[i] << 16), o[i]);
                    }
                } else if (FMT == FMT_INT2) {
#pragma unroll
                    for (int i = 0; i < CPW; ++i) {
                        if (BF16)
                            int2_row_to_bf16(qi[i][0], __half2float(__ushort_as_half(sv[i])), o[i]);
                        else
                            int2_row_to_f16(qi[i][0], (uint32_t)sv[i] | ((uint32_t)sv[i] << 16), o[i]);
                    }
                } else {
#pragma unroll
                for (int i = 0; i < CPW; ++i) {
                    if (FMT == FMT_INT4) {
                        Int4RowConsts kc = int4_row_consts((r >> 3) & 1);
                        if (p.zp) {
                            // zero point z of this unit's group and row: subtract b + z (b = 1024
                            // or 64 by row half) instead of b + 8, exactly as above
                            const uint8_t* zst = smem + C::OFF_ZP + s * C::ZP_STAGE;
                            const uint32_t z = zst[(((c0 + i) * 32) >> p.g_shift) * TILE_N + r];
                            const uint32_t b = ((r >> 3) & 1) ? (0x5400u + (z << 4)) : (0x6400u + z);
                            kc.bias = b | (b << 16);
                        }
                        if (BF16)
                            int4_row_to_bf16(qi[i], kc, __half2float(__ushort_as_half(sv[i])), o[i]);
                        else
                            int4_row_to_f16(qi[i], kc, (uint32_t)sv[i] | ((uint32_t)sv[i] << 16), o[i]);
                    } else {
                        fp4_to_bf16(q[i], sv[i], o[i]);
                    }
                }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(wempty_bar(s));   // codes consumed
#pragma unroll
                for (int i = 0; i < CPW; ++i) ptx::tmem_st16(a_col + (c0 + i) * 16, o[i]);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !issuer)
                    ptx::mbar_arrive_cluster(at_issuer(afull_bar(a)));
                else
                    ptx::mbar_arrive(afull_bar(a));
            }
            if (++s == WSTAGES) {
                s = 0;
                ph ^= 1u;
            }
            if (++a == C::A_ST) {
                a = 0;
                aph ^= 1u;
            }
            return true;
        };
        // Epilogue of one item: accumulator -> output (or split-K partial), then the
        // accumulator is handed back to the MMA issuer.
        auto epilogue = [&](const Item& it) -> bool {
            const bool wacc = bounded_wait(accfull_bar, accph, abort_flag, p.status, DEVICE_TIMEOUT_EPILOGUE,
                                                 p.timeout_ns);
            if (!__all_sync(0xffffffffu, wacc)) {
                return false;
            }
            accph ^= 1u;
            ptx::tc_fence_after();
            ptx::grid_dependency_wait();   // outputs and workspace may still be in use by the previous kernel
            const int n = w_tile(it) * TILE_N + r;
            const int m0 = it.m_tile * BN + it.m_sub;   // pair: accumulator column j is token m0 + j
            // accumulator columns per warpgroup (a half tile has BN / 2 of them)
            const int COLS = (it.half ? BN / 2 : BN) / NWG;
            constexpr int STEP = BN / NWG / 2 >= 16 ? 16 : 8;
            const int c_begin = wg * COLS;
            const uint32_t acc_addr = tmem + lane_addr;
            const int tile = it.n_tile + p.tiles_n * it.m_tile;
            const bool nvalid = n < p.N;
            float bias_v = 0.0f;
            if (FMT == FMT_FP8 && p.bias != nullptr && nvalid) bias_v = load_16bit<BF16>(p.bias, (size_t)n);

            if (C::STAGE_OUT) {
                // accumulator -> 16-bit -> staging [token][weight row]; the accumulator is
                // handed back as soon as it is read, then one thread copies the staged
                // tile out with TMA while the next item runs (rows >= M and columns >= N
                // are not written by the copy)
                if (warp == 4 && lane == 0) ptx::bulk_wait_group_read0();   // previous copy-out read it
                if (!epi_sync()) return false;
                uint16_t* stg = reinterpret_cast<uint16_t*>(smem + C::OFF_STG);
#pragma unroll 1
                for (int cc = c_begin; cc < c_begin + COLS; cc += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld16(acc_addr + cc, *reinterpret_cast<uint32_t(*)[16]>(v));
                    ptx::tmem_ld16(acc_addr + cc + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        stg[(cc + j) * TILE_N + r] = to_16bit<BF16>(alpha * __uint_as_float(v[j]) + bias_v);
                }
                ptx::tc_fence_before();
                ptx::fence_proxy_async_smem();   // staging writes visible to the copy engine
                __syncwarp();
                if (lane == 0) {
                    if (PAIR && !issuer)
                        ptx::mbar_arrive_cluster(at_issuer(accempty_bar));
                    else
                        ptx::mbar_arrive(accempty_bar);
                }
                if (!epi_sync()) return false;   // the whole tile is staged
                if (warp == 4 && lane == 0 && w_tile(it) * TILE_N < p.N) {
                    const int rows = it.half ? BN / 2 : BN;
                    for (int h = 0; h < rows && m0 + h < p.M; h += C::OUT_BOX_M)
                        ptx::tma_store_2d(&p.tmap_out, ptx::smem_u32(stg) + h * TILE_N * 2, w_tile(it) * TILE_N,
                                          m0 + h);
                    ptx::bulk_commit_group();
                }
                return true;
            }
            if (p.splits == 1) {
                // CH accumulator columns per wait on tensor memory: the loads of a
                // chunk are issued back to back, so the epilogue pays the TMEM
                // latency once per chunk instead of once per 16 columns
                constexpr int CH = (BN / NWG / 2 >= 64) ? 64 : (BN / NWG / 2 >= 8 ? BN / NWG / 2 : 8);
#pragma unroll 1
                for (int cc = c_begin; cc < c_begin + COLS; cc += CH) {
                    uint32_t v[CH];
                    if (CH >= 16) {
#pragma unroll
                        for (int q = 0; q < CH / 16; ++q)
                            ptx::tmem_ld16(acc_addr + cc + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * q));
                    } else {
                        ptx::tmem_ld8(acc_addr + cc, *reinterpret_cast<uint32_t(*)[8]>(v));
                    }
                    ptx::tmem_wait_ld();
                    if (nvalid) {
#pragma unroll
                        for (int j = 0; j < CH; ++j) {
                            const int m = m0 + cc + j;
                            if (m < p.M)
                                store_out<BF16>(p.out, (size_t)m * p.N + n, alpha * __uint_as_float(v[j]) + bias_v);
                        }
                    }
                }
            } else {
                // deterministic split-K: every slice writes its fp32 partial, the last
                // slice to arrive sums all slices in slice order 0..S-1 and stores.
                float* part = p.ws_part + (size_t)(tile * p.splits + it.slice) * BN * TILE_N;
#pragma unroll 1
                for (int cc = c_begin; cc < c_begin + COLS; cc += STEP) {
                    uint32_t v[16];
                    if (STEP == 16) {
                        ptx::tmem_ld16(acc_addr + cc, v);
                    } else {
                        uint32_t v8[8];
                        ptx::tmem_ld8(acc_addr + cc, v8);
#pragma unroll
                        for (int j = 0; j < 8; ++j) v[j] = v8[j];
                    }
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < STEP; ++j) {
                        if (m0 + cc + j < p.M) __stcg(part + (size_t)(cc + j) * TILE_N + r, __uint_as_float(v[j]));
                    }
                }
                // Each epilogue warp owns 32 rows x COLS columns of the tile and takes
                // its own ticket, so no warp ever waits for another one.
                __threadfence();
                __syncwarp();
                uint32_t last = 0;
                if (lane == 0) {
                    uint32_t* cnt = p.ws_count + (size_t)tile * 8 + ew;
                    const uint32_t old = atomicAdd(cnt, 1u);
                    last = (old == (uint32_t)(p.splits - 1)) ? 1u : 0u;
                    if (last) atomicExch(cnt, 0u);
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    const float* base = p.ws_part + (size_t)(tile * p.splits) * BN * TILE_N;
                    // CB columns at a time, two slices per round: 2 CB independent loads
                    // in flight per thread (one L2 round trip per round instead of one
                    // per column), each column summed in slice order 0..S-1
                    constexpr int CB = 8;
                    const int ncols = min(COLS, p.M - (m0 + c_begin));
#pragma unroll 1
                    for (int c0 = 0; c0 < ncols; c0 += CB) {
                        float acc[CB];
#pragma unroll
                        for (int j = 0; j < CB; ++j) acc[j] = 0.0f;
#pragma unroll 1
                        for (int sl = 0; sl < p.splits; sl += 2) {
                            const bool two = sl + 1 < p.splits;
                            float v0[CB], v1[CB];
#pragma unroll
                            for (int j = 0; j < CB; ++j) {
                                const bool in = c0 + j < ncols;
                                const size_t col = (size_t)(c_begin + c0 + j);
                                v0[j] = in ? __ldcg(base + ((size_t)sl * BN + col) * TILE_N + r) : 0.0f;
                                v1[j] = (in && two) ? __ldcg(base + ((size_t)(sl + 1) * BN + col) * TILE_N + r) : 0.0f;
                            }
#pragma unroll
                            for (int j = 0; j < CB; ++j) {
                                acc[j] += v0[j];
                                if (two) acc[j] += v1[j];
                            }
                        }
                        if (nvalid) {
#pragma unroll
                            for (int j = 0; j < CB; ++j)
                                if (c0 + j < ncols)
                                    store_out<BF16>(p.out, (size_t)(m0 + c_begin + c0 + j) * p.N + n,
                                                    alpha * acc[j] + bias_v);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !issuer)
                    ptx::mbar_arrive_cluster(at_issuer(accempty_bar));
                else
                    ptx::mbar_arrive(accempty_bar);
            }
            return true;
        };
        // The epilogue of an item runs after the transform of the first A_ST k-blocks
        // of the next one: those fill the operand stages while the item's last MMAs
        // run, so the MMA issuer starts the next item as soon as the accumulator is
        // free instead of waiting for the epilogue and then for a transform.
        Item pend{};
        bool has_pend = false;
        for (int item = item0; item < p.n_items && ok; item += istride) {
            const Item it = decode_item(p, item);
            int done = 0;
            for (int kb = it.kb_begin; kb < it.kb_end && ok; ++kb) {
                ok = transform_one();
                if (ok && has_pend && ++done == C::A_ST) {
                    ok = epilogue(pend);
                    has_pend = false;
                }
            }
            if (ok && has_pend) {
                ok = epilogue(pend);
                has_pend = false;
            }
            pend = it;
            has_pend = true;
        }
        if (ok && has_pend) {
            if (!PAIR && p.csplit) {
                // split-K inside a cluster: the accumulator is read after the cluster
                // barrier below, once every slice of the tile has finished its main loop
                ok = __all_sync(0xffffffffu, bounded_wait(accfull_bar, accph, abort_flag, p.status,
                                                          DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns));
                accph ^= 1u;
            } else {
                ok = epilogue(pend);
            }
        }
        // the last copies out have completed before the CTA exits
        if (C::STAGE_OUT && warp == 4 && lane == 0) ptx::bulk_wait_group0();
        if (ok) {
            // tail: every MMA commit aimed at this CTA's operand stages has landed
            for (int j = 0; j < C::A_ST && ok; ++j) {
                ok = __all_sync(0xffffffffu, bounded_wait(aempty_bar(a), aph ^ 1u, abort_flag, p.status,
                                                                DEVICE_TIMEOUT_TRANSFORM, p.timeout_ns));
                if (++a == C::A_ST) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (!PAIR && p.csplit) {
        // Deterministic split-K inside a thread-block cluster (one CTA per slice, one
        // item per CTA, slice = rank).  Every thread of every CTA of the cluster passes
        // both cluster barriers, also after an abort, so no CTA can strand a peer.
        // (1) every slice is past its main loop: the peers' stage memory is free;
        // (2) each CTA sends its accumulator rows to the CTA that owns them (rows
        //     [q R, q R + R) belong to rank q, R = ceil(128 / S)) as remote
        //     shared-memory stores; (3) each CTA adds its own rows over the slices in
        //     order 0..S-1 and stores them.
        const bool good = *abort_flag == 0u;
        const int S = p.splits;
        const int R = (TILE_N + S - 1) / S;
        const int q = (int)ptx::cluster_ctarank();
        const Item it = decode_item(p, (int)blockIdx.x);
        const int m0 = it.m_tile * BN;
        ptx::cluster_sync();
        if (good && warp >= 4) {
            ptx::tc_fence_after();
            const int ew = warp - 4, wg = ew >> 2, quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int owner = r / R;
            const uint32_t dst = ptx::mapa_shared(
                sbase + (uint32_t)(((q * R + (r - owner * R)) * C::CS_PITCH) * 4), (uint32_t)owner);
            constexpr int COLS = BN / NWG;
            constexpr int STEP = COLS >= 16 ? 16 : 8;
            const uint32_t acc_addr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(wg * COLS);
#pragma unroll 1
            for (int cc = 0; cc < COLS; cc += STEP) {
                uint32_t v[16];
                if (STEP == 16) {
                    ptx::tmem_ld16(acc_addr + cc, v);
                } else {
                    uint32_t v8[8];
                    ptx::tmem_ld8(acc_addr + cc, v8);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = v8[j];
                }
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < STEP; j += 4)
                    ptx::st_shared_cluster_v4f32(dst + (uint32_t)(wg * COLS + cc + j) * 4u, __uint_as_float(v[j]),
                                                 __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                                 __uint_as_float(v[j + 3]));
            }
        }
        ptx::tc_fence_before();
        ptx::cluster_sync();
        if (good) {
            ptx::grid_dependency_wait();   // outputs may still be in use by the previous kernel
            const float alpha = group_scaled(FMT) ? 1.0f : __ldg(p.alpha);
            const int row0 = q * R;
            const int rows = min(TILE_N, row0 + R) - row0;
            const int mval = min(BN, p.M - m0);
            const float* box = reinterpret_cast<const float*>(smem);
            const int nbase = it.n_tile * TILE_N + row0;
            const int groups = (mval + 3) / 4;
            // consecutive threads take consecutive weight rows (coalesced output
            // stores), each four tokens with one 16-byte load per slice; every column
            // is summed in slice order 0..S-1
            for (int e = threadIdx.x; e < rows * groups; e += C::NT) {
                const int j = e % rows, c4 = (e / rows) * 4;
                const int n = nbase + j;
                float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                for (int sl = 0; sl < S; ++sl) {
                    const float4 v = *reinterpret_cast<const float4*>(box + (sl * R + j) * C::CS_PITCH + c4);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                if (n < p.N) {
                    float b = 0.0f;
                    if (FMT == FMT_FP8 && p.bias != nullptr) b = load_16bit<BF16>(p.bias, (size_t)n);
                    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (c4 + i < mval) store_out<BF16>(p.out, (size_t)(m0 + c4 + i) * p.N + n, alpha * a4[i] + b);
                }
            }
        }
    }
    // pair: neither CTA leaves (or frees its tensor memory) while the other may
    // still signal it or run MMAs on its operands
    if (PAIR) ptx::cluster_sync();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem, C::TMEM_COLS);
    }
}

// Host-side launcher for one instantiation.
template <int FMT, bool BF16, int BN, int BK, int STAGES, int NWG, bool PAIR = false, int WSTAGES = STAGES>
struct GemmLauncher {
    using C = GemmCfg<FMT, BF16, BN, BK, STAGES, NWG, PAIR, WSTAGES>;
    static constexpr auto kernel = wq_gemm_kernel<FMT, BF16, BN, BK, STAGES, NWG, PAIR, WSTAGES>;
    static cudaError_t prepare() {
        // per device: allow the dynamic shared memory this configuration needs
        static int attr_set[64] = {0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 64 && attr_set[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        // all of L1 as shared memory, so that two CTAs fit where the sizes allow it
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        // split-K clusters of up to 16 CTAs (non-portable size)
        if (e == cudaSuccess && C::CSPLIT_OK)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess && dev < 64) attr_set[dev] = 1;
        return e;
    }
    // Static configuration; with query_device, also the resident CTAs per SM on
    // the current device, from the kernel's registers, its shared memory (plus the
    // per-block reservation), threads per SM and tensor memory (512 columns).
    static KernelConfig config(bool query_device = false) {
        KernelConfig k{FMT, BF16 ? 1 : 0, BN, BK, STAGES, NWG, C::NT, C::SMEM_BYTES, C::TMEM_COLS, C::MIN_BLOCKS};
        if (!query_device || prepare() != cudaSuccess) return k;
        int dev = 0, smem_sm = 0, smem_rsv = 0, regs_sm = 0, thr_sm = 0;
        cudaFuncAttributes fa;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess)
            return k;
        const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
        int n = regs_sm / (regs_warp * (C::NT / 32));
        const int by_smem = smem_sm / (C::SMEM_BYTES + fa.sharedSizeBytes + smem_rsv);
        const int by_thr = thr_sm / C::NT;
        const int by_tmem = 512 / C::TMEM_COLS;
        if (by_smem < n) n = by_smem;
        if (by_thr < n) n = by_thr;
        if (by_tmem < n) n = by_tmem;
        if (n >= 1) k.ctas_per_sm = n;
        if (PAIR) {
            // pairs the GPU holds at once
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(2, 1, 1);
            lc.blockDim = dim3(C::NT, 1, 1);
            lc.dynamicSmemBytes = C::SMEM_BYTES;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            lc.attrs = at;
            lc.numAttrs = 1;
            int nc = 0;
            if (cudaOccupancyMaxActiveClusters(&nc, kernel, &lc) == cudaSuccess) k.max_clusters[2] = nc;
            else (void)cudaGetLastError();
            k.pair = 1;
        }
        if (C::CSPLIT_OK) {
            // split-K clusters of S = 2..16 CTAs the GPU holds at once (0: not launchable)
            for (int S = 2; S <= kMaxDecodeCluster; ++S) {
                cudaLaunchConfig_t lc = {};
                lc.gridDim = dim3((unsigned)S, 1, 1);
                lc.blockDim = dim3(C::NT, 1, 1);
                lc.dynamicSmemBytes = C::SMEM_BYTES;
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeClusterDimension;
                at[0].val.clusterDim.x = (unsigned)S;
                at[0].val.clusterDim.y = 1;
                at[0].val.clusterDim.z = 1;
                lc.attrs = at;
                lc.numAttrs = 1;
                int nc = 0;
                if (cudaOccupancyMaxActiveClusters(&nc, kernel, &lc) != cudaSuccess) {
                    (void)cudaGetLastError();
                    nc = 0;
                }
                k.max_clusters[S] = nc;
            }
            k.csplit_ok = 1;
        }
        return k;
    }
    static cudaError_t launch(const GemmParams& p, int grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(C::NT, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = st;
        // programmatic dependent launch: set-up overlaps the previous kernel's tail
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (PAIR) {
            if (grid % 2 != 0) return cudaErrorInvalidValue;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = 2;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        } else if (p.csplit) {
            // one CTA per (tile, slice), the slices of a tile one cluster
            if (!C::CSPLIT_OK || p.splits < 2 || p.splits > kMaxDecodeCluster || grid != p.n_items ||
                grid % p.splits != 0)
                return cudaErrorInvalidValue;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = (unsigned)p.splits;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        return cudaLaunchKernelEx(&cfg, kernel, p);
    }
};

}  // namespace wq
