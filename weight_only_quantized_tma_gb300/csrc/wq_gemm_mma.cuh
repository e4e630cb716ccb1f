// wq_gemm_mma.cuh -- W4A16 decode kernel (M <= 16 tokens).
//
// Decode is bound by HBM: each weight is used by at most 16 tokens.  The tcgen05
// path pays a fixed cost per MMA instruction that, at 16 tokens, is larger than the
// time HBM takes to deliver the instruction's weights (measured on GB300: ~38 ns per
// M=128 N=16 K=16 MMA, ~50 ns per commit, ~170 ns per TMEM operand hand-off).  This
// kernel keeps the contraction in registers instead: packed weights stream through a
// bulk-copy ring into shared memory, each lane turns its 32-bit word straight into an
// m16n8k16 A fragment, and mma.sync accumulates in fp32.  At full HBM rate an SM has
// ~360 cycles per 8 KB of weights, so the instruction count per word decides the
// speed: one shift, four AND-ORs and four subtractions per word (8 weights).
//
// Operand: the fragment-order layout puts the codes of a fragment register at bits
// 0-3/16-19 (rows g) or 4-7/20-23 (rows g + 8) of a word.  One AND-OR with an fp16
// "magic number" gives b + q with b = 1024 (exponent 2^10) or b = 64 (exponent 2^6,
// whose mantissa unit is 1/16); bf16 operands give 128 + q.  Subtracting b + 8 (or
// b + z with a zero point z) leaves q - 8 exactly (small integers), so the MMA sums
// A (q - 8) in fp32 and the group scale is applied once per group on those sums:
//
//   sum_{k in g} A[m,k] (q - 8) s  =  s * sum_{k in g} A[m,k] (q[n,k] - 8)
//
// ("Low Bit Triton Kernels", §03: the dequantized value is (q - 8) * s).  (Measured on
// GB300: one subtraction per register costs less than forming the sums of b + q and
// correcting them per group with activation sums computed by a separate warp, which
// the compute warps had to wait for on every stage: decode step 75.2 -> 73.7 us.)
//
// Work split: one CTA per (128-row tile, K slice).  Warps: 0-3 compute (warp w owns
// rows 32w .. 32w + 31 of the tile, so each row's sum lives in one warp), 4 is the
// producer.  When K is split, the S slices of a tile are the CTAs of one
// thread-block cluster: each sends the fp32 partial sums of every row to the row's
// owner (CTA r owns rows [r R, r R + R), R = ceil(128 / S)) with st.async, which
// completes on the owner's inbox barrier, and each adds its own rows over the ranks in
// rank order, reading only its own shared memory -- deterministic, no workspace, and
// the reduction is spread over all S CTAs.  The producer streams the weights and scales
// of its first stages before waiting for the preceding kernel on the stream
// (programmatic dependent launch): they are constant inputs; activations and outputs
// are touched only after that wait.
#pragma once

#include "wq_common.cuh"

namespace wq {

// Split-K inbox row: token slots of one weight row (8 per 8-token tile), and the row
// pitch in floats (the slots plus 4).
__host__ __device__ constexpr int inbox_row_floats(int NT) { return 8 * NT; }
__host__ __device__ constexpr int inbox_row_pitch(int NT) { return inbox_row_floats(NT) + 4; }

template <int BK, int STAGES, bool ZP = false>
struct MmaDecodeCfg {
    // compute warps: four of 32 weight rows each -- the two 16-row groups of a warp
    // share each activation fragment, which halves the activation reads from shared
    // memory (measured on GB300, in-graph decode step: ~5 % faster than eight warps of
    // 16 rows; two warps of 64 rows ~35 % slower)
    static constexpr int NCW = 4;
    static constexpr int RGW = TILE_N / 16 / NCW;             // 16-row groups per compute warp
    static constexpr int P_WARP = NCW;                        // producer warp
    static constexpr int NTHREADS = 32 * (NCW + 1);
    static constexpr int NZ = BK / 64;                        // 64-wide activation boxes per stage
    // Two rings.  Weights: STAGES slots of packed codes, each released as soon as the
    // compute warps hold its words in registers (at the start of the stage's MMAs), so
    // the next copy into it overlaps the stage's arithmetic (measured on GB300, in-graph
    // decode step: 70.2 -> 68.1 us against one ring released after the MMAs).  Activations, scales (up to
    // BK / 32 groups, G = 32) and zero points (uint8 [BK / 32][128]): AS_STAGES =
    // STAGES + 1 slots, released after the stage's MMAs; one more slot than the weights,
    // so that a weight slot freed for k-block i + STAGES always finds the activation
    // slot of that k-block free as well (its previous user, k-block i - 1, finished
    // before k-block i's words were loaded).  The 128-byte-swizzled activation boxes
    // are 1024-byte aligned.
    static constexpr int AS_STAGES = STAGES + 1;
    static constexpr int W_STAGE = TILE_N * BK / 2;
    static constexpr int A_STAGE = 16 * 128 * NZ;             // up to 16 token rows of 128 bytes per box
    static constexpr int SC_BYTES = (BK / 32) * TILE_N * 2;
    static constexpr int SC_STAGE = SC_BYTES + (ZP ? (BK / 32) * TILE_N : 0);   // zero points at SC_BYTES
    static constexpr int A_BASE = STAGES * W_STAGE;
    static constexpr int SC_BASE = A_BASE + AS_STAGES * A_STAGE;
    // split-K inbox: the partial sums the S CTAs of a cluster send to the CTA that
    // owns at most R = ceil(128 / S) of the tile's rows, fp32 [S][R][16 token slots] --
    // at most 16 * (128 + 15) values; never used by the main loop, so a peer may write
    // into it while this CTA is still streaming.  Token slot 4c + i holds token
    // 2c + (i & 1) + 8 (i >> 1): the order of a lane's accumulator values, so each
    // lane sends a row's values with one vector store.
    static constexpr int INBOX = SC_BASE + AS_STAGES * SC_STAGE;
    static constexpr int INBOX_BYTES = inbox_row_pitch(2) * (TILE_N + 16) * 4;
    static constexpr int OFF_BAR = INBOX + INBOX_BYTES;
    // barriers: full and empty per weight slot, full and empty per activation slot; then
    // the abort flag (4 B, padded to 8) and the inbox barrier (8 B, split-K)
    static constexpr int OFF_INBOX_BAR = OFF_BAR + 2 * (STAGES + AS_STAGES) * 8 + 8;
    static constexpr int SMEM_USED = OFF_INBOX_BAR + 8;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(BK == 128 || BK == 256, "BK");
    static_assert(W_STAGE % 1024 == 0 && A_STAGE % 1024 == 0 && SC_STAGE % 16 == 0,
                  "bulk-copy and swizzle alignment");
};

// Pure register operations: not volatile, so the compiler may interleave them.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          bool bf16) {
    if (bf16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory reads: volatile with a memory clobber, so they stay after the
// barrier wait that makes the data valid.
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// ---------------------------------------------------------------- split-K exchange
// Shared by the decode kernels.  The S slices of a 128-row tile are the CTAs of one
// cluster; CTA `rank` owns rows [128 rank / S, 128 (rank + 1) / S) of the tile (an even
// split: 8 to 64 rows each, none empty for any S <= 16).
// Each CTA sends every row's fp32 partial sums to the row's owner (its own rows to
// itself) with st.async, which completes on the owner's inbox barrier; the owner then
// adds the S slices of its rows in rank order (deterministic) and reads only its own
// shared memory.  No cluster-wide barrier has to wait for the remote stores to
// complete (measured on GB300: a barrier.cluster with release semantics after remote
// stores cost ~1 us per launch).  Inbox: fp32 [S][R = ceil(128 / S)][inbox_row_pitch(NT)]
// per row and slice, the token slots in the order of a lane's accumulator values:
// lane c's values for MMA columns 2c, 2c + 1 of the 8-token tiles nt = 0 .. NT - 1 at
// slots 2 NT c + 2 nt + {0, 1}, so a lane sends a row's values with one to four vector
// stores.  The row pitch is the slot count plus 4: the reduction's
// warps read one slot of 32 consecutive rows, which a pitch of 16 or 32 floats puts on
// 2 or 1 banks (16- or 32-way conflicts); the extra 16 bytes spread them over 8 bank
// quads and keep the rows 16-byte aligned for the vector stores.
// (inbox_row_floats / inbox_row_pitch: the split-K inbox layout, described with the
// exchange helpers below)

// Compute warp `warp` holds rows 16 RGW warp + 16 j + g (+ 8) of the tile in
// acc[j][nt][e] (e = 0, 1: row g, MMA columns 8 nt + 2c + e; e = 2, 3: row g + 8).
template <int NT, int RGW>
__device__ __forceinline__ void decode_send_partials(const float (&acc)[RGW][NT][4], int warp, int lane, int rank,
                                                     int S, int R, uint32_t inbox, uint32_t inbox_bar) {
    constexpr int ROWF = inbox_row_floats(NT);
    constexpr int PITCH = inbox_row_pitch(NT);
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = (warp * RGW + j) * 16 + g + 8 * h;   // e = 2h, 2h + 1
            const int owner = ((r + 1) * S - 1) / TILE_N;       // 128 owner / S <= r < 128 (owner + 1) / S
            const uint32_t off =
                inbox + (uint32_t)((rank * R + (r - owner * TILE_N / S)) * PITCH + (ROWF / 4) * c) * 4u;
            const uint32_t dst = ptx::mapa_shared(off, (uint32_t)owner);
            const uint32_t rbar = ptx::mapa_shared(inbox_bar, (uint32_t)owner);
            if constexpr (NT == 1) {
                ptx::st_async_v2f32(dst, acc[j][0][2 * h], acc[j][0][2 * h + 1], rbar);
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; nt += 2)
                    ptx::st_async_v4f32(dst + 8u * nt, acc[j][nt][2 * h], acc[j][nt][2 * h + 1], acc[j][nt + 1][2 * h],
                                        acc[j][nt + 1][2 * h + 1], rbar);
            }
        }
}

// MMA column n (0..7) of an 8-token tile holds token n, or with SPREAD token
// 2 (n % 4) + n / 4: the half-warp that loads columns 0-3 then reads tokens 0, 2, 4, 6
// (and the other half 1, 3, 5, 7), whose rows of a 128-byte-swizzled activation box
// fall on distinct banks for 8-byte loads.  Inverse: token t sits in column
// t / 2 + 4 (t % 2).
template <bool SPREAD>
__device__ __forceinline__ int token_of_column(int n) { return SPREAD ? 2 * (n & 3) + (n >> 2) : n; }
template <bool SPREAD>
__device__ __forceinline__ int column_of_token(int t) { return SPREAD ? (t >> 1) + 4 * (t & 1) : t; }

// After the inbox phase completed: store(m, r, v) for token m < M and the r-th owned
// row, with v the sum of the S slices in rank order.  Weight row fastest: a warp stores
// consecutive output columns of one token.
template <int NT, bool SPREAD = false, typename Store>
__device__ __forceinline__ void decode_reduce_rows(const float* box, int S, int R, int rows_own, int M, Store store) {
    constexpr int ROWF = inbox_row_floats(NT);
    constexpr int PITCH = inbox_row_pitch(NT);
    for (int e = threadIdx.x; e < M * rows_own; e += blockDim.x) {
        const int m = e / rows_own;
        const int r = e - m * rows_own;
        const int n = column_of_token<SPREAD>(m & 7);   // lane 4 g + n / 2 holds it as value n % 2
        const int slot = (ROWF / 4) * (n >> 1) + (n & 1) + 2 * (m >> 3);
        float tot = 0.0f;
        for (int q = 0; q < S; ++q) tot += box[(q * R + r) * PITCH + slot];
        store(m, r, tot);
    }
}

// b + z of rows g (upper = false) or g + 8 (upper = true) as a pair of 16-bit values:
// fp16 1024 + z and 64 + z (mantissa unit 1/16), bf16 128 + z; z = 8 without zero points.
template <bool BF16>
__device__ __forceinline__ uint32_t int4_offset(bool upper, uint32_t z) {
    const uint32_t v = BF16 ? 0x4300u + z : upper ? 0x5400u + (z << 4) : 0x6400u + z;
    return v | (v << 16);
}

__device__ __forceinline__ uint32_t sub_16x2(uint32_t a, uint32_t b, bool bf16) {
    uint32_t r;
    if (bf16)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// One 32-bit word of the fragment-order layout -> the four A-fragment registers of
// one k step, each holding two values q - z, exact: b + q from an AND-OR with the
// magic number, minus b + z (off_lo for rows g, off_hi for rows g + 8).
template <bool BF16>
__device__ __forceinline__ void int4_word_to_frag(uint32_t w, uint32_t off_lo, uint32_t off_hi, uint32_t (&a)[4]) {
    if (BF16) {
        a[0] = sub_16x2((w & 0x000F000Fu) | 0x43004300u, off_lo, true);           // rows g,     k
        a[1] = sub_16x2(((w >> 4) & 0x000F000Fu) | 0x43004300u, off_hi, true);    // rows g + 8, k
        a[2] = sub_16x2(((w >> 8) & 0x000F000Fu) | 0x43004300u, off_lo, true);    // rows g,     k + 8
        a[3] = sub_16x2(((w >> 12) & 0x000F000Fu) | 0x43004300u, off_hi, true);   // rows g + 8, k + 8
    } else {
        const uint32_t w8 = w >> 8;
        a[0] = sub_16x2((w & 0x000F000Fu) | 0x64006400u, off_lo, false);          // 1024 + q
        a[1] = sub_16x2((w & 0x00F000F0u) | 0x54005400u, off_hi, false);          // 64 + q
        a[2] = sub_16x2((w8 & 0x000F000Fu) | 0x64006400u, off_lo, false);
        a[3] = sub_16x2((w8 & 0x00F000F0u) | 0x54005400u, off_hi, false);
    }
}

// NT: 8-token MMA column tiles (1 for M <= 8, 2 for M <= 16).  GSTEPS: 16-wide k
// steps per scale group inside a stage (2, 4, 8 or 16; G >= BK folds once per stage).
// One CTA per item (tile, K slice): gridDim.x == n_items, and the slices of a tile form
// one cluster of p.splits CTAs.  ZP: per-(group, row) zero points, operands q - z.
// LUT: the codebook format (fp16 activations), operands LUT[q] looked up with byte
// permutes from a table in registers (lut16_word gives rows g / g + 8 of a word for
// shifts 0 / 4, pairs k, k + 1 and k + 8, k + 9: the fragment registers a0 .. a3); the
// group scale multiplies the fp32 sums, so an output is RN16(s * sum A LUT[q]).
template <bool BF16, int NT, int GSTEPS, int BK, int STAGES, bool ZP = false, bool LUT = false>
__global__ void __launch_bounds__(MmaDecodeCfg<BK, STAGES, ZP>::NTHREADS, LUT ? 3 : 2)
    wq_decode_mma_kernel(const __grid_constant__ GemmParams p) {
    static_assert(!LUT || (!ZP && !BF16), "codebook decode: fp16 activations, no zero points");
    using C = MmaDecodeCfg<BK, STAGES, ZP>;
    constexpr int NZ = C::NZ;
    constexpr int NCW = C::NCW;
    constexpr int RGW = C::RGW;
    constexpr int KSTEPS = BK / 16;
    constexpr int SETS = NT == 1 ? 2 : 1;               // accumulator sets per chain (even / odd k steps)
    static_assert((GSTEPS == 2 || GSTEPS == 4 || GSTEPS == 8 || GSTEPS == 16) && GSTEPS <= KSTEPS, "GSTEPS");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    constexpr int AS = C::AS_STAGES;
    auto full_w = [&](int s) { return bar0 + 8u * s; };
    auto empty_w = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto full_as = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto empty_as = [&](int s) { return bar0 + 8u * (2 * STAGES + AS + s); };
    volatile uint32_t* abort_flag =
        reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + 2 * (STAGES + AS) * 8);
    const uint32_t inbox_bar = sbase + C::OFF_INBOX_BAR;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Item it = decode_item(p, (int)blockIdx.x);
    const int nunits = it.kb_end - it.kb_begin;
    const int tile = it.n_tile;
    // split-K: CTA `rank` of the tile's cluster owns rows [128 rank / S, 128 (rank + 1) / S)
    const int S = p.splits;
    const int R = (TILE_N + S - 1) / S;   // inbox rows per slice: an owner's rows, at most
    const int rank = S > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int row0 = rank * TILE_N / S;
    const int rows_own = (rank + 1) * TILE_N / S - row0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_w(s), 1);
            ptx::mbar_init(empty_w(s), NCW);
        }
        for (int s = 0; s < AS; ++s) {
            ptx::mbar_init(full_as(s), 1);
            ptx::mbar_init(empty_as(s), NCW);
        }
        ptx::mbar_init(inbox_bar, 1);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
        // the inbox phase completes once the S slices' partial rows of this CTA's rows
        // (NT x 32 bytes per row and slice) have landed
        if (S > 1) ptx::mbar_arrive_expect_tx(inbox_bar, (uint32_t)(S * rows_own * NT * 32));
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::P_WARP && lane == 0) ptx::prefetch_tmap(&p.tmap_a);
    __syncthreads();
    // every CTA of the cluster arrives once its barriers exist; the matching wait,
    // before the first remote store, is long satisfied by then
    if (S > 1) ptx::cluster_arrive_relaxed();
    if (threadIdx.x == 0) ptx::grid_launch_dependents();

    // activation fragment addresses inside a stage's boxes (box z = t / 4 holds k
    // 64z .. 64z + 63 as 128-byte token rows, row z * M + m, 128-byte swizzle);
    // ldmatrix lane l addresses row l % 8 of matrix l / 8: (tokens 0-7, k 0-7),
    // (0-7, k 8-15), (8-15, k 0-7), (8-15, k 8-15) of a k step
    uint32_t a_off[KSTEPS];
    {
        const int mi = lane >> 3;
        const int a_row = (NT == 2 ? (mi >> 1) * 8 : 0) + (lane & 7);
#pragma unroll
        for (int t = 0; t < KSTEPS; ++t) {
            const int row = (t >> 2) * p.a_box_rows + a_row;
            const int chunk = (t & 3) * 2 + (mi & 1);
            a_off[t] = row * 128 + ((chunk ^ (row & 7)) << 4);
        }
    }

    // compute warps: rows 16 RGW w + 16j + g (e = 0, 1) and + 8 (e = 2, 3) of the tile
    float acc[RGW][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.0f;

    if (warp == C::P_WARP) {
        // ------------------------------------------------------------ producer
        // Lane 0 streams both rings.  The weights of the first STAGES k-blocks and the
        // scales (and zero points) of the first AS go out at once, before the grid
        // dependency wait (constant inputs), the activation copies right after it.  The
        // order in which a slot's bytes land does not matter: its phase cannot complete
        // before this lane's arrive-expect-tx.  The loop after that can stop early only
        // at a wait, and it waits only after passing those slots, so every barrier armed
        // here gets all of its bytes.
        const int pre_w = nunits < STAGES ? nunits : STAGES;
        const int pre_as = nunits < AS ? nunits : AS;
        const uint32_t a_bytes = (uint32_t)NZ * (uint32_t)p.a_box_rows * 128u;
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_a = ptx::policy_evict_last();
            const int gcnt = (p.G >= BK) ? 1 : (BK >> p.g_shift);
            const uint32_t sc_bytes = (uint32_t)gcnt * TILE_N * 2;
            const uint32_t zp_bytes = ZP ? (uint32_t)gcnt * TILE_N : 0u;
            auto load_w = [&](int s, int kb) {
                const uint32_t fb = full_w(s);
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)C::W_STAGE);
                const uint8_t* wsrc =
                    p.w + ((size_t)tile * p.nchunks_pad + (size_t)kb * (BK / 32)) * (TILE_N * 16);
                ptx::bulk_load(sbase + s * C::W_STAGE, wsrc, C::W_STAGE, fb, pol_w);
            };
            // scales (+ zero points) of k-block kb; arms the slot for them and its activations
            auto load_s = [&](int s, int kb) {
                const uint32_t fb = full_as(s);
                const uint32_t dst = sbase + C::SC_BASE + s * C::SC_STAGE;
                ptx::mbar_arrive_expect_tx(fb, sc_bytes + zp_bytes + a_bytes);
                const int g0 = (kb * BK) >> p.g_shift;
                ptx::bulk_load(dst, p.sc + ((size_t)tile * p.ngroups_pad + g0) * (TILE_N * 2), sc_bytes, fb, pol_w);
                if (ZP)
                    ptx::bulk_load(dst + C::SC_BYTES, p.zp + ((size_t)tile * p.ngroups_pad + g0) * TILE_N, zp_bytes,
                                   fb, pol_w);
            };
            // activation box {64 k, M tokens, NZ}: k-block kb starts at z = kb * NZ
            auto load_a = [&](int s, int kb) {
                ptx::tma_load_3d(sbase + C::A_BASE + s * C::A_STAGE, &p.tmap_a, 0, 0, kb * NZ, full_as(s), pol_a);
            };
            for (int i = 0; i < pre_w; ++i) load_w(i, it.kb_begin + i);
            for (int i = 0; i < pre_as; ++i) load_s(i, it.kb_begin + i);
            ptx::grid_dependency_wait();
            for (int i = 0; i < pre_as; ++i) load_a(i, it.kb_begin + i);
            int sw = pre_w % STAGES, sa = pre_as % AS;
            uint32_t phw = pre_w == STAGES ? 1u : 0u, pha = pre_as == AS ? 1u : 0u;
            int issued_w = pre_w, issued_as = pre_as;
            for (int i = pre_w; i < nunits; ++i) {
                const int kb = it.kb_begin + i;
                if (!bounded_wait(empty_w(sw), phw ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_PRODUCER,
                                  p.timeout_ns))
                    break;
                load_w(sw, kb);
                ++issued_w;
                if (++sw == STAGES) {
                    sw = 0;
                    phw ^= 1u;
                }
                if (i < pre_as) continue;
                if (!bounded_wait(empty_as(sa), pha ^ 1u, abort_flag, p.status, DEVICE_TIMEOUT_PRODUCER,
                                  p.timeout_ns))
                    break;
                load_s(sa, kb);
                load_a(sa, kb);
                ++issued_as;
                if (++sa == AS) {
                    sa = 0;
                    pha ^= 1u;
                }
            }
            if (*abort_flag) {
                for (int j = issued_w > STAGES ? issued_w - STAGES : 0; j < issued_w; ++j)
                    if (!drain_wait(full_w(j % STAGES), (uint32_t)((j / STAGES) & 1), p.timeout_ns))
                        atomicOr(p.status, DEVICE_TIMEOUT_DRAIN);
                for (int j = issued_as > AS ? issued_as - AS : 0; j < issued_as; ++j)
                    if (!drain_wait(full_as(j % AS), (uint32_t)((j / AS) & 1), p.timeout_ns))
                        atomicOr(p.status, DEVICE_TIMEOUT_DRAIN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute warps
        const int g = lane >> 2, c = lane & 3;
        const int slot = int4_slot(lane);
        // the table may be written by the kernel before this one on the stream: read it
        // after the dependency wait (the first stage's activations wait for it anyway)
        Lut16 tab{};
        if constexpr (LUT) {
            ptx::grid_dependency_wait();
            tab = lut16_load(p.lut);
        }
        const int w_off = warp * RGW * 512 + slot * 16;   // this warp's first 16-row group, this lane's slot
        int sw = 0, sa = 0;
        uint32_t phw = 0, pha = 0;
        for (int i = 0; i < nunits; ++i) {
            // the stage's weight words into registers, then the weight slot is free
            // (the arrive releases the loads before it, and __syncwarp orders the other
            // lanes' loads before lane 0's arrive)
            const bool okw = bounded_wait(full_w(sw), phw, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM,
                                          p.timeout_ns);
            if (!__all_sync(0xffffffffu, okw)) break;
            const uint8_t* wst = smem + sw * C::W_STAGE;
            uint4 wv[KSTEPS / 4][RGW];
#pragma unroll
            for (int tq = 0; tq < KSTEPS / 4; ++tq)
#pragma unroll
                for (int j = 0; j < RGW; ++j)
                    wv[tq][j] = *reinterpret_cast<const uint4*>(wst + tq * 4096 + w_off + j * 512);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty_w(sw));
            if (++sw == STAGES) {
                sw = 0;
                phw ^= 1u;
            }
            const bool oka = bounded_wait(full_as(sa), pha, abort_flag, p.status, DEVICE_TIMEOUT_TRANSFORM,
                                          p.timeout_ns);
            if (!__all_sync(0xffffffffu, oka)) break;
            const uint8_t* scp = smem + C::SC_BASE + sa * C::SC_STAGE;
            const uint32_t st = sbase + C::A_BASE + sa * C::A_STAGE;   // this stage's activation boxes
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(scp);
            float tmp[RGW][SETS][NT][4];
            uint32_t off_lo[RGW], off_hi[RGW];   // b + z of the group, rows g and g + 8
#pragma unroll
            for (int t = 0; t < KSTEPS; ++t) {
                if (t % GSTEPS == 0) {
                    // group start: sums from zero; the zero points of the group's rows
#pragma unroll
                    for (int j = 0; j < RGW; ++j) {
#pragma unroll
                        for (int h = 0; h < SETS; ++h)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) tmp[j][h][nt][e] = 0.0f;
                        uint32_t z_lo = 8u, z_hi = 8u;
                        if constexpr (ZP) {
                            const uint8_t* zp = scp + C::SC_BYTES + (t / GSTEPS) * TILE_N + (warp * RGW + j) * 16 + g;
                            z_lo = zp[0];
                            z_hi = zp[8];
                        }
                        off_lo[j] = int4_offset<BF16>(false, z_lo);
                        off_hi[j] = int4_offset<BF16>(true, z_hi);
                    }
                }
                uint32_t b[NT][2];
                if constexpr (NT == 2)
                    ldmatrix_x4(st + a_off[t], b[0][0], b[0][1], b[NT - 1][0], b[NT - 1][1]);
                else
                    ldmatrix_x2(st + a_off[t], b[0][0], b[0][1]);
#pragma unroll
                for (int j = 0; j < RGW; ++j) {
                    const uint4& q4 = wv[t >> 2][j];
                    const uint32_t word = (t & 3) == 0 ? q4.x : (t & 3) == 1 ? q4.y : (t & 3) == 2 ? q4.z : q4.w;
                    uint32_t a[4];
                    if constexpr (LUT) {
                        lut16_word(word, 0u, tab, a[0], a[2]);   // rows g:     k, k + 1 / k + 8, k + 9
                        lut16_word(word, 4u, tab, a[1], a[3]);   // rows g + 8
                    } else {
                        int4_word_to_frag<BF16>(word, off_lo[j], off_hi[j], a);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_16816(tmp[j][t % SETS][nt], a, b[nt][0], b[nt][1], BF16);
                }
                if ((t + 1) % GSTEPS == 0) {
                    // acc += s * sum_{k in group} A (q - z)
                    const int gi = t / GSTEPS;
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
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty_as(sa));
            if (++sa == AS) {
                sa = 0;
                pha ^= 1u;
            }
        }
    }
    // Every stage was consumed, or drained after an abort: the stage memory is free.
    // From here on every thread of the CTA runs the same sequence (no early exit), so
    // the cluster barriers below are always reached.
    __syncthreads();
    ptx::grid_dependency_wait();   // out may still be read upstream
    const int g = lane >> 2, c = lane & 3;
    if (p.splits == 1) {
        if (warp < NCW) {
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
        // split-K: partial rows to their owners, the owners add them in rank order
        ptx::cluster_wait();   // every CTA of the cluster has initialised its barriers
        if (warp < NCW) decode_send_partials<NT, RGW>(acc, warp, lane, rank, S, R, sbase + C::INBOX, inbox_bar);
        // (bounded like every wait: a timeout sets the status word; nothing is read then)
        if (!bounded_wait<true>(inbox_bar, 0u, abort_flag, p.status, DEVICE_TIMEOUT_EPILOGUE, p.timeout_ns)) return;
        decode_reduce_rows<NT>(reinterpret_cast<const float*>(smem + C::INBOX), S, R, rows_own, p.M,
                           [&](int m, int r, float v) {
                               const int n = tile * TILE_N + row0 + r;
                               if (n < p.N) store_out<BF16>(p.out, (size_t)m * p.N + n, v);
                           });
    }
}

// Resident CTAs per SM of a decode kernel from registers, shared memory, threads and
// the block limit; and, per cluster size S = 2..16, how many S-CTA clusters the device
// can hold at once (the plan keeps a split-K grid within one such wave).
template <typename Kernel>
void decode_residency(Kernel kernel, int threads, int smem_bytes, KernelConfig* k) {
    // the occupancy calculator rather than registers / (registers per CTA): a CTA of
    // five warps spreads unevenly over the SM's four schedulers, whose register files
    // are separate (at 133 registers three CTAs fit the SM's total but not the
    // scheduler that holds four of the fifteen warps)
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, (size_t)smem_bytes) != cudaSuccess) return;
    if (n >= 1) k->ctas_per_sm = n;
    for (int S = 2; S <= kMaxDecodeCluster; ++S) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)S, 1, 1);
        cfg.blockDim = dim3((unsigned)threads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            nc = 0;
        }
        k->max_clusters[S] = nc;
    }
}

// One CTA per (tile, slice); the slices of a tile form one cluster.  Programmatic
// dependent launch: the kernel waits for its predecessor only where it must.
template <typename Kernel>
cudaError_t launch_decode_grid(Kernel kernel, const GemmParams& p, int grid, int threads, int smem_bytes,
                               cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)(p.splits > 1 ? p.splits : 1);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.splits > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <bool BF16, int NT, int GSTEPS, int BK, int STAGES, bool ZP = false, bool LUT = false>
struct MmaDecodeLauncher {
    using C = MmaDecodeCfg<BK, STAGES, ZP>;
    static constexpr auto kernel = wq_decode_mma_kernel<BF16, NT, GSTEPS, BK, STAGES, ZP, LUT>;
    static cudaError_t prepare() {
        static int attr_set[64] = {0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 64 && attr_set[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        // clusters of up to 16 CTAs (the split-K slices of one tile)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess && dev < 64) attr_set[dev] = 1;
        return e;
    }
    static KernelConfig config(bool query_device) {
        KernelConfig k{LUT ? FMT_LUT4 : FMT_INT4, BF16 ? 1 : 0, 16, BK, STAGES, 0, C::NTHREADS, C::SMEM_BYTES, 0, 1};
        if (!query_device || prepare() != cudaSuccess) return k;
        decode_residency(kernel, C::NTHREADS, C::SMEM_BYTES, &k);
        return k;
    }
    static cudaError_t launch(const GemmParams& p, int grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        if (p.splits > kMaxDecodeCluster || grid != p.n_items || p.M > 16 || p.M < 1) return cudaErrorInvalidValue;
        return launch_decode_grid(kernel, p, grid, C::NTHREADS, C::SMEM_BYTES, st);
    }
};

}  // namespace wq
