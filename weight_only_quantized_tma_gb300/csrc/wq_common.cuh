// wq_common.cuh -- device helpers shared by the tile kernel (wq_gemm.cuh) and the
// register decode kernel (wq_gemm_mma.cuh): the swizzle of TMA tiles, bounded
// mbarrier waits, 16-bit output conversion and the work-item decoding of a GEMM
// launch.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "wq_internal.h"

namespace wq {

// Physical byte offset of a logical offset inside a TMA-swizzled tile whose base
// is 1024-byte aligned (16-byte chunk index XOR the 128-byte row index bits).
__device__ __forceinline__ uint32_t swz(uint32_t a, uint32_t mask) { return a ^ (((a >> 7) & mask) << 4); }

// Bounded wait on an mbarrier phase, executed by every lane that calls it.
// Returns false if the CTA is aborting or the wait timed out (which starts the
// abort).  The global timer is slow to read, so it is only consulted every 256
// failed probes; the abort flag (shared memory) is checked on every probe.
// CLUSTER: the barrier receives arrivals from the other CTA of a cluster pair.
template <bool CLUSTER = false>
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             uint32_t* status, uint32_t code, long long timeout_ns) {
    if (ptx::mbar_try_wait<CLUSTER>(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 255u) == 0u) {
            const uint64_t now = ptx::globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if ((long long)(now - t0) > timeout_ns) {
                *abort_flag = 1u;
                atomicOr(status, code);
                return false;
            }
        }
    }
}

// Wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, long long timeout_ns) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1; !ptx::mbar_try_wait(bar, parity); ++i) {
        if ((i & 255u) == 0u && (long long)(ptx::globaltimer() - t0) > timeout_ns) return false;
    }
    return true;
}

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
    if (BF16)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

template <bool BF16>
__device__ __forceinline__ uint16_t to_16bit(float v) {
    if (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return __half_as_ushort(__float2half_rn(v));
}

template <bool BF16>
__device__ __forceinline__ float load_16bit(const void* p, size_t idx) {
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
    return __half2float(reinterpret_cast<const __half*>(p)[idx]);
}

struct Item {
    int n_tile, m_tile, slice, kb_begin, kb_end;
    int half;    // 1: a half tile (half_bn tokens starting at m_sub), 0: a whole tile
    int m_sub;
};

// Items below p.n_full are whole tiles (or split-K slices of them); the tiles past
// them -- fewer than half the persistent CTAs -- are each split into two half tiles
// along the tokens, so that the last round of work is spread over twice as many
// CTAs without any cross-CTA reduction.
__device__ __forceinline__ Item decode_item(const GemmParams& p, int item) {
    Item it;
    it.half = 0;
    it.m_sub = 0;
    uint32_t t;
    if (item < p.n_full) {
        t = fastdiv((uint32_t)item, p.div_splits);
        it.slice = item - (int)t * p.splits;
    } else {
        const int j = item - p.n_full;
        t = (uint32_t)(p.n_full + (j >> 1));
        it.slice = 0;
        it.half = 1;
        it.m_sub = (j & 1) * p.half_bn;
    }
    if (p.walk_n_fast) {
        const uint32_t mt = fastdiv(t, p.div_walk);
        it.m_tile = (int)mt;
        it.n_tile = (int)t - (int)mt * p.tiles_n;
    } else {
        const uint32_t nt = fastdiv(t, p.div_walk);
        it.n_tile = (int)nt;
        it.m_tile = (int)t - (int)nt * p.tiles_m;
    }
    // no division on the device: nkb = kb_base * splits + kb_rem, the first kb_rem
    // slices take one extra k-block
    it.kb_begin = it.slice * p.kb_base + min(it.slice, p.kb_rem);
    it.kb_end = it.kb_begin + p.kb_base + (it.slice < p.kb_rem ? 1 : 0);
    return it;
}

// INT4 codebook ("Low Bit Triton Kernels": NF4's 16 non-uniform values are a
// lookup table held in registers).  The 16 fp16 entries are split into their low
// bytes (lo[i] byte j = low byte of entry 4i + j) and high bytes, so that byte
// permutes look up four codes at once: one permute over an 8-byte half of a table
// per code range 0-7 / 8-15, a select by bit 3 of each code, and two permutes that
// interleave low and high bytes into fp16 pairs.
struct Lut16 {
    uint32_t lo[4], hi[4];
};
__device__ __forceinline__ Lut16 lut16_load(const uint16_t* lut) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(lut));       // entries 0-7
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(lut) + 1);   // entries 8-15
    const uint32_t e[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};   // word i: entries 2i, 2i + 1
    Lut16 t;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        t.lo[i] = ptx::prmt(e[2 * i], e[2 * i + 1], 0x6420u);
        t.hi[i] = ptx::prmt(e[2 * i], e[2 * i + 1], 0x7531u);
    }
    return t;
}

// The four codes of one row in one fragment-order word (bits 0-3 / 16-19 / 8-11 /
// 24-27 for k, k + 1, k + 8, k + 9 in the lower row half; 4 bits higher in the
// upper half, hshift = 4) -> the fp16 pairs LUT(k, k + 1) and LUT(k + 8, k + 9).
__device__ __forceinline__ void lut16_word(uint32_t w, uint32_t hshift, const Lut16& t, uint32_t& p_lo,
                                           uint32_t& p_hi) {
    const uint32_t u = w >> hshift;                                     // the row's codes in low nibbles
    const uint32_t sel = ((u & 0x0F0Fu) | ((u >> 12) & 0xF0F0u)) & 0x7777u;   // k, k+1, k+8, k+9 (3 bits)
    // 0xFF in the result bytes whose code is >= 8: the sign of word bytes 0, 2, 1, 3
    // after moving each code's bit 3 to bit 7
    const uint32_t m = ptx::prmt(u << 4, 0u, 0xB9A8u);
    const uint32_t lo = ptx::lop3_select(ptx::prmt(t.lo[0], t.lo[1], sel), ptx::prmt(t.lo[2], t.lo[3], sel), m);
    const uint32_t hi = ptx::lop3_select(ptx::prmt(t.hi[0], t.hi[1], sel), ptx::prmt(t.hi[2], t.hi[3], sel), m);
    p_lo = ptx::prmt(lo, hi, 0x5140u);
    p_hi = ptx::prmt(lo, hi, 0x7362u);
}

}  // namespace wq
