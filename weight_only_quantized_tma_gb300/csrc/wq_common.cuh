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

}  // namespace wq
