// wq_api.cu -- the C ABI (include/wq.h): argument validation, launch planning,
// tensor-map encoding and kernel launches.  Host code only, apart from the
// per-device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/wq.h"
#include "wq_internal.h"

namespace wq {

// One status word per device (bounded-wait timeouts, see include/wq.h).
__device__ uint32_t g_device_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kTimeoutNs = 2000000000LL;  // 2 s bound on every barrier wait

struct DeviceInfo {
    std::once_flag once;
    bool supported = false;
    int sms = 0;
    uint32_t* status = nullptr;
    cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

wq_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WQ_ERR_UNSUPPORTED_DEVICE;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&]() {
        int major = 0, minor = 0;
        d.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        d.supported = (d.err == cudaSuccess) && major == 10 && minor == 3;
        if (d.supported) {
            void* p = nullptr;
            d.err = cudaGetSymbolAddress(&p, g_device_status);
            d.status = static_cast<uint32_t*>(p);
            if (d.err != cudaSuccess) d.supported = false;
        }
    });
    if (d.err != cudaSuccess) return WQ_ERR_CUDA;
    if (!d.supported) return WQ_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return WQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_group(int32_t G) { return G == 32 || G == 64 || G == 128 || G == 256; }

// ------------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, []() {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

CUtensorMapSwizzle swizzle_for_pitch(int pitch_bytes) {
    switch (pitch_bytes) {
        case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
        case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
        default: return CU_TENSOR_MAP_SWIZZLE_32B;
    }
}

// ------------------------------------------------------------------ planning

struct Plan {
    KernelConfig cfg;
    int tiles_n, tiles_m, nkb, splits, n_items, grid, walk_n_fast;
    int n_full;    // tile kernel: whole-tile items; the rest are half tiles
    size_t ws_bytes;
    bool decode;   // register-resident mma.sync decode kernel (M <= 16; FP8 M <= 32)
    bool pair;     // tile kernel on two-CTA clusters (256 weight rows per tile)
    bool csplit;   // tile kernel split-K reduced inside thread-block clusters (no workspace)
};

// Configuration codes past the tile formats: the decode kernels, then the pair kernels.
constexpr int kCfgDecodeInt4 = 16;     // + decode_kind (0 symmetric, 1 zero points)
constexpr int kCfgDecodeFp8 = 18;
constexpr int kCfgDecodeFp4 = 19;
constexpr int kCfgDecodeFp8N4 = 20;   // FP8 decode with 4 token tiles (M <= 32)
constexpr int kCfgDecodeFp4N1 = 21;   // FP4 decode with one token tile (M <= 8)
constexpr int kCfgDecodeLut = 22;     // codebook INT4 decode (fp16 activations)
constexpr int kCfgDecodeInt2 = 23;    // INT2 decode with two / one token tiles
constexpr int kCfgDecodeInt2N1 = 24;
constexpr int kNumDecodeCfgs = 9;
constexpr int kCfgPair = 32;           // + format

bool get_config_uncached(int fmt, bool bf16, int bn, bool query, KernelConfig* cfg) {
    if (fmt == kCfgDecodeInt4) return config_int4_decode(bf16, query, cfg);
    if (fmt == kCfgDecodeInt4 + 1) return config_int4_decode_zp(bf16, query, cfg);
    if (fmt == kCfgDecodeFp8) return config_fp8_decode(bf16, 2, query, cfg);
    if (fmt == kCfgDecodeFp8N4) return config_fp8_decode(bf16, 4, query, cfg);
    if (fmt == kCfgDecodeFp4) return bf16 && config_fp4_decode(2, query, cfg);
    if (fmt == kCfgDecodeFp4N1) return bf16 && config_fp4_decode(1, query, cfg);
    if (fmt == kCfgDecodeLut) return !bf16 && config_int4_decode_lut(query, cfg);
    if (fmt == kCfgDecodeInt2) return config_int2_decode(bf16, 2, query, cfg);
    if (fmt == kCfgDecodeInt2N1) return config_int2_decode(bf16, 1, query, cfg);
    if (fmt == kCfgPair + FMT_INT4) return config_int4_pair(bf16, query, cfg);
    if (fmt == kCfgPair + FMT_FP8) return config_fp8_pair(bf16, query, cfg);
    if (fmt == kCfgPair + FMT_FP4) return bf16 && config_fp4_pair(query, cfg);
    if (fmt == kCfgPair + FMT_LUT4) return config_lut4_pair(bf16, query, cfg);
    if (fmt == kCfgPair + FMT_INT2) return config_int2_pair(bf16, query, cfg);
    switch (fmt) {
        case FMT_INT4: return config_int4(bf16, bn, query, cfg);
        case FMT_FP8: return config_fp8(bf16, bn, query, cfg);
        case FMT_FP4: return config_fp4(bf16, bn, query, cfg);
        case FMT_LUT4: return config_lut4(bf16, bn, query, cfg);
        case FMT_INT2: return config_int2(bf16, bn, query, cfg);
    }
    return false;
}

// The device query behind a configuration (attributes, residency) is done once per
// device and instantiation; later calls read the cached answer.
// Slots: the tile formats 0 .. kNumFmts - 1, the decode kernels (W4A16 symmetric, W4A16
// zero point, FP8, FP4, FP8 with 4 and 8 token tiles), the pair kernels.
constexpr int kCfgSlots = 2 * kNumFmts + kNumDecodeCfgs;
struct ConfigCache {
    std::mutex mu;
    bool have[kMaxDevices][kCfgSlots][2][4] = {};
    bool found[kMaxDevices][kCfgSlots][2][4] = {};
    KernelConfig cfg[kMaxDevices][kCfgSlots][2][4];
};
ConfigCache g_cfg_cache;

bool get_config(int fmt, bool bf16, int bn, bool query, KernelConfig* cfg) {
    const int bi = bn == 16 ? 0 : bn == 64 ? 1 : bn == 128 ? 2 : bn == 256 ? 3 : -1;
    const int fi = (fmt >= kCfgDecodeInt4 && fmt < kCfgPair) ? kNumFmts + (fmt - kCfgDecodeInt4)
                   : fmt >= kCfgPair                          ? kNumFmts + kNumDecodeCfgs + (fmt - kCfgPair)
                                                              : fmt;
    int dev = 0;
    if (!query || bi < 0 || fi < 0 || fi >= kCfgSlots || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices)
        return get_config_uncached(fmt, bf16, bn, query, cfg);
    std::lock_guard<std::mutex> lock(g_cfg_cache.mu);
    const int b = bf16 ? 1 : 0;
    if (!g_cfg_cache.have[dev][fi][b][bi]) {
        g_cfg_cache.found[dev][fi][b][bi] = get_config_uncached(fmt, bf16, bn, true, &g_cfg_cache.cfg[dev][fi][b][bi]);
        g_cfg_cache.have[dev][fi][b][bi] = true;
    }
    if (g_cfg_cache.found[dev][fi][b][bi]) *cfg = g_cfg_cache.cfg[dev][fi][b][bi];
    return g_cfg_cache.found[dev][fi][b][bi];
}

// Split-K workspace: the arrival counters (kSplitCounterBytes) followed by the fp32
// partials.  Keeping the counters at a fixed place lets calls of different shapes
// share one workspace: every call leaves the counters zero again.
size_t split_ws_bytes(int tiles, int splits, int bn) {
    if (splits <= 1) return 0;
    return kSplitCounterBytes + (size_t)tiles * splits * bn * TILE_N * sizeof(float);
}

// WQ_DISABLE_DECODE=1 in the environment keeps decode shapes on the tile kernel, e.g. to
// compare the two.
bool decode_disabled() {
    const char* e = std::getenv("WQ_DISABLE_DECODE");
    return e && e[0] == '1';
}

// Deterministic in (fmt, dtype, M, N, K) and the device's SM count.
//  * token tile BN: the smallest compiled tile that covers M (16, 64, 128), 256
//    for larger M;
//  * split-K when the output tiles cannot occupy every CTA slot of the GPU
//    (decode): slices = slots / tiles, each slice at least two k-blocks, at most
//    16 -- the motivation is the "fused split-K fix-up for grids that do not fill
//    the SMs" of "FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis", §1.  The decode
//    kernel reduces its slices inside a thread-block cluster instead (no workspace);
//  * tile walk order ("FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis", §4): when
//    the weight is the smaller operand, walk weight-row tiles fastest so the
//    activation panel being reused stays in L2, else walk token tiles fastest.
wq_status make_plan(int fmt, bool bf16, int64_t M, int64_t N, int64_t K, int sms, int w_bits, Plan* plan,
                    int G = 0, int decode_kind = 0) {
    static const int kTiles[4] = {16, 64, 128, 256};
    KernelConfig cfg{};
    bool found = false;
    // decode (M <= 16; FP8 M <= 32): the register-resident kernels (W4A16, codebook INT4
    // with fp16 activations, INT2 with G >= 64, FP8, FP4);
    // their activation copy views A as 64-wide boxes, so they need K % 64 == 0 (FP4:
    // whole 256-code stages, K % 256 == 0, so that no stage reads block scales past K;
    // INT2: whole 256-code stages too, and G >= 64 so that each 64-code chunk lies in
    // one group)
    // decode_kind (W4A16): 0 symmetric, 1 zero points, -1 no decode kernel
    const bool decode = decode_kind >= 0 &&
                        (fmt == FMT_INT4 || fmt == FMT_FP8 || fmt == FMT_FP4 || (fmt == FMT_LUT4 && !bf16) ||
                         (fmt == FMT_INT2 && G >= 64)) &&
                        M <= (fmt == FMT_FP8 ? 32 : 16) &&
                        K % ((fmt == FMT_FP4 || fmt == FMT_INT2) ? 256 : 64) == 0 && !decode_disabled();
    if (decode && fmt == FMT_FP4) {
        found = get_config(M <= 8 ? kCfgDecodeFp4N1 : kCfgDecodeFp4, bf16, 16, sms > 0, &cfg);
    } else if (decode && fmt == FMT_INT2) {
        found = get_config(M <= 8 ? kCfgDecodeInt2N1 : kCfgDecodeInt2, bf16, 16, sms > 0, &cfg);
    } else if (decode && fmt == FMT_FP8) {
        found = get_config(M <= 16 ? kCfgDecodeFp8 : kCfgDecodeFp8N4, bf16, 16, sms > 0, &cfg);
    } else if (decode) {
        found = get_config(fmt == FMT_LUT4 ? kCfgDecodeLut : kCfgDecodeInt4 + decode_kind, bf16, 16, sms > 0, &cfg);
        // stages of 256 values when K allows (the launch picks the same instantiation,
        // half as many stages); the codebook kernel keeps stages of 128
        if (found && K % 256 == 0 && fmt != FMT_LUT4) {
            cfg.bk = 256;
            cfg.stages /= 2;
        }
    }
    for (int i = 0; i < 4 && !found; ++i) {
        if (M <= kTiles[i] || i == 3) found = get_config(fmt, bf16, kTiles[i], sms > 0, &cfg);
    }
    for (int i = 3; i >= 0 && !found; --i) found = get_config(fmt, bf16, kTiles[i], sms > 0, &cfg);
    if (!found) return WQ_ERR_DTYPE;
    Plan p{};
    p.cfg = cfg;
    p.decode = decode;
    p.tiles_n = (int)((N + TILE_N - 1) / TILE_N);
    p.tiles_m = (int)((M + cfg.bn - 1) / cfg.bn);
    p.nkb = (int)((K + cfg.bk - 1) / cfg.bk);
    const long long tiles = (long long)p.tiles_n * p.tiles_m;
    const int slots = (sms > 0 ? sms : 148) * (cfg.ctas_per_sm > 0 ? cfg.ctas_per_sm : 1);
    int splits = 1;
    if (tiles < slots && tiles <= kMaxSplitTiles) {
        splits = (int)(slots / tiles);
        const int max_by_k = p.nkb / 2 > 1 ? p.nkb / 2 : 1;
        if (splits > max_by_k) splits = max_by_k;
        if (splits > 16) splits = 16;
        if (splits < 1) splits = 1;
    }
    p.splits = splits;
    long long items = tiles * splits;
    if (decode) {
        // split-K across a cluster of S CTAs (one slice each): S <= 16, at least two
        // k-blocks per slice, tiles x S within the CTAs the GPU holds at once (two or
        // three per SM by the kernel's shared memory), and all clusters in one wave
        // with a margin of 1/16 below the cluster
        // count the occupancy query reports: the hardware does not place that many at
        // once (measured on GB300, 3-CTA clusters, capacity reported 97: W4A16 M = 1,
        // K = 4096 takes 8.7 us at 90 tiles, 9.7 at 93, 11.7 at 95 and 13.0 at 96,
        // against 10.5 us with 2 slices at 96 tiles); the largest such S
        const long long budget = (long long)(sms > 0 ? sms : 148) * (cfg.ctas_per_sm > 0 ? cfg.ctas_per_sm : 1);
        int best = 1;
        for (int S = 2; S <= kMaxDecodeCluster; ++S) {
            const int cap = cfg.max_clusters[S];
            if (p.nkb >= 2 * S && tiles * S <= budget && tiles <= cap - (cap + 15) / 16) best = S;
        }
        p.splits = best;
        items = tiles * best;
    }
    if (items >= (1LL << 31)) return WQ_ERR_SHAPE;
    p.n_items = (int)items;
    p.n_full = (int)items;
    p.grid = (int)(items < slots || decode ? items : slots);   // decode: one CTA per item
    // Tile kernel without split-K: whole tiles in rounds over the persistent CTAs; the
    // R tiles left after the last full round, if at most half the CTAs, become 2R half
    // tiles (BN / 2 tokens each), so the last round takes half a tile's time on twice
    // as many CTAs (e.g. 512 tiles on 152 CTAs: 3.5 instead of 4 tile-times).
    if (!decode && p.splits == 1 && cfg.bn >= 64 && slots > 0) {
        const long long n_full = tiles / slots * slots;
        const long long rem = tiles - n_full;
        if (rem > 0 && 2 * rem <= slots) {
            p.n_full = (int)n_full;
            p.n_items = (int)(n_full + 2 * rem);
            p.grid = (int)(p.n_items < slots ? p.n_items : slots);
        }
    }
    // Large M: 256 x 256 tiles on two-CTA clusters halve the activation bytes each
    // SM reads per MMA.  Used when the pair tiles fill every pair slot at least once.
    // (WQ_DISABLE_PAIR=1 in the environment keeps the one-CTA tile kernel, e.g. to
    // compare the two)
    const char* no_pair = std::getenv("WQ_DISABLE_PAIR");
    const bool pair_allowed = !(no_pair && no_pair[0] == '1');
    if (pair_allowed && !decode && cfg.bn == 256 && p.splits == 1 && sms > 0 && N % 8 == 0) {
        KernelConfig pc{};
        if (get_config(kCfgPair + fmt, bf16, 256, true, &pc) && pc.max_clusters[2] > 0) {
            const long long tn2 = (p.tiles_n + 1) / 2;
            const long long items2 = tn2 * p.tiles_m;
            const long long pslots = pc.max_clusters[2];
            if (items2 >= pslots && items2 < (1LL << 30)) {
                p.cfg = pc;
                p.pair = true;
                p.nkb = (int)((K + pc.bk - 1) / pc.bk);   // the pair kernel's k-block may differ
                p.tiles_n = (int)tn2;
                p.n_items = (int)items2;
                p.n_full = (int)items2;
                // the same half-tile tail as the one-CTA walk, over pair slots
                const long long n_full = items2 / pslots * pslots;
                const long long rem = items2 - n_full;
                if (rem > 0 && 2 * rem <= pslots) {
                    p.n_full = (int)n_full;
                    p.n_items = (int)(n_full + 2 * rem);
                }
                p.grid = 2 * (int)(p.n_items < pslots ? p.n_items : pslots);
            }
        }
    }
    // Split-K on the one-CTA tile kernel with token tiles of 64 or more: the S slices
    // of a tile can form one thread-block cluster and reduce through distributed
    // shared memory (one item per CTA, no workspace).  The device holds fewer S-CTA
    // clusters of this kernel than slots / S (about one CTA per SM), and all clusters
    // must be resident at once, so the cluster path runs S_c <= S slices: the largest
    // count with tiles <= max_clusters[S_c].  It is taken when a cost estimate in
    // quarter microseconds, from per-CTA globaltimer traces and timings on GB300,
    // favours it:
    //   workspace: 3 per k-block of a slice (two CTAs share an SM) plus, for the last
    //              arriving warp, 2 per round of 8 columns x 2 slices;
    //   cluster:   2 per k-block (about one CTA per SM) plus 6 for the exchange.
    // (Measured: 4096 x 4096 at M = 128, 20.7 us with 4 slices in clusters against
    // 37 us with 9 through the workspace; 2048 x 8192 at M = 128, 22.5 against 47 us;
    // 6656 x 19968 at M = 128, 71 us with 2 slices in clusters against 61 us with 5.)
    // WQ_SPLITK_WORKSPACE=1 keeps the workspace reduction; WQ_SPLITK_CLUSTER=1 takes the
    // cluster reduction whenever the clusters fit in one wave (any token tile), e.g. to
    // compare the two.
    const char* cl_env = std::getenv("WQ_SPLITK_CLUSTER");
    const bool force_cluster = cl_env && cl_env[0] == '1';
    if (!decode && !p.pair && p.splits > 1 && cfg.csplit_ok && p.grid == p.n_items && sms > 0 &&
        (force_cluster || cfg.bn >= 64)) {
        const char* ws_env = std::getenv("WQ_SPLITK_WORKSPACE");
        int best = 0;
        for (int S = 2; S <= p.splits && S <= kMaxDecodeCluster; ++S)
            if (tiles <= cfg.max_clusters[S] && p.nkb >= 2 * S) best = S;
        const int cols = cfg.bn / (cfg.nwg > 0 ? cfg.nwg : 2);   // output columns per epilogue warp
        const long long est_ws = 3LL * ((p.nkb + p.splits - 1) / p.splits) +
                                 2LL * ((p.splits + 1) / 2) * ((cols + 7) / 8);
        const long long est_cl = best >= 2 ? 2LL * ((p.nkb + best - 1) / best) + 6 : 0;
        if (best >= 2 && (force_cluster || est_cl < est_ws) && !(ws_env && ws_env[0] == '1')) {
            p.csplit = true;
            p.splits = best;
            splits = best;
            p.n_items = p.n_full = p.grid = (int)(tiles * best);
        }
    }
    const double w_bytes = (double)N * (double)K * w_bits / 8.0;
    const double a_bytes = (double)M * (double)K * 2.0;
    p.walk_n_fast = w_bytes < a_bytes ? 1 : 0;
    // WQ_WALK=n (weight-row tiles fastest) or WQ_WALK=m (token tiles fastest) in the
    // environment overrides the rule, e.g. to measure both orders on one shape
    const char* walk_env = std::getenv("WQ_WALK");
    if (walk_env && walk_env[0] == 'n' && walk_env[1] == '\0') p.walk_n_fast = 1;
    if (walk_env && walk_env[0] == 'm' && walk_env[1] == '\0') p.walk_n_fast = 0;
    p.ws_bytes = (decode || p.csplit) ? 0 : split_ws_bytes((int)tiles, splits, cfg.bn);
    *plan = p;
    return WQ_OK;
}

int w_bits_of(int fmt) { return fmt == FMT_FP8 ? 8 : fmt == FMT_INT2 ? 2 : 4; }

wq_status plan_for(int fmt, bool bf16, int64_t M, int64_t N, int64_t K, Plan* plan, int G, int decode_kind) {
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    return make_plan(fmt, bf16, M, N, K, d->sms, w_bits_of(fmt), plan, G, decode_kind);
}

void fill_common(GemmParams& gp, const Plan& pl, int64_t M, int64_t N, int64_t K, void* out, void* ws,
                 uint32_t* status) {
    gp.out = out;
    gp.M = (int)M;
    gp.N = (int)N;
    gp.K = (int)K;
    gp.tiles_n = pl.tiles_n;
    gp.tiles_m = pl.tiles_m;
    gp.splits = pl.splits;
    gp.nkb = pl.nkb;
    gp.kb_base = pl.nkb / pl.splits;
    gp.kb_rem = pl.nkb % pl.splits;
    gp.n_items = pl.n_items;
    gp.n_full = pl.n_full;
    gp.half_bn = pl.cfg.bn / 2;
    gp.walk_n_fast = pl.walk_n_fast;
    gp.w_evict_first = pl.tiles_m == 1 ? 1 : 0;
    gp.div_walk = make_fastdiv(pl.walk_n_fast ? pl.tiles_n : pl.tiles_m,
                               (uint32_t)((long long)pl.tiles_n * pl.tiles_m));
    gp.div_splits = make_fastdiv(pl.splits, (uint32_t)pl.n_items);
    gp.csplit = pl.csplit ? 1 : 0;
    gp.status = status;
    gp.timeout_ns = kTimeoutNs;
    if (pl.ws_bytes > 0) {
        gp.ws_count = static_cast<uint32_t*>(ws);
        gp.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kSplitCounterBytes);
    }
}

wq_status check_ws(const Plan& pl, const void* ws, size_t ws_bytes) {
    if (pl.ws_bytes == 0) return WQ_OK;
    if (ws == nullptr || ws_bytes < pl.ws_bytes) return WQ_ERR_WORKSPACE;
    if (!aligned(ws, 16)) return WQ_ERR_MISALIGNED;
    return WQ_OK;
}

// Activation tensor map.  When one token tile covers all M rows, the box holds only
// those rows: the tile's remaining rows stay unwritten (they only reach accumulator
// columns that are never stored) and the copy engine does no out-of-range fill.
// A second map with boxes half as high serves the half tiles of the last round.
bool encode_a(GemmParams& gp, const void* A, bool bf16, int64_t M, int64_t K, int bn) {
    const auto dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int rows = M < bn ? (int)M : bn;
    const int half = M < bn / 2 ? (int)M : bn / 2;
    gp.a_box_rows = rows;
    gp.a_box_rows_half = half;
    return encode_2d(&gp.tmap_a, dt, A, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, (uint32_t)rows,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_2d(&gp.tmap_a_half, dt, A, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, (uint32_t)half,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output map of the pair kernel: out [M][N] 16-bit, boxes of 128 weight rows x 128
// tokens copied from the shared-memory staging area.  Needs N % 8 == 0 (16-byte
// row pitch).
bool encode_out(GemmParams& gp, void* out, bool bf16, int64_t M, int64_t N) {
    return encode_2d(&gp.tmap_out, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, out,
                     (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Activation tensor map of the decode kernel: A [M][K] viewed as {64 k, M rows,
// K / 64 boxes} (strides 2K and 128 bytes), so one copy brings a whole k-block of
// every token row, 64-wide boxes one after the other in shared memory (row
// z * M + m), each row 128 bytes with the 128-byte swizzle.  Needs K % 64 == 0.
bool encode_a_boxes(GemmParams& gp, const void* A, bool bf16, int64_t M, int64_t K, int bk) {
    auto fn = encode_fn();
    if (!fn || K % 64 != 0 || M > 32) return false;
    gp.a_box_rows = (int)M;
    cuuint64_t dims[3] = {64, (cuuint64_t)M, (cuuint64_t)(K / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)M, (cuuint32_t)(bk / 64)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(&gp.tmap_a, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(A), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

wq_status finish_launch(cudaError_t e) { return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA; }

const int64_t kMaxDim = (1LL << 31) - 1;

}  // namespace
}  // namespace wq

using namespace wq;

extern "C" {

const char* wq_status_string(wq_status s) {
    switch (s) {
        case WQ_OK: return "WQ_OK";
        case WQ_ERR_NULL: return "WQ_ERR_NULL: a required pointer is NULL";
        case WQ_ERR_SHAPE: return "WQ_ERR_SHAPE: unsupported problem shape";
        case WQ_ERR_GROUP: return "WQ_ERR_GROUP: group size must be 32, 64, 128 or 256 and divide K";
        case WQ_ERR_MISALIGNED: return "WQ_ERR_MISALIGNED: pointer misses its required alignment";
        case WQ_ERR_DTYPE: return "WQ_ERR_DTYPE: activation dtype not supported by this op";
        case WQ_ERR_WORKSPACE: return "WQ_ERR_WORKSPACE: workspace missing or too small";
        case WQ_ERR_UNSUPPORTED_DEVICE: return "WQ_ERR_UNSUPPORTED_DEVICE: requires compute capability 10.3";
        case WQ_ERR_CUDA: return "WQ_ERR_CUDA: CUDA runtime error";
        case WQ_ERR_TIMEOUT: return "WQ_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    }
    return "unknown wq_status";
}

wq_status wq_int4_packed_bytes(int64_t N, int64_t K, int32_t G, size_t* w_bytes, size_t* s_bytes) {
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim || K % 32 != 0) return WQ_ERR_SHAPE;
    if (!valid_group(G) || K % G != 0) return WQ_ERR_GROUP;
    const int64_t Np = round_up(N, TILE_N), Kp = round_up(K, KPAD_INT4);
    if (w_bytes) *w_bytes = (size_t)(Np * Kp / 2);
    if (s_bytes) *s_bytes = (size_t)(Np * (Kp / G) * 2);
    return WQ_OK;
}

static wq_status check_pack_args(const void* a, const void* b, const void* c, const void* d, int64_t N, int64_t K,
                                 int32_t G) {
    if (!a || !b || !c || !d) return WQ_ERR_NULL;
    return wq_int4_packed_bytes(N, K, G, nullptr, nullptr);
}

wq_status wq_pack_int4(const uint8_t* w_canon, const void* s_canon, int64_t N, int64_t K, int32_t G,
                       uint8_t* w_kernel, void* s_kernel, wq_stream_t stream) {
    wq_status st = check_pack_args(w_canon, s_canon, w_kernel, s_kernel, N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(w_kernel, 16) || !aligned(s_kernel, 16) || !aligned(s_canon, 2)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_pack_int4(w_canon, static_cast<const uint16_t*>(s_canon), N, K, G, w_kernel,
                                          static_cast<uint16_t*>(s_kernel), (cudaStream_t)stream));
}

wq_status wq_int4_packed_zeros_bytes(int64_t N, int64_t K, int32_t G, size_t* z_bytes) {
    size_t s_bytes = 0;
    const wq_status st = wq_int4_packed_bytes(N, K, G, nullptr, &s_bytes);
    if (st == WQ_OK && z_bytes) *z_bytes = s_bytes / 2;   // one byte per (group, row) instead of two
    return st;
}

wq_status wq_pack_int4_zeros(const uint8_t* z_canon, int64_t N, int64_t K, int32_t G, uint8_t* z_kernel,
                             wq_stream_t stream) {
    wq_status st = check_pack_args(z_canon, z_kernel, z_canon, z_kernel, N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(z_kernel, 16)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_pack_int4_zeros(z_canon, N, K, G, z_kernel, (cudaStream_t)stream));
}

wq_status wq_quantize_int4(const void* w, int64_t N, int64_t K, int32_t G, uint8_t* w_canon, void* s_canon,
                           wq_stream_t stream) {
    if (!w || !w_canon || !s_canon) return WQ_ERR_NULL;
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim || K % 32 != 0) return WQ_ERR_SHAPE;
    if (!valid_group(G) || K % G != 0) return WQ_ERR_GROUP;
    if (!aligned(w, 16) || !aligned(w_canon, 4) || !aligned(s_canon, 2)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    return finish_launch(launch_quantize_int4(static_cast<const uint16_t*>(w), N, K, G, w_canon,
                                              static_cast<uint16_t*>(s_canon), (cudaStream_t)stream));
}

wq_status wq_unpack_int4(const uint8_t* w_kernel, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                         uint8_t* w_canon, void* s_canon, wq_stream_t stream) {
    wq_status st = check_pack_args(w_kernel, s_kernel, w_canon, s_canon, N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(w_kernel, 16) || !aligned(s_kernel, 16) || !aligned(s_canon, 2)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_unpack_int4(w_kernel, static_cast<const uint16_t*>(s_kernel), N, K, G, w_canon,
                                            static_cast<uint16_t*>(s_canon), (cudaStream_t)stream));
}

wq_status wq_debug_dequant_int4(const uint8_t* w_kernel, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                                float* w_f32, wq_stream_t stream) {
    wq_status st = check_pack_args(w_kernel, s_kernel, w_f32, w_f32, N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(w_kernel, 16) || !aligned(s_kernel, 16) || !aligned(w_f32, 4)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_dequant_int4(w_kernel, static_cast<const uint16_t*>(s_kernel), nullptr, N, K, G,
                                             w_f32, (cudaStream_t)stream));
}

wq_status wq_debug_dequant_int4_lut(const uint8_t* w_kernel, const void* s_kernel, const void* lut, int64_t N,
                                    int64_t K, int32_t G, float* w_f32, wq_stream_t stream) {
    if (!lut) return WQ_ERR_NULL;
    wq_status st = check_pack_args(w_kernel, s_kernel, w_f32, w_f32, N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(w_kernel, 16) || !aligned(s_kernel, 16) || !aligned(w_f32, 4) || !aligned(lut, 2))
        return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_dequant_int4(w_kernel, static_cast<const uint16_t*>(s_kernel),
                                             static_cast<const uint16_t*>(lut), N, K, G, w_f32,
                                             (cudaStream_t)stream));
}

wq_status wq_fp4_packed_sf_bytes(int64_t N, int64_t K, size_t* sf_bytes) {
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim || K % 32 != 0) return WQ_ERR_SHAPE;
    if (sf_bytes) *sf_bytes = (size_t)(round_up(N, TILE_N) * (round_up(K, KPAD_FP4SF) / 64) * 4);
    return WQ_OK;
}

wq_status wq_pack_fp4_sf(const uint8_t* sf_canon, int64_t N, int64_t K, uint8_t* sf_kernel, wq_stream_t stream) {
    if (!sf_canon || !sf_kernel) return WQ_ERR_NULL;
    wq_status st = wq_fp4_packed_sf_bytes(N, K, nullptr);
    if (st != WQ_OK) return st;
    if (!aligned(sf_kernel, 16)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_pack_fp4_sf(sf_canon, N, K, sf_kernel, (cudaStream_t)stream));
}

wq_status wq_debug_dequant_fp4(const uint8_t* w_e2m1, const uint8_t* sf_kernel, int64_t N, int64_t K, float* w_f32,
                               wq_stream_t stream) {
    if (!w_e2m1 || !sf_kernel || !w_f32) return WQ_ERR_NULL;
    wq_status st = wq_fp4_packed_sf_bytes(N, K, nullptr);
    if (st != WQ_OK) return st;
    if (!aligned(sf_kernel, 16) || !aligned(w_f32, 4)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_dequant_fp4(w_e2m1, sf_kernel, N, K, w_f32, (cudaStream_t)stream));
}

wq_status wq_debug_dequant_fp8(const uint8_t* w_e4m3, int64_t N, int64_t K, wq_dtype operand, float* w_f32,
                               wq_stream_t stream) {
    if (!w_e4m3 || !w_f32) return WQ_ERR_NULL;
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim || K % 16 != 0) return WQ_ERR_SHAPE;
    if (operand != WQ_F16 && operand != WQ_BF16) return WQ_ERR_DTYPE;
    if (!aligned(w_f32, 4)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    return finish_launch(launch_dequant_fp8(w_e4m3, N, K, operand == WQ_BF16, w_f32, (cudaStream_t)stream));
}

wq_status wq_get_plan(wq_op op, wq_dtype a_dtype, int64_t M, int64_t N, int64_t K, int32_t G, wq_plan* plan,
                      size_t* ws_bytes) {
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return WQ_ERR_SHAPE;
    int fmt = -1;
    switch (op) {
        case WQ_OP_W4A16: case WQ_OP_W4A16_ZP: fmt = FMT_INT4; break;
        case WQ_OP_FP8: fmt = FMT_FP8; break;
        case WQ_OP_FP4: fmt = FMT_FP4; break;
        case WQ_OP_W4A16_LUT: fmt = FMT_LUT4; break;
        case WQ_OP_W2A16: fmt = FMT_INT2; break;
    }
    if (fmt < 0) return WQ_ERR_SHAPE;
    const bool grouped = group_scaled(fmt);
    if (grouped && (!valid_group(G) || K % G != 0)) return WQ_ERR_GROUP;
    if (a_dtype != WQ_F16 && a_dtype != WQ_BF16) return WQ_ERR_DTYPE;
    const bool bf16 = (op == WQ_OP_FP4) ? true : (a_dtype == WQ_BF16);
    Plan pl{};
    // the decode kind the GEMM entry points pass (0 for every format but zero-point
    // INT4; make_plan picks the decode kernel by format)
    wq_status st = plan_for(fmt, bf16, M > 0 ? M : 1, N, K, &pl, grouped ? G : 0, op == WQ_OP_W4A16_ZP ? 1 : 0);
    if (st != WQ_OK) return st;
    if (plan) {
        plan->bn = pl.cfg.bn;
        plan->bk = pl.cfg.bk;
        plan->stages = pl.cfg.stages;
        plan->splits = pl.splits;
        plan->grid = pl.grid;
        plan->threads = pl.cfg.threads;
        plan->smem_bytes = pl.cfg.smem_bytes;
        plan->n_items = pl.n_items;
        plan->walk_n_fast = pl.walk_n_fast;
        plan->tiles_n = pl.tiles_n;
        plan->tiles_m = pl.tiles_m;
        plan->ctas_per_sm = pl.cfg.ctas_per_sm;
        plan->kernel = pl.decode ? WQ_KERNEL_DECODE : pl.pair ? WQ_KERNEL_TILE_PAIR : WQ_KERNEL_TILE;
        plan->cluster_split = pl.csplit ? 1 : 0;
        plan->cluster_capacity =
            (pl.splits >= 2 && pl.splits <= kMaxDecodeCluster && !pl.pair) ? pl.cfg.max_clusters[pl.splits] : 0;
    }
    if (ws_bytes) *ws_bytes = (M == 0) ? 0 : pl.ws_bytes;
    return WQ_OK;
}

wq_status wq_workspace_bytes(wq_op op, wq_dtype a_dtype, int64_t M, int64_t N, int64_t K, int32_t G, size_t* bytes) {
    if (!bytes) return WQ_ERR_NULL;
    return wq_get_plan(op, a_dtype, M, N, K, G, nullptr, bytes);
}

// W4A16 with the symmetric zero point 8 (z_kernel and lut null), packed zero points,
// or a 16-entry codebook.  M <= 16 with K % 64 == 0 runs on the register decode kernel
// (the codebook with fp16 activations only).
static wq_status gemm_int4(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                           const uint8_t* z_kernel, const uint16_t* lut, int64_t M, int64_t N, int64_t K, int32_t G,
                           void* out, void* ws, size_t ws_bytes, wq_stream_t stream) {
    const int fmt = lut ? FMT_LUT4 : FMT_INT4;
    if (M == 0 && N > 0 && K > 0) return WQ_OK;   // empty problem: A and out may be NULL
    if (!A || !w_kernel || !s_kernel || !out) return WQ_ERR_NULL;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return WQ_ERR_SHAPE;
    if (K % 32 != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
    if (!valid_group(G) || K % G != 0) return WQ_ERR_GROUP;
    if (a_dtype != WQ_F16 && a_dtype != WQ_BF16) return WQ_ERR_DTYPE;
    if (!aligned(A, 16) || !aligned(w_kernel, 16) || !aligned(s_kernel, 16) || !aligned(out, 16) ||
        !aligned(z_kernel, 16) || !aligned(lut, 16))
        return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    if (M == 0) return WQ_OK;
    const bool bf16 = a_dtype == WQ_BF16;
    Plan pl{};
    if ((st = make_plan(fmt, bf16, M, N, K, d->sms, 4, &pl, G, z_kernel ? 1 : 0)) != WQ_OK) return st;
    if ((st = check_ws(pl, ws, ws_bytes)) != WQ_OK) return st;
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    // pair kernel: each CTA copies half of the 256-token tile
    if (pl.decode ? !encode_a_boxes(gp, A, bf16, M, K, pl.cfg.bk)
                  : !encode_a(gp, A, bf16, M, K, pl.pair ? pl.cfg.bn / 2 : pl.cfg.bn))
        return WQ_ERR_CUDA;
    if (pl.pair && !encode_out(gp, out, bf16, M, N)) return WQ_ERR_CUDA;
    gp.w = w_kernel;
    gp.sc = static_cast<const uint8_t*>(s_kernel);
    gp.zp = z_kernel;
    gp.lut = lut;
    gp.G = G;
    gp.g_shift = G == 32 ? 5 : G == 64 ? 6 : G == 128 ? 7 : 8;
    const int64_t Kp = round_up(K, KPAD_INT4);
    gp.ngroups_pad = (int)(Kp / G);
    gp.nchunks_pad = (int)(Kp / 32);
    fill_common(gp, pl, M, N, K, out, ws, d->status);
    if (pl.decode)
        return finish_launch(z_kernel ? launch_gemm_int4_decode_zp(gp, bf16, pl.grid, (cudaStream_t)stream)
                             : lut    ? launch_gemm_int4_decode_lut(gp, pl.grid, (cudaStream_t)stream)
                                      : launch_gemm_int4_decode(gp, bf16, pl.grid, (cudaStream_t)stream));
    if (fmt == FMT_LUT4)
        return finish_launch(pl.pair ? launch_gemm_lut4_pair(gp, bf16, pl.grid, (cudaStream_t)stream)
                                     : launch_gemm_lut4(gp, bf16, pl.cfg.bn, pl.grid, (cudaStream_t)stream));
    if (pl.pair) return finish_launch(launch_gemm_int4_pair(gp, bf16, pl.grid, (cudaStream_t)stream));
    return finish_launch(launch_gemm_int4(gp, bf16, pl.cfg.bn, pl.grid, (cudaStream_t)stream));
}

wq_status wq_gemm_w4a16(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel, int64_t M,
                        int64_t N, int64_t K, int32_t G, void* out, void* ws, size_t ws_bytes, wq_stream_t stream) {
    return gemm_int4(A, a_dtype, w_kernel, s_kernel, nullptr, nullptr, M, N, K, G, out, ws, ws_bytes, stream);
}

wq_status wq_gemm_w4a16_zp(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                           const uint8_t* z_kernel, int64_t M, int64_t N, int64_t K, int32_t G, void* out, void* ws,
                           size_t ws_bytes, wq_stream_t stream) {
    if (M == 0 && N > 0 && K > 0) return WQ_OK;
    if (!z_kernel) return WQ_ERR_NULL;
    return gemm_int4(A, a_dtype, w_kernel, s_kernel, z_kernel, nullptr, M, N, K, G, out, ws, ws_bytes, stream);
}

wq_status wq_gemm_w4a16_lut(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel, const void* s_kernel,
                            const void* lut, int64_t M, int64_t N, int64_t K, int32_t G, void* out, void* ws,
                            size_t ws_bytes, wq_stream_t stream) {
    if (M == 0 && N > 0 && K > 0) return WQ_OK;
    if (!lut) return WQ_ERR_NULL;
    return gemm_int4(A, a_dtype, w_kernel, s_kernel, nullptr, static_cast<const uint16_t*>(lut), M, N, K, G, out,
                     ws, ws_bytes, stream);
}

// ------------------------------------------------------------------ INT2

static wq_status check_int2_shape(int64_t N, int64_t K, int32_t G) {
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim || K % 64 != 0) return WQ_ERR_SHAPE;
    if (!valid_group(G) || K % G != 0) return WQ_ERR_GROUP;
    return WQ_OK;
}

wq_status wq_int2_packed_scales_bytes(int64_t N, int64_t K, int32_t G, size_t* s_bytes) {
    wq_status st = check_int2_shape(N, K, G);
    if (st != WQ_OK) return st;
    if (s_bytes) *s_bytes = (size_t)(round_up(N, TILE_N) * (round_up(K, KPAD_INT4) / G) * 2);
    return WQ_OK;
}

wq_status wq_pack_int2_scales(const void* s_canon, int64_t N, int64_t K, int32_t G, void* s_kernel,
                              wq_stream_t stream) {
    if (!s_canon || !s_kernel) return WQ_ERR_NULL;
    wq_status st = check_int2_shape(N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(s_canon, 2) || !aligned(s_kernel, 16)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_pack_group_scales(static_cast<const uint16_t*>(s_canon), N, K, G,
                                                  static_cast<uint16_t*>(s_kernel), (cudaStream_t)stream));
}

wq_status wq_debug_dequant_int2(const uint8_t* w_canon, const void* s_kernel, int64_t N, int64_t K, int32_t G,
                                float* w_f32, wq_stream_t stream) {
    if (!w_canon || !s_kernel || !w_f32) return WQ_ERR_NULL;
    wq_status st = check_int2_shape(N, K, G);
    if (st != WQ_OK) return st;
    if (!aligned(s_kernel, 16) || !aligned(w_f32, 4)) return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    return finish_launch(launch_dequant_int2(w_canon, static_cast<const uint16_t*>(s_kernel), N, K, G, w_f32,
                                             (cudaStream_t)stream));
}

wq_status wq_gemm_w2a16(const void* A, wq_dtype a_dtype, const uint8_t* w_canon, const void* s_kernel, int64_t M,
                        int64_t N, int64_t K, int32_t G, void* out, void* ws, size_t ws_bytes, wq_stream_t stream) {
    if (M == 0 && N > 0 && K > 0) return WQ_OK;   // empty problem: A and out may be NULL
    if (!A || !w_canon || !s_kernel || !out) return WQ_ERR_NULL;
    if (M < 0 || M > kMaxDim || N % 8 != 0) return WQ_ERR_SHAPE;
    wq_status st = check_int2_shape(N, K, G);
    if (st != WQ_OK) return st;
    if (a_dtype != WQ_F16 && a_dtype != WQ_BF16) return WQ_ERR_DTYPE;
    if (!aligned(A, 16) || !aligned(w_canon, 16) || !aligned(s_kernel, 16) || !aligned(out, 16))
        return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    if ((st = device_info(&d)) != WQ_OK) return st;
    const bool bf16 = a_dtype == WQ_BF16;
    Plan pl{};
    if ((st = make_plan(FMT_INT2, bf16, M, N, K, d->sms, 2, &pl, G)) != WQ_OK) return st;
    if ((st = check_ws(pl, ws, ws_bytes)) != WQ_OK) return st;
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (pl.decode ? !encode_a_boxes(gp, A, bf16, M, K, pl.cfg.bk)
                  : !encode_a(gp, A, bf16, M, K, pl.pair ? pl.cfg.bn / 2 : pl.cfg.bn))
        return WQ_ERR_CUDA;
    if (pl.pair && !encode_out(gp, out, bf16, M, N)) return WQ_ERR_CUDA;
    const int pitch = pl.cfg.bk / 4;   // bytes of one row's codes per k-block (decode: 64, a 256-code stage)
    if (!encode_2d(&gp.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_canon, (uint64_t)(K / 4), (uint64_t)N,
                   (uint64_t)(K / 4), (uint32_t)pitch, TILE_N, swizzle_for_pitch(pitch)))
        return WQ_ERR_CUDA;
    gp.sc = static_cast<const uint8_t*>(s_kernel);
    gp.G = G;
    gp.g_shift = G == 32 ? 5 : G == 64 ? 6 : G == 128 ? 7 : 8;
    gp.ngroups_pad = (int)(round_up(K, KPAD_INT4) / G);
    fill_common(gp, pl, M, N, K, out, ws, d->status);
    if (pl.decode) return finish_launch(launch_gemm_int2_decode(gp, bf16, pl.grid, (cudaStream_t)stream));
    if (pl.pair) return finish_launch(launch_gemm_int2_pair(gp, bf16, pl.grid, (cudaStream_t)stream));
    return finish_launch(launch_gemm_int2(gp, bf16, pl.cfg.bn, pl.grid, (cudaStream_t)stream));
}

wq_status wq_gemm_w8a16_fp8(const void* A, wq_dtype a_dtype, const uint8_t* w_e4m3, const float* alpha,
                            const void* bias, int64_t M, int64_t N, int64_t K, void* out, void* ws, size_t ws_bytes,
                            wq_stream_t stream) {
    if (M == 0 && N > 0 && K > 0) return WQ_OK;   // empty problem: A and out may be NULL
    if (!A || !w_e4m3 || !alpha || !out) return WQ_ERR_NULL;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return WQ_ERR_SHAPE;
    if (K % 16 != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
    if (a_dtype != WQ_F16 && a_dtype != WQ_BF16) return WQ_ERR_DTYPE;
    if (!aligned(A, 16) || !aligned(w_e4m3, 16) || !aligned(out, 16) || !aligned(alpha, 4) ||
        (bias && !aligned(bias, 2)))
        return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    if (M == 0) return WQ_OK;
    const bool bf16 = a_dtype == WQ_BF16;
    Plan pl{};
    if ((st = make_plan(FMT_FP8, bf16, M, N, K, d->sms, 8, &pl)) != WQ_OK) return st;
    if ((st = check_ws(pl, ws, ws_bytes)) != WQ_OK) return st;
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (pl.decode ? !encode_a_boxes(gp, A, bf16, M, K, pl.cfg.bk)
                  : !encode_a(gp, A, bf16, M, K, pl.pair ? pl.cfg.bn / 2 : pl.cfg.bn))
        return WQ_ERR_CUDA;
    if (pl.pair && !encode_out(gp, out, bf16, M, N)) return WQ_ERR_CUDA;
    const int bk = pl.cfg.bk;
    if (!encode_2d(&gp.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_e4m3, (uint64_t)K, (uint64_t)N, (uint64_t)K,
                   (uint32_t)bk, TILE_N, swizzle_for_pitch(bk)))
        return WQ_ERR_CUDA;
    gp.alpha = alpha;
    gp.bias = bias;
    fill_common(gp, pl, M, N, K, out, ws, d->status);
    if (pl.decode) return finish_launch(launch_gemm_fp8_decode(gp, bf16, pl.grid, (cudaStream_t)stream));
    if (pl.pair) return finish_launch(launch_gemm_fp8_pair(gp, bf16, pl.grid, (cudaStream_t)stream));
    return finish_launch(launch_gemm_fp8(gp, bf16, pl.cfg.bn, pl.grid, (cudaStream_t)stream));
}

wq_status wq_gemm_bf16_fp4(const void* A, const uint8_t* w_e2m1, const uint8_t* sf_kernel, const float* alpha,
                           int64_t M, int64_t N, int64_t K, void* out, void* ws, size_t ws_bytes,
                           wq_stream_t stream) {
    if (M == 0 && N > 0 && K > 0) return WQ_OK;   // empty problem: A and out may be NULL
    if (!A || !w_e2m1 || !sf_kernel || !alpha || !out) return WQ_ERR_NULL;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return WQ_ERR_SHAPE;
    if (K % 32 != 0 || N % 8 != 0) return WQ_ERR_SHAPE;
    if (!aligned(A, 16) || !aligned(w_e2m1, 16) || !aligned(sf_kernel, 16) || !aligned(out, 16) ||
        !aligned(alpha, 4))
        return WQ_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    if (M == 0) return WQ_OK;
    Plan pl{};
    if ((st = make_plan(FMT_FP4, true, M, N, K, d->sms, 4, &pl)) != WQ_OK) return st;
    if ((st = check_ws(pl, ws, ws_bytes)) != WQ_OK) return st;
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (pl.decode ? !encode_a_boxes(gp, A, true, M, K, pl.cfg.bk)
                  : !encode_a(gp, A, true, M, K, pl.pair ? pl.cfg.bn / 2 : pl.cfg.bn))
        return WQ_ERR_CUDA;
    if (pl.pair && !encode_out(gp, out, true, M, N)) return WQ_ERR_CUDA;
    const int pitch = pl.cfg.bk / 2;
    if (!encode_2d(&gp.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_e2m1, (uint64_t)(K / 2), (uint64_t)N,
                   (uint64_t)(K / 2), (uint32_t)pitch, TILE_N, swizzle_for_pitch(pitch)))
        return WQ_ERR_CUDA;
    gp.sc = sf_kernel;
    gp.alpha = alpha;
    gp.nchunks_pad = (int)(round_up(K, KPAD_FP4SF) / 64);
    fill_common(gp, pl, M, N, K, out, ws, d->status);
    if (pl.decode) return finish_launch(launch_gemm_fp4_decode(gp, pl.grid, (cudaStream_t)stream));
    if (pl.pair) return finish_launch(launch_gemm_fp4_pair(gp, pl.grid, (cudaStream_t)stream));
    return finish_launch(launch_gemm_fp4(gp, true, pl.cfg.bn, pl.grid, (cudaStream_t)stream));
}

wq_status wq_debug_fastdiv(uint32_t d, uint32_t x_max, const uint32_t* x, int64_t n, uint32_t* q,
                           int32_t* uses_multiply) {
    if (!uses_multiply || (n > 0 && (!x || !q))) return WQ_ERR_NULL;
    if (d == 0 || n < 0) return WQ_ERR_SHAPE;
    for (int64_t i = 0; i < n; ++i)
        if (x[i] > x_max) return WQ_ERR_SHAPE;
    const FastDiv f = make_fastdiv(d, x_max);
    *uses_multiply = f.magic != 0 ? 1 : 0;
    for (int64_t i = 0; i < n; ++i) q[i] = fastdiv(x[i], f);
    return WQ_OK;
}

wq_status wq_device_status(uint32_t* bits) {
    if (!bits) return WQ_ERR_NULL;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    if (cudaMemcpy(bits, d->status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return WQ_ERR_CUDA;
    return *bits ? WQ_ERR_TIMEOUT : WQ_OK;
}

wq_status wq_clear_device_status(void) {
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    return cudaMemset(d->status, 0, sizeof(uint32_t)) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess
               ? WQ_OK
               : WQ_ERR_CUDA;
}

wq_status wq_debug_wait_probe(int64_t timeout_ns, wq_stream_t stream) {
    if (timeout_ns <= 0 || timeout_ns > 10000000000LL) return WQ_ERR_SHAPE;
    DeviceInfo* d = nullptr;
    wq_status st = device_info(&d);
    if (st != WQ_OK) return st;
    return finish_launch(launch_wait_probe(d->status, (long long)timeout_ns, (cudaStream_t)stream));
}

}  // extern "C"
