// wq_noalloc.cu -- wq_gemm_w4a16_noalloc: the W4A16 GEMM without a caller workspace.
//
// Some callers cannot allocate device memory: a serving framework that hands every
// byte of the GPU to its own pool at start-up, or a decode loop in which a
// cudaMalloc (which may synchronise the whole device) is not allowed.  For them the
// split-K scratch of the W4A16 GEMM lives in a fixed array inside this library.
//
// The array is a file-scope __device__ variable: every GPU that loads the library
// holds WQ_NOALLOC_SCRATCH_BYTES of it until the process exits.  In host code its
// name only stands in for the symbol -- it is not a device address -- so the device
// address is looked up once per device with cudaGetSymbolAddress (with that device
// current) and that pointer is what the kernel gets.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/wq.h"
#include "wq_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[WQ_NOALLOC_SCRATCH_BYTES];

// The start of any split-K workspace holds the arrival counters, which must read
// zero when a call starts (see wq_gemm_w4a16 in include/wq.h).
constexpr size_t kCounterBytes = wq::kSplitCounterBytes;
static_assert(kCounterBytes <= (size_t)WQ_NOALLOC_SCRATCH_BYTES, "counters fit in the scratch array");
constexpr int kMaxDevices = 64;

struct ScratchSlot {
    std::mutex mu;
    void* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch array on the current device.  Looked up on first use
// and kept only once the lookup succeeds: a lookup that fails (for instance one made
// while the stream is being captured) is tried again on the next call.
wq_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WQ_ERR_UNSUPPORTED_DEVICE;
    ScratchSlot& s = g_slots[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.ptr == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();   // leave no sticky error behind for the caller
            return WQ_ERR_CUDA;
        }
        s.ptr = p;
    }
    *out = s.ptr;
    return WQ_OK;
}

}  // namespace

extern "C" wq_status wq_gemm_w4a16_noalloc(const void* A, wq_dtype a_dtype, const uint8_t* w_kernel,
                                           const void* s_kernel, int64_t M, int64_t N, int64_t K, int32_t G,
                                           void* out, wq_stream_t stream) {
    size_t need = 0;
    wq_status st = wq_workspace_bytes(WQ_OP_W4A16, a_dtype, M, N, K, G, &need);
    if (st != WQ_OK) return st;
    if (need > (size_t)WQ_NOALLOC_SCRATCH_BYTES) return WQ_ERR_WORKSPACE;
    if (need == 0) return wq_gemm_w4a16(A, a_dtype, w_kernel, s_kernel, M, N, K, G, out, nullptr, 0, stream);
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != WQ_OK) return st;
    // every call shares the array: clear the counters on the caller's stream first
    if (cudaMemsetAsync(scratch, 0, kCounterBytes, (cudaStream_t)stream) != cudaSuccess) return WQ_ERR_CUDA;
    return wq_gemm_w4a16(A, a_dtype, w_kernel, s_kernel, M, N, K, G, out, scratch, (size_t)WQ_NOALLOC_SCRATCH_BYTES,
                         stream);
}
