// permute_noalloc.cu -- moe_permute for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they route
// tokens: code that runs while another component owns every allocation (a fixed
// memory plan reserved up front), code in a region where cudaMalloc's implicit
// device synchronization is not allowed, or a host runtime with no allocator
// handle at all.  For them, moe_permute_noalloc keeps the permutation's scratch
// in a fixed array that lives in the library's device image, so the caller only
// supplies inputs and outputs.
//
// The array is allocated by the CUDA module loader when this file's device code is
// loaded on a device (with lazy loading: at its first use there, which may allocate and
// synchronize -- hence "make the first call during set-up"), and every device that loads
// the library keeps its own copy until the process exits.  The per-device address cache
// below belongs to that device's context; a cudaDeviceReset in the process invalidates
// it.  All calls share the array: two calls whose kernels overlap on the GPU (different
// streams, or different host threads without ordering) race on it.  Nothing in it needs
// clearing between calls: the histogram kernel overwrites every count it later reads and
// the scan kernel every base.
#include <cuda_runtime.h>

#include <mutex>

#include "mxmoe_internal.h"

namespace {

// 1 MiB: two int32 tables of ceil(T*k / 2048) x E entries each.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per
// device.  In host code `g_permute_scratch` only names a host-side stand-in, so the
// real device address has to come from cudaGetSymbolAddress.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MX_OK;
}

}  // namespace

extern "C" {

int moe_permute_noalloc(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* counts, int32_t* off,
                        int32_t* poff, int32_t* src_row, int32_t* dst_of, const uint8_t* q_in,
                        const uint8_t* sf_in, int64_t K, uint8_t* q_out, uint8_t* sf_out, int* dev_err,
                        mx_stream_t stream) {
    if (T < 0 || k < 1 || k > 64 || E < 1 || E > 1024) return MX_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (mx::permute_workspace_bytes(T, k, E) > kNoAllocScratchBytes) return MX_ERR_TOO_LARGE;
    void* scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != MX_OK) return st;
    return moe_permute(topk_ids, T, k, E, counts, off, poff, src_row, dst_of, q_in, sf_in, K, q_out, sf_out, scratch,
                       kNoAllocScratchBytes, dev_err, stream);
}

}  // extern "C"
