// rs_static.cu -- rs_sort_keys_u32_noalloc: the uint32 keys-only sort with its
// scratch in a fixed device array instead of a caller-provided temp buffer.
//
// Who needs this: callers that cannot allocate device memory at the point
// where they sort -- for example code running while a stream capture in
// global mode is active (cudaMalloc is not permitted then), plugins hosted by
// an application that owns the device memory pool and forbids allocations
// behind its back, and latency-critical loops where cudaMalloc/cudaFree would
// synchronise the device.  They still pass their own input and output.
//
// The scratch is one file-scope __device__ array of RS_NOALLOC_SCRATCH_BYTES,
// sized for RS_NOALLOC_MAX_N keys; every GPU that loads this code holds it
// until the process exits.  In host code the array's name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress once
// per device, on that device, and passed to the kernels.  All calls share the
// array: the sort clears the parts that must start at zero on every call, and
// calls that overlap on the GPU (e.g. on two streams at once) race.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "rs.h"
#include "rs_config.h"

namespace {

constexpr size_t kScratchBytes = rs::temp_layout(4, 0, RS_NOALLOC_MAX_N, 0, 32).total;
static_assert(kScratchBytes <= RS_NOALLOC_SCRATCH_BYTES, "scratch size in rs.h is too small");

static __device__ __align__(256) unsigned char g_noalloc_scratch[RS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device; the first call on a device performs the lookup).
rs_status scratch_on_current_device(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RS_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return RS_OK;
}

}  // namespace

extern "C" rs_status rs_sort_keys_u32_noalloc(const uint32_t* keys_in, uint32_t* keys_out, size_t n,
                                              int begin_bit, int end_bit, void* stream)
{
    if (n > (size_t)RS_NOALLOC_MAX_N) return RS_ERR_INVALID_ARG;
    if (n == 0) return rs_sort_keys_u32(keys_in, keys_out, 0, begin_bit, end_bit, nullptr, 0, stream);
    void* scratch = nullptr;
    rs_status st = scratch_on_current_device(&scratch);
    if (st != RS_OK) return st;
    return rs_sort_keys_u32(keys_in, keys_out, n, begin_bit, end_bit, scratch,
                            (size_t)RS_NOALLOC_SCRATCH_BYTES, stream);
}
