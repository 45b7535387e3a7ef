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
// per device, on that device, and passed to the kernels.  The address belongs
// to the context it was looked up in: it is cached together with that
// context's unique id, and looked up again when the device's current context
// is a different one (after cudaDeviceReset, or a context the caller made),
// so a stale address is never handed to a kernel.  All calls share the array:
// the sort clears the parts that must start at zero on every call, and calls
// that overlap on the GPU (e.g. on two streams at once) race.
#include <cuda.h>
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
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context g_scratch_ptr belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The driver's context queries, resolved once through the runtime (no link
// dependency on the driver library).  Caller holds g_mu.
bool resolve_context_queries()
{
    if (g_ctx_get_current && g_ctx_get_id) return true;
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa = cudaDriverEntryPointSymbolNotFound, qb = qa;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b)
        return false;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
    return true;
}

// Unique id of this thread's current context, or 0 if there is none yet.
// Caller holds g_mu and has resolved the queries.
unsigned long long current_context_id()
{
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current device's current
// context: looked up (cudaGetSymbolAddress, which also makes the context
// current if the runtime has not yet) on the first call on a device, and
// again whenever that device's current context is not the one the cached
// address was looked up in.
rs_status scratch_on_current_device(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!resolve_context_queries()) return RS_ERR_CUDA;
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RS_ERR_CUDA;
        const unsigned long long now = current_context_id();
        if (now == 0) return RS_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = now;
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
