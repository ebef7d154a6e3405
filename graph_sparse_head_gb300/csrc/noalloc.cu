// pmha_forward_noalloc: the forward pass with its scratch memory in a
// fixed-size array that lives inside this library, for callers that must not
// allocate device memory when they call the layer.
//
// Some callers cannot allocate: hosts whose allocator owns all device memory
// and hands out no raw buffers, and call sites where a cudaMalloc / cudaFree
// (which may synchronize the device) is not allowed. They pass only inputs
// and outputs; the workspace that pmha_forward needs is carved from
// g_scratch below instead of being supplied by the caller.
//
// g_scratch is a file-scope __device__ array: every GPU that loads this code
// holds PMHA_NOALLOC_SCRATCH_BYTES of device memory for it until the process
// exits. In host code its name only stands in for the symbol and is not a
// device address, so the device address is looked up with
// cudaGetSymbolAddress on the first call made with a device (and context)
// current, and cached for that device and context. Make that first call
// before any stream capture. With CUDA's lazy module loading (the default),
// the code of this file, and with it the array, is loaded onto a device at
// that first lookup: the first call on each device reserves the array and can
// fail for want of device memory, so make it before an allocator claims the
// device's memory. The cache does not survive cudaDeviceReset: a device that
// was reset in this process must not be used with this entry point again.
//
// Every call shares the one array. Calls whose work overlaps on the GPU (on
// different streams, or from different threads without ordering) race on it;
// calls on one stream run in order and are safe. The forward pass writes
// every workspace byte it later reads, so nothing needs clearing between
// calls, although the array keeps the previous call's contents.
#include <cuda.h>

#include <mutex>

#include "pmha_internal.h"

namespace {

__device__ __align__(256) unsigned char g_scratch[PMHA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};  // the context the address was looked up in

// The current driver context (the address of a __device__ array belongs to
// the context that loaded the module), or null when it cannot be read.
CUcontext current_context()
{
    typedef CUresult (*GetCurrent)(CUcontext *);
    static GetCurrent fn = []() -> GetCurrent {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return (GetCurrent)p;
    }();
    CUcontext c = nullptr;
    if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
}

}  // namespace

extern "C" pmha_status pmha_forward_noalloc(const pmha_graph *graph, const pmha_params *params, const void *query,
                                            const void *key, const void *value,
                                            const uint8_t *key_padding_mask, int64_t batch, void *output,
                                            pmha_wmode wmode, float *weights, pmha_stream stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pmha::cuda_fail(e, "pmha_forward_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        pmha::set_error("pmha_forward_noalloc: device %d is beyond the %d devices this entry point serves", dev,
                        kMaxDevices);
        return PMHA_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const CUcontext ctx = current_context();
        if (!g_scratch_addr[dev] || ctx != g_scratch_ctx[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_scratch);
            if (e != cudaSuccess) {
                pmha::set_error("pmha_forward_noalloc: could not reserve the %zu-byte scratch array on device %d "
                                "(%s): the first call on a device loads it; make that call before other "
                                "allocations claim the device's memory",
                                (size_t)PMHA_NOALLOC_SCRATCH_BYTES, dev, cudaGetErrorString(e));
                return PMHA_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_addr[dev];
    }
    const size_t need = pmha_forward_workspace_size(graph, params, batch, wmode);
    // need == 0: invalid arguments; pmha_forward reports which, before any launch
    if (need > (size_t)PMHA_NOALLOC_SCRATCH_BYTES) {
        pmha::set_error("pmha_forward_noalloc: this problem needs %zu bytes of scratch, more than the %zu bytes "
                        "built into the library; use pmha_forward with a caller workspace",
                        need, (size_t)PMHA_NOALLOC_SCRATCH_BYTES);
        return PMHA_ERR_WORKSPACE;
    }
    return pmha_forward(graph, params, query, key, value, key_padding_mask, batch, output, wmode, weights, scratch,
                        (size_t)PMHA_NOALLOC_SCRATCH_BYTES, stream);
}
