// noalloc.cu -- one refresh layer that allocates nothing and takes no
// workspace from its caller.
//
// Why: kvr_refresh_layer needs a device workspace for the layer's scratch
// (normalised rows, queries, attention output, residual, MLP activations and
// the split-K partial sums of the projections).  Some callers cannot provide
// one at the moment they refresh: a host framework whose caching allocator
// owns all device memory and hands out only the tensors it tracks, or a
// serving loop with a fixed memory budget that must not allocate after
// start-up.  This variant takes that scratch from a fixed array in device
// global memory that the library image itself carries.
//
// Rules of use:
//   - The array is kNoAllocScratchBytes (64 MiB).  Every GPU on which the
//     library's image is loaded holds it until the process exits.  A
//     selection whose layer scratch is larger is rejected with KVR_EINVAL
//     before anything is enqueued (kvr_workspace_bytes(c, 0) reports the
//     need; the Llama-3-8B-shaped refresh of 282 rows needs about 55 MB).
//   - The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and keeps it; make
//     that first call before any stream capture on that device.  A call
//     whose current device is not the cache's device is rejected with
//     KVR_EINVAL.
//   - Every call shares the one array.  Calls whose GPU work overlaps (other
//     streams, other threads, other caches) race on it: serialise them.
//   - The array keeps whatever the last call left in it.  Nothing in a layer
//     reads scratch it has not first written in the same call, so no
//     clearing is needed.
#include <mutex>
#include <string>

#include "kvr_internal.h"

namespace kvr {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_layer_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layer_scratch on the current device (looked up once per device).
kvr_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device index too large for the no-allocation scratch table");
        return KVR_EUNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layer_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress of the layer scratch");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVR_OK;
}

}  // namespace
}  // namespace kvr

using namespace kvr;

extern "C" kvr_status kvr_refresh_layer_noalloc(kvr_cache* c, int32_t layer, const kvr_layer_weights* w,
                                                void* hidden_inout, uint32_t flags, void* stream) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (!c->sel.valid) {
        set_error("no selection: call kvr_select first");
        return KVR_ESTATE;
    }
    // the array's address is looked up on the current device; the layer's
    // kernels work on the cache's buffers, which live on the device the
    // cache was created on
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) {
        set_error("kvr_refresh_layer_noalloc: the current device (" + std::to_string(dev) +
                  ") is not the device the cache was created on (" + std::to_string(c->device) +
                  "); make that device current first");
        return KVR_EINVAL;
    }
    const size_t need = kvr_workspace_bytes(c, 0);
    if (need > kNoAllocScratchBytes) {
        set_error("the layer scratch for " + std::to_string(c->sel.n_rows) + " rows needs " + std::to_string(need) +
                  " bytes; kvr_refresh_layer_noalloc holds at most " + std::to_string(kNoAllocScratchBytes) +
                  " bytes (use kvr_refresh_layer with a caller workspace)");
        return KVR_EINVAL;
    }
    void* scratch = nullptr;
    kvr_status st = scratch_address(&scratch);
    if (st != KVR_OK) return st;
    // per-launch timing would create CUDA events; keep it off for this call
    const bool prof = c->profiling;
    c->profiling = false;
    st = kvr_refresh_layer(c, layer, w, hidden_inout, scratch, kNoAllocScratchBytes, flags, stream);
    c->profiling = prof;
    return st;
}
