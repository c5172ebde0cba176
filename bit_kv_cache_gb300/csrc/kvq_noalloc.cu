// kvq_noalloc.cu -- decode attention whose workspace is a fixed region of device
// memory that belongs to the library module itself, for callers that cannot hand
// out device memory at all.
//
// The region is a file-scope __device__ array: the CUDA module reserves it when the
// library's code is loaded onto a device, so no call here (or anywhere in the
// library) asks an allocator for memory.  Host code cannot use the array's name as a
// device address, so its address is looked up once per device with
// cudaGetSymbolAddress while that device is current.
//
// Every call first zero-fills the status word and the per-sequence counters at the
// start of the region (a cudaMemsetAsync on the caller's stream, which allocates
// nothing).  Where the counters end depends on the configuration, so a call can
// never rely on what an earlier call with another configuration left there.  The
// kernels' device error bits go to the cache's own status word.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "kvq.h"
#include "kvq_host.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Address of the scratch region on the current device.  The first call on a device
// looks it up (this may load the library's module onto the device, which a stream
// capture does not allow: the first call is refused while `stream` is capturing).
int scratch_of_current_device(cudaStream_t stream, void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return KVQ_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return KVQ_ERR_INVALID_ARG;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return KVQ_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" int kvq_decode_attn_noalloc(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                                       uint16_t *out, void *stream) {
    int e = kvq::host::decode_check_args(cfg, cache, q, out);
    if (e != KVQ_OK) return e;
    if (!cache->status) return KVQ_ERR_INVALID_ARG;  // where device errors are reported
    if (kvq_decode_attn_workspace_bytes(cfg) > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
    void *ws = nullptr;
    if ((e = scratch_of_current_device((cudaStream_t)stream, &ws)) != KVQ_OK) return e;
    if (cudaMemsetAsync(ws, 0, kvq::host::decode_ws_counter_end(cfg), (cudaStream_t)stream) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return kvq::host::decode_attn_status(cfg, cache, q, out, ws, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream,
                                         cache->status);
}
