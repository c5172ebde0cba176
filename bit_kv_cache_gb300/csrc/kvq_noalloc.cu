// kvq_noalloc.cu -- decode attention whose workspace is a fixed region of device
// memory that belongs to the library module itself, for callers that cannot hand
// out device memory at all.
//
// The region is a file-scope __device__ array: the CUDA module reserves it when the
// library's code is loaded onto a device, so no call here (or anywhere in the
// library) asks an allocator for memory.  Its address is looked up once per device
// with cudaGetSymbolAddress while that device is current; the first call on a device
// also zero-fills the region on the caller's stream (the status word and the
// per-sequence counters of the split-T combine must start at zero; the decode
// kernel leaves the counters at zero again after every call).
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "kvq.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Address of the scratch region on the current device, zero-filled on first use
// (enqueued on `stream`, so it is ordered before the launch that follows it).
int scratch_of_current_device(cudaStream_t stream, void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return KVQ_ERR_CUDA;
        if (cudaMemsetAsync(ptr, 0, KVQ_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess) return KVQ_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" int kvq_decode_attn_noalloc(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                                       uint16_t *out, void *stream) {
    const size_t need = kvq_decode_attn_workspace_bytes(cfg);
    if (need == 0) return kvq_config_check(cfg) != KVQ_OK ? kvq_config_check(cfg) : KVQ_ERR_INVALID_ARG;
    if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
    void *ws = nullptr;
    const int e = scratch_of_current_device((cudaStream_t)stream, &ws);
    if (e != KVQ_OK) return e;
    return kvq_decode_attn(cfg, cache, q, out, ws, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
