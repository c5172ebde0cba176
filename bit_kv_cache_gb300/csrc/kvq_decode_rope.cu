// kvq_decode_rope.cu -- decode attention launches for pre-RoPE keys (KVQuant notes,
// mechanism two): the kernels of kvq_decode.cuh with keys turned by their position
// before the dot product.  KIVI mode, dense caches.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_rope(const DecodeParams &p, bool fast, cudaStream_t st) {
    if (p.kitty || p.lens) return cudaErrorInvalidValue;
    if (fast) return launch_tiles_any<false, true>(p, st);
    switch (p.D) {
        case 64: return launch_one<2, 2, false, false, false, 2, 8, false, true>(p, st);
        case 128: return launch_one<2, 2, false, false, false, 4, 8, false, true>(p, st);
        case 256: return launch_one<2, 2, false, false, false, 8, 8, false, true>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvq
