// kvq_decode_nvfp4.cu -- decode attention launches for NVFP4 pages on tensor-core
// tiles (F4Warp in kvq_decode_fast.cuh): the kernel of kvq_decode.cuh with 64-token
// FP4 tiles in its fast pool and the fp16 mini tiles as usual.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_nvfp4(const DecodeParams &p, cudaStream_t st) {
    if (p.kitty || p.lens || p.rope || p.D != 128) return cudaErrorInvalidValue;
    constexpr int U = tile_units(4, 4, false, 0);
    if (p.wpc != U) return cudaErrorInvalidValue;
    return launch_one<4, 4, false, true, false, 4, U, false, false, true>(p, st);
}

}  // namespace kvq
