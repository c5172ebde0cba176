// kvq_decode_paged.cu -- decode attention launches for paged caches: the tile kernels
// of kvq_decode.cuh with page-table lookups and per-slot lengths compiled in.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_paged(const DecodeParams &p, cudaStream_t st) { return launch_tiles_any<true>(p, st); }

}  // namespace kvq
