// kvq_decode.cu -- decode attention launches for dense caches (the kernel template is
// in kvq_decode.cuh; paged caches are instantiated in kvq_decode_paged.cu).
#include "kvq_decode.cuh"

namespace kvq {

int decode_warps_per_cta(int bits, int vbits, bool kitty, int n_boost, bool fast) {
    if (!fast) return 8;
    return tile_units(bits, vbits, kitty, n_boost);
}

size_t decode_smem_bytes(int bits, int vbits, bool kitty, int n_boost, int D, bool fast) {
    const int nw = decode_warps_per_cta(bits, vbits, kitty, n_boost, fast);
    if (fast) return (size_t)nw * WarpSmem(bits, vbits, kitty, n_boost).total;
    return (size_t)nw * gen_warp_bytes(D);
}

cudaError_t launch_decode(const DecodeParams &p, bool fast, cudaStream_t st) {
    if (p.rope) return launch_decode_rope(p, fast, st);
    if (p.nvfp4 && fast) return launch_decode_nvfp4(p, st);
    if (fast) {  // p.wpc units of one warp, or of a warp pair
        if (p.kitty) {
            if (p.wpc == 8) return launch_one<2, 2, true, true, false, 4, 8>(p, st);
            if (p.wpc == 6) return launch_one<2, 2, true, true, false, 4, 6>(p, st);
            return cudaErrorInvalidValue;  // n_boost <= 64 keeps 6 units in the CTA
        }
        if (p.lens) return launch_decode_paged(p, st);
        return launch_tiles_any<false>(p, st);
    }
    switch (p.D) {
        case 64: return launch_one<2, 2, false, false, false, 2, 8>(p, st);
        case 128: return launch_one<2, 2, false, false, false, 4, 8>(p, st);
        case 256: return launch_one<2, 2, false, false, false, 8, 8>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvq
