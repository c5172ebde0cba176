// kvq_host.h -- host-side helpers shared by the C ABI translation units (config
// arithmetic, device queries, the tile-path test).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvq.h"
#include "kvq_internal.h"

namespace kvq {
namespace host {

constexpr int kMaxBoostFast = 64;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int vbits_of(const kvq_config *c) { return c->v_bits ? c->v_bits : c->bits; }
inline int kfpi(const kvq_config *c) { return c->mode == KVQ_MODE_KITTY ? 16 : 32 / c->bits; }
inline int vfpi(const kvq_config *c) { return 32 / vbits_of(c); }
inline int gv_of(const kvq_config *c) { return std::min(c->G, c->D); }
// tokens per value tile of a page (the in-page value arrangement, kvq_internal.h)
inline int vtile_of(const kvq_config *c) { return v_tile_tokens(c->mode == KVQ_MODE_KITTY ? 2 : c->bits, c->G); }
inline bool kitty(const kvq_config *c) { return c->mode == KVQ_MODE_KITTY; }
inline bool nvfp4(const kvq_config *c) { return c->mode == KVQ_MODE_NVFP4; }
inline int64_t nvfp4_page_bytes(const kvq_config *c) { return 16 + (int64_t)c->G * c->D / 16; }
inline int64_t cap_k(const kvq_config *c) { return kitty(c) ? c->G : c->R; }
inline int64_t cap_v(const kvq_config *c) { return kitty(c) ? c->G : c->R; }
inline int64_t units(const kvq_config *c) { return (int64_t)c->B * c->H_kv; }

// Slices of the key quantizer: S slices of G/S tokens per thread, with G/S one of
// 16, 32, 64 and whole words per slice (the kernel is instantiated for those).
inline int key_slices(const kvq_config *c) {
    const int fpi = kfpi(c), pairs = c->D / 2, smax = 256 / pairs;
    for (int s = std::min(smax, c->G); s >= 1; s--) {
        if (c->G % s) continue;
        const int tps = c->G / s;
        if ((tps == 16 || tps == 32 || tps == 64) && tps % fpi == 0) return s;
    }
    return 0;
}
inline bool key_slices_ok(const kvq_config *c) { return key_slices(c) > 0; }

inline int status_of(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// SM count of the current device (cached per device; 148 if no device is usable).
inline int num_sms() {
    static int cache[64] = {0};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// Decode attention pieces shared by the C ABI translation units (kvq_api.cu):
//   decode_check_args: the argument checks of kvq_decode_attn other than the workspace;
//   decode_ws_counter_end: bytes [0, n) of a workspace that must be zero when a call
//     starts (status word and per-sequence counters; the partials after them need not);
//   decode_attn_status: kvq_decode_attn with the kernels' device error bits sent to
//     status_word instead of the workspace's own status word.
int decode_check_args(const kvq_config *c, const kvq_cache *k, const uint16_t *q, const uint16_t *out);
size_t decode_ws_counter_end(const kvq_config *c);
int decode_attn_status(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                       size_t ws_bytes, void *stream, int32_t *status_word);

inline bool fast_supported(const kvq_config *c) {
    const int tok = 256 / c->bits;  // a tile holds 8 key word rows
    if (nvfp4(c) && (c->rope || c->D != 128 || c->H_q / c->H_kv > 4 || c->G % 64 || (c->G & (c->G - 1))))
        return false;               // NVFP4 tiles: 64 tokens, D = 128; else the CUDA-core path
    if (nvfp4(c)) return true;
    // tiles: any key and value widths of 2, 4, 8 bits (Kitty: 2-bit planes, 2-bit values)
    if (kitty(c) && vbits_of(c) != 2) return false;
    if (c->D != 128 || c->H_q / c->H_kv > 4) return false;  // hi/lo q' columns need g <= 4
    if (c->G % tok != 0 || gv_of(c) != c->D) return false;
    if (c->G & (c->G - 1)) return false;  // pages of a power-of-two size (shift arithmetic)
    if (kitty(c) && (c->n_boost % 16 != 0 || c->n_boost > kMaxBoostFast)) return false;
    return true;
}

// Warps per pool CTA count for N items (n per sequence): every warp owns >= 1 item
// (so all CTAs between a sequence's first and last hold some of its items) and no
// warp range exceeds n + 1 items (so it touches at most two sequences).
inline int64_t clamp_pool(int64_t want, int64_t N, int64_t n, int wpc) {
    if (N == 0) return 0;
    const int64_t lo = std::max<int64_t>(1, cdiv(N, (int64_t)wpc * (n + 1)));
    const int64_t hi = std::max<int64_t>(1, N / wpc);
    return std::min(hi, std::max(lo, want));
}

// CTAs of the fast and mini pools (one wave of nsm CTAs in all) for N_f / N_m items,
// at most n_f / n_m per sequence (dense caches; a paged cache passes the totals).
// u_f / u_m (paged caches): sequences with items in each pool; a warp range crosses
// about items / (N / u) of them, and each crossing restarts the warp's copy pipeline.
inline void split_pools(int64_t N_f, int64_t n_f, int64_t N_m, int64_t n_m, int wpc, int nsm, int &C_f,
                        int &C_m, int64_t u_f = 0, int64_t u_m = 0) {
    // cost of a mini tile relative to a fast tile (bytes of 16 fp16 tokens vs a packed
    // tile, lighter arithmetic); a pipeline restart costs about 1.5 tiles (measured)
    const double kMini = u_m ? 0.8 : 0.6, kSeg = 1.5;
    auto cost = [&](int64_t N, int64_t C, double per_item, int64_t u) -> double {
        if (!C) return 0.0;
        const double items = (double)cdiv(N, C * wpc);
        const double segs = u ? items * (double)u / (double)N + 1.0 : 0.0;
        return items * per_item + segs * kSeg;
    };
    double best = 1e300;
    int64_t bf = 0, bm = 0;
    const int64_t cm_max = N_m > 0 ? nsm : 0;
    for (int64_t cm0 = (N_m > 0 ? 1 : 0); cm0 <= cm_max; cm0++) {
        const int64_t cm = clamp_pool(cm0, N_m, n_m, wpc);
        const int64_t cf = clamp_pool(std::max<int64_t>(1, nsm - cm), N_f, n_f, wpc);
        const double tf = cost(N_f, cf, 1.0, u_f), tm = cost(N_m, cm, kMini, u_m);
        const double est = (double)cdiv(cf + cm, nsm) * std::max(tf, tm) + 1e-3 * (double)(cf + cm);
        if (est < best) {
            best = est;
            bf = cf;
            bm = cm;
        }
        if (N_f == 0 && cm0 > 0 && cm >= clamp_pool(nsm, N_m, n_m, wpc)) break;
    }
    C_f = (int)bf;
    C_m = (int)bm;
}

}  // namespace host
}  // namespace kvq
