// kvq_api.cu -- the C ABI of libkvq (declared in include/kvq.h): argument checks,
// the cache bookkeeping of prefill / append / flush, and the decode scheduler.
// Every entry point validates before it enqueues anything, returns a status, and
// leaves the cache untouched on an argument error.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "kvq.h"
#include "kvq_internal.h"

using namespace kvq;

namespace {

constexpr int kMaxBoostFast = 64;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int kfpi(const kvq_config *c) { return c->mode == KVQ_MODE_KITTY ? 16 : 32 / c->bits; }
inline int vfpi(const kvq_config *c) { return 32 / c->bits; }
inline int gv_of(const kvq_config *c) { return std::min(c->G, c->D); }
inline bool kitty(const kvq_config *c) { return c->mode == KVQ_MODE_KITTY; }
inline int64_t cap_k(const kvq_config *c) { return kitty(c) ? c->G : c->R; }
inline int64_t cap_v(const kvq_config *c) { return kitty(c) ? c->G : c->R; }
inline int64_t units(const kvq_config *c) { return (int64_t)c->B * c->H_kv; }

// Slices of the key quantizer (rows of tokens per thread must be 16, 32 or 64).
bool key_slices_ok(const kvq_config *c) {
    const int fpi = kfpi(c), pairs = c->D / 2, smax = 256 / pairs, nwords = c->G / fpi;
    int S = 1;
    for (int s = 1; s <= smax && s <= nwords; s++)
        if (nwords % s == 0 && (c->G / s) <= 64) S = s;
    const int tps = c->G / S;
    return tps == 16 || tps == 32 || tps == 64;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

bool fast_supported(const kvq_config *c) {
    const int tok = c->bits == 2 ? 128 : 64;
    if (c->D != 128 || c->H_q / c->H_kv > 4) return false;  // hi/lo q' columns need g <= 4
    if (c->G % tok != 0 || gv_of(c) != c->D) return false;
    if (kitty(c) && (c->n_boost % 16 != 0 || c->n_boost > kMaxBoostFast)) return false;
    return true;
}

// Partial-slot bound per sequence for a workspace: CTAs of one wave spread over the
// sequences, plus the two CTAs a range can straddle, for each of the two pools.
int64_t slot_bound(const kvq_config *c) { return cdiv(4 * (int64_t)num_sms(), units(c)) + 6; }

struct WsLayout {
    size_t status, tickets, scratch, partials, total;
};

// Upper bound of fast CTAs in one launch: at most nsm, or the minimum that keeps
// every warp range within two sequences (ceil(U / kWarps) when n_fast >= 1).
int64_t max_fast_ctas(const kvq_config *c) { return std::max<int64_t>(num_sms(), cdiv(units(c), kWarps)); }

WsLayout ws_layout(const kvq_config *c) {
    WsLayout w;
    const int64_t U = units(c), g = c->H_q / c->H_kv;
    const int64_t max_cf = max_fast_ctas(c);
    w.status = 0;
    w.tickets = 256;
    w.scratch = w.tickets + (size_t)cdiv(U * 4, 256) * 256;
    w.partials = w.scratch + (size_t)max_cf * kWarps * 8 * (c->D + 2) * 4;
    w.total = w.partials + (size_t)U * slot_bound(c) * g * (c->D + 2) * 4;
    return w;
}

int check_cache_ptrs(const kvq_config *c, const kvq_cache *k) {
    if (!k) return KVQ_ERR_INVALID_ARG;
    const void *need[] = {k->k_codes, k->k_meta, k->v_codes, k->v_meta, k->k_res, k->v_res};
    for (const void *p : need)
        if (!p || !aligned16(p)) return KVQ_ERR_INVALID_ARG;
    if (c->S > 0 && (!k->k_sink || !k->v_sink || !aligned16(k->k_sink) || !aligned16(k->v_sink)))
        return KVQ_ERR_INVALID_ARG;
    if (kitty(c)) {
        if (!k->k_bidx || !aligned16(k->k_bidx) || !k->v_local || !aligned16(k->v_local))
            return KVQ_ERR_INVALID_ARG;
        if (c->n_boost > 0 && (!k->k_hi || !aligned16(k->k_hi))) return KVQ_ERR_INVALID_ARG;
    }
    if (k->n_sink < 0 || k->T_k < 0 || k->n_kres < 0 || k->T_v < 0 || k->n_vres < 0 || k->n_local < 0 ||
        k->local_head < 0 || k->n_sink > c->S || k->T_k > c->max_T || k->T_v > c->max_T ||
        k->T_k % c->G || k->T_v % c->G || k->n_kres > cap_k(c) || k->n_vres > cap_v(c) ||
        (kitty(c) && (k->n_local > c->R || (c->R > 0 && k->local_head >= c->R))))
        return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

QuantKParams qk_params(const kvq_config *c, kvq_cache *k) {
    QuantKParams p;
    memset(&p, 0, sizeof(p));
    p.max_T = c->max_T;
    p.U = (int)units(c);
    p.D = c->D;
    p.G = c->G;
    p.n_boost = kitty(c) ? c->n_boost : 0;
    p.k_codes = k->k_codes;
    p.k_hi = k->k_hi;
    p.k_bidx = k->k_bidx;
    p.k_meta = k->k_meta;
    return p;
}

QuantVParams qv_params(const kvq_config *c, kvq_cache *k) {
    QuantVParams p;
    memset(&p, 0, sizeof(p));
    p.max_T = c->max_T;
    p.U = (int)units(c);
    p.D = c->D;
    p.G = c->G;
    p.Gv = gv_of(c);
    p.v_codes = k->v_codes;
    p.v_meta = k->v_meta;
    return p;
}

cudaError_t copy_rows(const kvq_config *c, const uint16_t *src, int64_t src_rows, int64_t src_r0, uint16_t *dst,
                      int64_t dst_rows, int64_t dst_r0, int64_t n, cudaStream_t st) {
    CopyRowsParams p;
    p.src = src;
    p.dst = dst;
    p.src_rows = src_rows;
    p.src_r0 = src_r0;
    p.dst_rows = dst_rows;
    p.dst_r0 = dst_r0;
    p.n_rows = n;
    p.U = (int)units(c);
    p.D = c->D;
    return launch_copy_rows(p, st);
}

}  // namespace

extern "C" {

const char *kvq_status_str(int s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVQ_ERR_CAPACITY: return "capacity exceeded";
        case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
        case KVQ_ERR_CUDA: return "CUDA error";
        case KVQ_ERR_DEVICE: return "device-side error reported";
    }
    return "unknown status";
}

int kvq_config_check(const kvq_config *c) {
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (c->B <= 0 || c->H_q <= 0 || c->H_kv <= 0 || c->D <= 0 || c->G <= 0 || c->max_T < 0 || c->S < 0 ||
        c->R < 0 || c->n_boost < 0)
        return KVQ_ERR_INVALID_ARG;
    if (c->mode != KVQ_MODE_KIVI && c->mode != KVQ_MODE_KITTY) return KVQ_ERR_INVALID_ARG;
    if (c->bits != 2 && c->bits != 4) return KVQ_ERR_UNSUPPORTED;
    if (kitty(c) && c->bits != 2) return KVQ_ERR_UNSUPPORTED;
    if (c->H_q % c->H_kv) return KVQ_ERR_INVALID_ARG;
    if (c->H_q / c->H_kv > 8) return KVQ_ERR_UNSUPPORTED;
    if (c->D != 64 && c->D != 128 && c->D != 256) return KVQ_ERR_UNSUPPORTED;
    if (c->G % kfpi(c) || c->G % vfpi(c) || c->D % vfpi(c)) return KVQ_ERR_INVALID_ARG;
    const int gv = gv_of(c);
    if (c->D % gv) return KVQ_ERR_INVALID_ARG;
    if (gv != 32 && gv != 64 && gv != 128 && gv != 256) return KVQ_ERR_UNSUPPORTED;
    if (!key_slices_ok(c)) return KVQ_ERR_UNSUPPORTED;
    if (c->max_T % c->G) return KVQ_ERR_INVALID_ARG;
    if (!kitty(c)) {
        if (c->n_boost != 0) return KVQ_ERR_INVALID_ARG;
        if (c->R < c->G || c->R % c->G) return KVQ_ERR_INVALID_ARG;
    } else {
        if (c->n_boost > std::min(c->D, 254)) return KVQ_ERR_INVALID_ARG;
        if (c->R < 1) return KVQ_ERR_INVALID_ARG;
    }
    return KVQ_OK;
}

size_t kvq_buffer_bytes(const kvq_config *c, int which) {
    if (kvq_config_check(c) != KVQ_OK) return 0;
    const size_t U = (size_t)units(c), D = c->D, T = (size_t)c->max_T, G = c->G;
    switch (which) {
        case 0: return U * (T / kfpi(c)) * D * 4;
        case 1: return kitty(c) && c->n_boost ? U * (T / 16) * c->n_boost * 4 : 0;
        case 2: return kitty(c) ? U * (T / G) * D : 0;
        case 3: return U * (T / G) * D * 4;
        case 4: return U * T * (D / vfpi(c)) * 4;
        case 5: return U * T * (D / gv_of(c)) * 4;
        case 6: return U * (size_t)c->S * D * 2;
        case 7: return U * (size_t)cap_k(c) * D * 2;
        case 8: return U * (size_t)cap_v(c) * D * 2;
        case 9: return kitty(c) ? U * (size_t)c->R * D * 2 : 0;
    }
    return 0;
}

int kvq_quant_pack_k(const kvq_config *c, kvq_cache *k, const uint16_t *src, int64_t L0, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!src || !aligned16(src) || L0 < 1) return KVQ_ERR_INVALID_ARG;
    if (k->T_k != 0 || k->n_kres != 0) return KVQ_ERR_INVALID_ARG;  // key side must be empty
    const int64_t ns = std::min<int64_t>(c->S, L0);
    if (k->n_sink != 0 && k->n_sink != ns) return KVQ_ERR_INVALID_ARG;
    const int64_t rest = L0 - ns, tk = rest / c->G * c->G, kres = rest - tk;
    if (tk > c->max_T) return KVQ_ERR_CAPACITY;
    if (kres > cap_k(c)) return KVQ_ERR_CAPACITY;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t ce = cudaSuccess;
    if (ns > 0) ce = copy_rows(c, src, L0, 0, k->k_sink, c->S, 0, ns, st);
    if (ce == cudaSuccess && tk > 0) {
        QuantKParams p = qk_params(c, k);
        p.src = src;
        p.src_ustride = L0 * c->D;
        p.src_t0 = ns;
        p.n_pages = tk / c->G;
        p.pg0 = 0;
        ce = launch_quant_k(p, c->bits, kitty(c), st);
    }
    if (ce == cudaSuccess && kres > 0) ce = copy_rows(c, src, L0, ns + tk, k->k_res, cap_k(c), 0, kres, st);
    if (ce != cudaSuccess) return KVQ_ERR_CUDA;
    k->n_sink = ns;
    k->T_k = tk;
    k->n_kres = kres;
    return KVQ_OK;
}

int kvq_quant_pack_v(const kvq_config *c, kvq_cache *k, const uint16_t *src, int64_t L0, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!src || !aligned16(src) || L0 < 1) return KVQ_ERR_INVALID_ARG;
    if (k->T_v != 0 || k->n_vres != 0 || k->n_local != 0) return KVQ_ERR_INVALID_ARG;
    const int64_t ns = std::min<int64_t>(c->S, L0);
    if (k->n_sink != 0 && k->n_sink != ns) return KVQ_ERR_INVALID_ARG;
    const int64_t rest = L0 - ns;
    int64_t nl = 0, older = rest;
    if (kitty(c)) {
        nl = std::min<int64_t>(c->R, rest);
        older = rest - nl;
    }
    const int64_t tv = older / c->G * c->G, vres = older - tv;
    if (tv > c->max_T) return KVQ_ERR_CAPACITY;
    if (vres > cap_v(c)) return KVQ_ERR_CAPACITY;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t ce = cudaSuccess;
    if (ns > 0) ce = copy_rows(c, src, L0, 0, k->v_sink, c->S, 0, ns, st);
    if (ce == cudaSuccess && tv > 0) {
        QuantVParams p = qv_params(c, k);
        p.src = src;
        p.src_ustride = L0 * c->D;
        p.src_t0 = ns;
        p.n_tok = tv;
        p.tok0 = 0;
        ce = launch_quant_v(p, c->bits, st);
    }
    if (ce == cudaSuccess && vres > 0) ce = copy_rows(c, src, L0, ns + tv, k->v_res, cap_v(c), 0, vres, st);
    if (ce == cudaSuccess && nl > 0) ce = copy_rows(c, src, L0, ns + older, k->v_local, c->R, 0, nl, st);
    if (ce != cudaSuccess) return KVQ_ERR_CUDA;
    k->n_sink = ns;
    k->T_v = tv;
    k->n_vres = vres;
    k->n_local = nl;
    k->local_head = 0;
    return KVQ_OK;
}

int kvq_append_token(const kvq_config *c, kvq_cache *k, const uint16_t *kn, const uint16_t *vn, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!kn || !vn || !aligned16(kn) || !aligned16(vn)) return KVQ_ERR_INVALID_ARG;
    AppendParams p;
    memset(&p, 0, sizeof(p));
    p.k_new = kn;
    p.v_new = vn;
    p.U = (int)units(c);
    p.D = c->D;
    p.evict_row = -1;
    kvq_cache nk = *k;
    if (k->n_sink < c->S) {
        if (k->T_k || k->n_kres || k->T_v || k->n_vres || k->n_local) return KVQ_ERR_INVALID_ARG;
        p.k_dst = k->k_sink;
        p.k_rows = c->S;
        p.k_row = k->n_sink;
        p.v_dst = k->v_sink;
        p.v_rows = c->S;
        p.v_row = k->n_sink;
        nk.n_sink++;
    } else {
        if (k->n_kres >= cap_k(c)) return KVQ_ERR_CAPACITY;
        p.k_dst = k->k_res;
        p.k_rows = cap_k(c);
        p.k_row = k->n_kres;
        nk.n_kres++;
        if (!kitty(c)) {
            if (k->n_vres >= cap_v(c)) return KVQ_ERR_CAPACITY;
            p.v_dst = k->v_res;
            p.v_rows = cap_v(c);
            p.v_row = k->n_vres;
            nk.n_vres++;
        } else if (k->n_local < c->R) {
            p.v_dst = k->v_local;
            p.v_rows = c->R;
            p.v_row = (k->local_head + k->n_local) % c->R;
            nk.n_local++;
        } else {
            if (k->n_vres >= cap_v(c)) return KVQ_ERR_CAPACITY;
            p.v_dst = k->v_local;
            p.v_rows = c->R;
            p.v_row = k->local_head;
            p.v_evict = k->v_res;
            p.evict_rows = cap_v(c);
            p.evict_row = k->n_vres;
            nk.n_vres++;
            nk.local_head = (k->local_head + 1) % c->R;
        }
    }
    if (launch_append(p, (cudaStream_t)stream) != cudaSuccess) return KVQ_ERR_CUDA;
    *k = nk;
    return KVQ_OK;
}

int kvq_flush_group(const kvq_config *c, kvq_cache *k, int *flushed_k, int *flushed_v, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    const bool fk = k->n_kres == cap_k(c), fv = k->n_vres == cap_v(c);
    if ((fk && k->T_k + cap_k(c) > c->max_T) || (fv && k->T_v + cap_v(c) > c->max_T)) return KVQ_ERR_CAPACITY;
    cudaStream_t st = (cudaStream_t)stream;
    if (fk) {
        QuantKParams p = qk_params(c, k);
        p.src = k->k_res;
        p.src_ustride = cap_k(c) * c->D;
        p.src_t0 = 0;
        p.n_pages = cap_k(c) / c->G;
        p.pg0 = k->T_k / c->G;
        if (launch_quant_k(p, c->bits, kitty(c), st) != cudaSuccess) return KVQ_ERR_CUDA;
        k->T_k += cap_k(c);
        k->n_kres = 0;
    }
    if (fv) {
        QuantVParams p = qv_params(c, k);
        p.src = k->v_res;
        p.src_ustride = cap_v(c) * c->D;
        p.src_t0 = 0;
        p.n_tok = cap_v(c);
        p.tok0 = k->T_v;
        if (launch_quant_v(p, c->bits, st) != cudaSuccess) return KVQ_ERR_CUDA;
        k->T_v += cap_v(c);
        k->n_vres = 0;
    }
    if (flushed_k) *flushed_k = fk ? 1 : 0;
    if (flushed_v) *flushed_v = fv ? 1 : 0;
    return KVQ_OK;
}

size_t kvq_decode_attn_workspace_bytes(const kvq_config *c) {
    if (kvq_config_check(c) != KVQ_OK) return 0;
    return ws_layout(c).total;
}

int kvq_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!ws || ws_bytes == 0) return KVQ_ERR_INVALID_ARG;
    return status_of(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

int kvq_decode_attn(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                    size_t ws_bytes, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
    const int64_t L = k->n_sink + k->T_k + k->n_kres;
    const int64_t Lv = k->n_sink + k->T_v + k->n_vres + k->n_local;
    if (L < 1 || L != Lv) return KVQ_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(c);
    if (!ws || !aligned16(ws) || ws_bytes < wl.total) return KVQ_ERR_WORKSPACE;

    const int U = (int)units(c), g = c->H_q / c->H_kv, nsm = num_sms();
    const bool fast = fast_supported(c);
    const int tok = c->bits == 2 ? 128 : 64;
    const int64_t n_fast = fast ? std::min(k->T_k, k->T_v) / tok : 0;
    const int64_t n_gen = L - n_fast * tok;
    const int64_t N_f = (int64_t)U * n_fast;

    // Schedule: split the GPU between fast CTAs (tiles) and generic CTAs (chunks of
    // the remaining tokens) so that the longest warp is as short as possible.
    // Cost unit: one fast tile; a generic token costs about kGen of a tile.
    const double kGen = fast ? 5.0 / tok : 1.0 / 32.0;
    int best_cf = 0, best_cg = 0, best_ngc = 0;
    int64_t best_chunk = 0;
    double best = 1e300;
    const int64_t gmax = std::max<int64_t>(32, cdiv(n_gen, 32) * 32);
    int64_t cands[40];
    int nc = 0;
    for (int64_t ch = 32; ch <= 256 && ch < gmax; ch += 32) cands[nc++] = ch;
    for (int64_t ch = 512; ch < gmax && nc < 39; ch *= 2) cands[nc++] = ch;
    cands[nc++] = gmax;  // the whole generic part of a sequence in one chunk
    for (int ci = 0; ci < nc; ci++) {
        const int64_t chunk = cands[ci];
        const int64_t ngc = n_gen > 0 ? cdiv(n_gen, chunk) : 0;
        const int64_t cg = cdiv((int64_t)U * ngc, kWarps);
        if (cg > 4 * (int64_t)nsm && chunk < gmax) continue;  // too many generic CTAs
        // Fast CTAs: every warp must own >= 1 tile (W_f <= N_f, so the CTAs between the
        // first and last CTA of a sequence all hold some of its tiles) and no warp range
        // may exceed n_fast + 1 tiles (so a warp touches at most two sequences).
        int64_t cf = 0;
        if (N_f > 0) {
            const int64_t lo = std::max<int64_t>(1, cdiv(N_f, (int64_t)kWarps * (n_fast + 1)));
            const int64_t hi = std::max<int64_t>(1, N_f / kWarps);
            cf = std::min(hi, std::max(lo, (int64_t)nsm - cg));
        }
        const double tf = N_f > 0 ? (double)cdiv(N_f, cf * kWarps) : 0.0;
        const double tg = ngc > 0 ? (double)std::min(chunk, n_gen) * kGen : 0.0;
        const int64_t waves = cdiv(cf + cg, nsm);
        const double est = (double)waves * std::max(tf, tg) + 0.02 * (double)(cf + cg) / U;
        if (est < best) {
            best = est;
            best_cf = (int)cf;
            best_cg = (int)cg;
            best_ngc = (int)ngc;
            best_chunk = chunk;
        }
    }

    DecodeParams p;
    memset(&p, 0, sizeof(p));
    p.B = c->B;
    p.H_kv = c->H_kv;
    p.g = g;
    p.D = c->D;
    p.G = c->G;
    p.bits = c->bits;
    p.Gv = gv_of(c);
    p.n_boost = kitty(c) ? c->n_boost : 0;
    p.kitty = kitty(c) ? 1 : 0;
    p.S_cap = c->S;
    p.cap_k = (int)cap_k(c);
    p.cap_v = (int)cap_v(c);
    p.R_local = kitty(c) ? c->R : 1;
    p.max_T = c->max_T;
    p.n_sink = k->n_sink;
    p.T_k = k->T_k;
    p.n_kres = k->n_kres;
    p.T_v = k->T_v;
    p.n_vres = k->n_vres;
    p.n_local = k->n_local;
    p.local_head = k->local_head;
    p.L = L;
    p.k_codes = k->k_codes;
    p.k_hi = k->k_hi;
    p.k_bidx = k->k_bidx;
    p.k_meta = k->k_meta;
    p.v_codes = k->v_codes;
    p.v_meta = k->v_meta;
    p.k_sink = k->k_sink;
    p.v_sink = k->v_sink;
    p.k_res = k->k_res;
    p.v_res = k->v_res;
    p.v_local = k->v_local;
    p.q = q;
    p.out = out;
    char *w = static_cast<char *>(ws);
    p.status = reinterpret_cast<int32_t *>(w + wl.status);
    p.tickets = reinterpret_cast<int32_t *>(w + wl.tickets);
    p.scratch = reinterpret_cast<float *>(w + wl.scratch);
    p.partials = reinterpret_cast<float *>(w + wl.partials);
    p.U = U;
    p.C_f = best_cf;
    p.C_g = best_cg;
    p.n_gc = best_ngc;
    p.n_fast = n_fast;
    p.N_f = N_f;
    p.n_gen = n_gen;
    p.gen_chunk = best_chunk;
    // slots per sequence: fast CTAs touching it + generic CTAs touching it
    int64_t max_slots = 0;
    const int64_t Wf = (int64_t)best_cf * kWarps;
    auto warp_of = [&](int64_t x) { return std::min(Wf - 1, ((x + 1) * Wf - 1) / N_f); };
    for (int64_t u = 0; u < U; u++) {
        int64_t s = 0;
        if (n_fast > 0) s += warp_of((u + 1) * n_fast - 1) / kWarps - warp_of(u * n_fast) / kWarps + 1;
        if (best_ngc > 0) s += ((u + 1) * best_ngc - 1) / kWarps - (u * best_ngc) / kWarps + 1;
        max_slots = std::max(max_slots, s);
    }
    if (best == 1e300 || max_slots > slot_bound(c) || (int64_t)best_cf > max_fast_ctas(c))
        return KVQ_ERR_UNSUPPORTED;
    p.max_slots = (int)max_slots;
    return status_of(launch_decode(p, fast, (cudaStream_t)stream));
}

int kvq_read_status(const kvq_cache *k, void *ws, int32_t *dev_status, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    int32_t acc = 0, v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (ws) {
        if (cudaMemcpy(&v, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
        acc |= v;
        if (v && cudaMemset(ws, 0, 4) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    if (k && k->status) {
        if (cudaMemcpy(&v, k->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
        acc |= v;
        if (v && cudaMemset(k->status, 0, 4) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    if (dev_status) *dev_status = acc;
    return acc ? KVQ_ERR_DEVICE : KVQ_OK;
}

}  // extern "C"
