// kvq_api.cu -- the C ABI of libkvq (declared in include/kvq.h): argument checks,
// the cache bookkeeping of prefill / append / flush, and the decode scheduler.
// Every entry point validates before it enqueues anything, returns a status, and
// leaves the cache untouched on an argument error.
#include <cuda_runtime.h>

#include <chrono>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "kvq.h"
#include "kvq_host.h"
#include "kvq_internal.h"

using namespace kvq;
using namespace kvq::host;

namespace {

// Partial-slot bound per sequence: the CTAs of the pools spread over the sequences,
// plus the CTAs a range can straddle at both ends, for each pool.
int64_t slot_bound(const kvq_config *c) { return cdiv(4 * (int64_t)num_sms(), units(c)) + 8; }

// Upper bound of the CTAs of one pool: one wave, or the minimum that keeps every warp
// range within two sequences (about U / warps-per-CTA).
int64_t max_pool_ctas(const kvq_config *c) { return std::max<int64_t>(num_sms(), cdiv(units(c), 6)); }

// Workspace: [status word][item counters U x 8 B][partials].  The counters are zero
// between calls (the combining CTA resets them); the partials need no initial value.
struct WsLayout {
    size_t status, item_ctr, partials, total;
};

WsLayout ws_layout(const kvq_config *c) {
    WsLayout w;
    const int64_t U = units(c), g = c->H_q / c->H_kv;
    w.status = 0;
    w.item_ctr = 256;
    w.partials = w.item_ctr + (size_t)cdiv(U * 8, 256) * 256;
    w.total = w.partials + (size_t)U * slot_bound(c) * g * (c->D + 4) * 4;
    return w;
}

// Packed pages a prefill or flush has written since the cache's last decode, per cache
// (keyed by its key-code buffer): the first such key and value token.  Decode launches
// may start before the preceding kernel in the stream has completed, and copy the
// packed pages below these tokens early; the others only after that kernel is done.
constexpr int64_t kNoFresh = INT64_MAX;
struct Fresh {
    int64_t k = kNoFresh, v = kNoFresh;
};
std::mutex g_fresh_mu;
std::unordered_map<const void *, Fresh> g_fresh;

void mark_fresh(const kvq_cache *k, int64_t k_tok, int64_t v_tok) {
    std::lock_guard<std::mutex> lock(g_fresh_mu);
    Fresh &f = g_fresh[k->k_codes];
    f.k = std::min(f.k, k_tok);
    f.v = std::min(f.v, v_tok);
}

// The first fresh token of the cache (keys or values), which is then forgotten: a
// later decode is preceded by this one, which writes no packed page.
int64_t take_fresh(const kvq_cache *k) {
    std::lock_guard<std::mutex> lock(g_fresh_mu);
    auto it = g_fresh.find(k->k_codes);
    if (it == g_fresh.end()) return kNoFresh;
    const int64_t r = std::min(it->second.k, it->second.v);
    g_fresh.erase(it);
    return r;
}

// CTAs of a pool (C CTAs, wpc warps each, N items, n per sequence) holding items of u.
int64_t pool_ctas_host(int64_t C, int wpc, int64_t N, int64_t n, int64_t u) {
    if (n == 0 || C == 0) return 0;
    const int64_t W = C * wpc;
    auto warp_of = [&](int64_t x) { return std::min(W - 1, ((x + 1) * W - 1) / N); };
    return warp_of((u + 1) * n - 1) / wpc - warp_of(u * n) / wpc + 1;
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
    p.status = k->status;
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
    p.TV = vtile_of(c);
    p.v_codes = k->v_codes;
    p.v_meta = k->v_meta;
    p.status = k->status;
    return p;
}

// Key / value page quantization of either format: the KIVI / Kitty quantizers, or the
// NVFP4 page kernel with the same source rows and destination pages.
cudaError_t launch_keys(const kvq_config *c, kvq_cache *k, const QuantKParams &p, cudaStream_t st) {
    if (!nvfp4(c)) return launch_quant_k(p, c->bits, kitty(c), st);
    QuantNvParams q;
    q.src = p.src;
    q.src_ustride = p.src_ustride;
    q.src_t0 = p.src_t0;
    q.n_pages = p.n_pages;
    q.pg0 = p.pg0;
    q.max_T = c->max_T;
    q.U = (int)units(c);
    q.D = c->D;
    q.G = c->G;
    q.ms = (int)nvfp4_page_bytes(c);
    q.codes = reinterpret_cast<uint8_t *>(k->k_codes);
    q.meta = reinterpret_cast<uint8_t *>(k->k_meta);
    return launch_nvfp4(q, false, st);
}
cudaError_t launch_values(const kvq_config *c, kvq_cache *k, const QuantVParams &p, cudaStream_t st) {
    if (!nvfp4(c)) return launch_quant_v(p, vbits_of(c), st);
    QuantNvParams q;
    q.src = p.src;
    q.src_ustride = p.src_ustride;
    q.src_t0 = p.src_t0;
    q.n_pages = p.n_tok / c->G;
    q.pg0 = p.tok0 / c->G;
    q.max_T = c->max_T;
    q.U = (int)units(c);
    q.D = c->D;
    q.G = c->G;
    q.ms = (int)nvfp4_page_bytes(c);
    q.codes = reinterpret_cast<uint8_t *>(k->v_codes);
    q.meta = reinterpret_cast<uint8_t *>(k->v_meta);
    return launch_nvfp4(q, true, st);
}

// Adds a row copy (same arguments as copy_rows) to the copies a quant launch carries.
void add_rows(RowCopies &rc, const uint16_t *src, int64_t src_rows, int64_t src_r0, uint16_t *dst, int64_t dst_rows,
              int64_t dst_r0, int64_t n) {
    if (n <= 0) return;
    RowCopy &r = rc.c[rc.n++];
    r.src = src;
    r.dst = dst;
    r.src_rows = src_rows;
    r.src_r0 = src_r0;
    r.dst_rows = dst_rows;
    r.dst_r0 = dst_r0;
    r.n_rows = n;
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
    if (c->mode != KVQ_MODE_KIVI && c->mode != KVQ_MODE_KITTY && c->mode != KVQ_MODE_NVFP4)
        return KVQ_ERR_INVALID_ARG;
    if (nvfp4(c)) {
        if (c->bits != 4 || (c->v_bits != 0 && c->v_bits != 4)) return KVQ_ERR_UNSUPPORTED;
        if (c->G % 16 || c->D % 16 || c->G > 256) return KVQ_ERR_UNSUPPORTED;
    }
    if (c->bits != 2 && c->bits != 4 && c->bits != 8) return KVQ_ERR_UNSUPPORTED;
    if (c->v_bits != 0 && c->v_bits != 2 && c->v_bits != 4 && c->v_bits != 8) return KVQ_ERR_UNSUPPORTED;
    if (kitty(c) && c->bits != 2) return KVQ_ERR_UNSUPPORTED;
    if (c->H_q % c->H_kv) return KVQ_ERR_INVALID_ARG;
    if (c->H_q / c->H_kv > 8) return KVQ_ERR_UNSUPPORTED;
    if (c->D != 64 && c->D != 128 && c->D != 256) return KVQ_ERR_UNSUPPORTED;
    if (c->G % kfpi(c) || c->G % vfpi(c) || c->D % vfpi(c)) return KVQ_ERR_INVALID_ARG;
    const int gv = gv_of(c);
    if (c->D % gv) return KVQ_ERR_INVALID_ARG;
    if (gv != 32 && gv != 64 && gv != 128 && gv != 256) return KVQ_ERR_UNSUPPORTED;
    if (!nvfp4(c) && !key_slices_ok(c)) return KVQ_ERR_UNSUPPORTED;
    if (c->max_T % c->G) return KVQ_ERR_INVALID_ARG;
    if (c->rope != 0 && c->rope != 1) return KVQ_ERR_INVALID_ARG;
    if (!(c->rope_base >= 0.0f) || c->rope_base > 3.0e38f) return KVQ_ERR_INVALID_ARG;
    if (c->rope && kitty(c)) return KVQ_ERR_UNSUPPORTED;
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
    if (nvfp4(c)) {
        switch (which) {
            case 0: case 4: return U * T * D / 2;
            case 3: case 5: return U * (T / G) * (size_t)nvfp4_page_bytes(c);
            case 6: return U * (size_t)c->S * D * 2;
            case 7: case 8: return U * (size_t)c->R * D * 2;
        }
        return 0;
    }
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
    if (tk > 0 && !nvfp4(c)) {  // one launch: the pages, with the sink and residual rows
        QuantKParams p = qk_params(c, k);
        p.src = src;
        p.src_ustride = L0 * c->D;
        p.src_t0 = ns;
        p.n_pages = tk / c->G;
        p.pg0 = 0;
        add_rows(p.rc, src, L0, 0, k->k_sink, c->S, 0, ns);
        add_rows(p.rc, src, L0, ns + tk, k->k_res, cap_k(c), 0, kres);
        ce = launch_keys(c, k, p, st);
    } else {
        if (ns > 0) ce = copy_rows(c, src, L0, 0, k->k_sink, c->S, 0, ns, st);
        if (ce == cudaSuccess && tk > 0) {
            QuantKParams p = qk_params(c, k);
            p.src = src;
            p.src_ustride = L0 * c->D;
            p.src_t0 = ns;
            p.n_pages = tk / c->G;
            p.pg0 = 0;
            ce = launch_keys(c, k, p, st);
        }
        if (ce == cudaSuccess && kres > 0) ce = copy_rows(c, src, L0, ns + tk, k->k_res, cap_k(c), 0, kres, st);
    }
    if (ce != cudaSuccess) return KVQ_ERR_CUDA;
    if (tk > 0) mark_fresh(k, 0, kNoFresh);
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
    if (tv > 0 && !nvfp4(c)) {  // one launch: the pages, with the sink, residual and window rows
        QuantVParams p = qv_params(c, k);
        p.src = src;
        p.src_ustride = L0 * c->D;
        p.src_t0 = ns;
        p.n_tok = tv;
        p.tok0 = 0;
        add_rows(p.rc, src, L0, 0, k->v_sink, c->S, 0, ns);
        add_rows(p.rc, src, L0, ns + tv, k->v_res, cap_v(c), 0, vres);
        add_rows(p.rc, src, L0, ns + older, k->v_local, c->R, 0, nl);
        ce = launch_values(c, k, p, st);
    } else {
        if (ns > 0) ce = copy_rows(c, src, L0, 0, k->v_sink, c->S, 0, ns, st);
        if (ce == cudaSuccess && tv > 0) {
            QuantVParams p = qv_params(c, k);
            p.src = src;
            p.src_ustride = L0 * c->D;
            p.src_t0 = ns;
            p.n_tok = tv;
            p.tok0 = 0;
            ce = launch_values(c, k, p, st);
        }
        if (ce == cudaSuccess && vres > 0) ce = copy_rows(c, src, L0, ns + tv, k->v_res, cap_v(c), 0, vres, st);
        if (ce == cudaSuccess && nl > 0) ce = copy_rows(c, src, L0, ns + older, k->v_local, c->R, 0, nl, st);
    }
    if (ce != cudaSuccess) return KVQ_ERR_CUDA;
    if (tv > 0) mark_fresh(k, kNoFresh, 0);
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
        if (launch_keys(c, k, p, st) != cudaSuccess) return KVQ_ERR_CUDA;
        mark_fresh(k, k->T_k, kNoFresh);
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
        if (launch_values(c, k, p, st) != cudaSuccess) return KVQ_ERR_CUDA;
        mark_fresh(k, kNoFresh, k->T_v);
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

// Decode attention over cache k.  kn / vn (may be null): append them in the same launch
// (k already holds the lengths after the append); returns kDeclined, with nothing
// enqueued, if the packed-tile path does not serve this call.
static constexpr int kDeclined = 1;
static int decode_impl(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                       size_t ws_bytes, void *stream, const uint16_t *kn, const uint16_t *vn,
                       int32_t *status_word = nullptr, unsigned int *done = nullptr);

int kvq_decode_attn(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                    size_t ws_bytes, void *stream) {
    return decode_impl(c, k, q, out, ws, ws_bytes, stream, nullptr, nullptr);
}

// kvq_append_decode; done (device address, may be null): the decode kernel's
// completion count (DecodeParams::done).
static int append_decode_impl(const kvq_config *c, kvq_cache *k, const uint16_t *kn, const uint16_t *vn,
                              const uint16_t *q, uint16_t *out, void *ws, size_t ws_bytes, int *fused,
                              void *stream, unsigned int *done) {
    if (fused) *fused = 0;
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!kn || !vn || !aligned16(kn) || !aligned16(vn)) return KVQ_ERR_INVALID_ARG;
    // one launch: the token goes to both residuals of a KIVI cache, and the tile path
    // serves the attention over the lengths after the append
    if (!kitty(c) && k->n_sink >= c->S && k->n_kres < cap_k(c) && k->n_vres < cap_v(c) &&
        k->n_sink + k->T_k + k->n_kres == k->n_sink + k->T_v + k->n_vres + k->n_local) {
        kvq_cache nk = *k;
        nk.n_kres++;
        nk.n_vres++;
        e = decode_impl(c, &nk, q, out, ws, ws_bytes, stream, kn, vn, nullptr, done);
        if (e != kDeclined) {
            if (e == KVQ_OK) {
                *k = nk;
                if (fused) *fused = 1;
            }
            return e;
        }
    }
    if ((e = kvq_append_token(c, k, kn, vn, stream))) return e;
    return decode_impl(c, k, q, out, ws, ws_bytes, stream, nullptr, nullptr, nullptr, done);
}

int kvq_append_decode(const kvq_config *c, kvq_cache *k, const uint16_t *kn, const uint16_t *vn,
                      const uint16_t *q, uint16_t *out, void *ws, size_t ws_bytes, int *fused, void *stream) {
    return append_decode_impl(c, k, kn, vn, q, out, ws, ws_bytes, fused, stream, nullptr);
}

static int decode_impl(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                       size_t ws_bytes, void *stream, const uint16_t *kn, const uint16_t *vn,
                       int32_t *status_word, unsigned int *done) {
    int e = kvq::host::decode_check_args(c, k, q, out);
    if (e) return e;
    const int64_t L = k->n_sink + k->T_k + k->n_kres;
    const WsLayout wl = ws_layout(c);
    if (!ws || !aligned16(ws) || ws_bytes < wl.total) return KVQ_ERR_WORKSPACE;

    const int U = (int)units(c), g = c->H_q / c->H_kv, nsm = num_sms();
    const int tok = 256 / c->bits;
    // The tile paths cover: D = 128, g <= 4, pages of whole tiles, one value group per
    // token, packed values never ahead of packed keys, mixed key blocks only at 2 bits.
    bool fast = fast_supported(c) && k->T_v <= k->T_k && k->T_v % tok == 0 &&
                (k->T_k == k->T_v || (kitty(c) && (k->T_k - k->T_v) % 16 == 0));
    if (kn && !fast) return kDeclined;
    const int wpc = decode_warps_per_cta(c->bits, vbits_of(c), kitty(c), kitty(c) ? c->n_boost : 0, fast);

    DecodeParams p;
    memset(&p, 0, sizeof(p));
    p.U = U;
    p.wpc = wpc;
    // The schedule depends only on these numbers.  Decode steps repeat them for 16
    // tokens at a time, and the layers of a model share them; a small per-thread cache
    // (direct-mapped on a hash of the numbers) keeps recent ones.
    struct SchedKey {
        int64_t U, wpc, nsm, fast, T_k, T_v, n_sink, n_kres, L, tok;
        bool operator==(const SchedKey &o) const { return memcmp(this, &o, sizeof(*this)) == 0; }
    };
    struct SchedVal {
        int C_f, C_m, C_g, n_gc, max_slots;
        int64_t n_fast, n_mini, N_f, N_m, n_gen, gen_chunk;
    };
    struct SchedEntry {
        SchedKey key;
        SchedVal val;
        bool valid;
    };
    static thread_local SchedEntry sched_cache[32];
    SchedKey key;
    memset(&key, 0, sizeof(key));
    key.U = U;
    key.wpc = wpc;
    key.nsm = nsm;
    key.fast = fast;
    key.T_k = k->T_k;
    key.T_v = k->T_v;
    key.n_sink = k->n_sink;
    key.n_kres = k->n_kres;
    key.L = L;
    key.tok = tok;
    uint64_t hsh = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(key) / sizeof(int64_t); i++)
        hsh = (hsh ^ (uint64_t)reinterpret_cast<const int64_t *>(&key)[i]) * 1099511628211ull;
    SchedEntry &ce = sched_cache[(hsh >> 29) & 31];
    const bool hit = ce.valid && key == ce.key;
    if (hit) {
        const SchedVal &v = ce.val;
        p.C_f = v.C_f;
        p.C_m = v.C_m;
        p.C_g = v.C_g;
        p.n_gc = v.n_gc;
        p.max_slots = v.max_slots;
        p.n_fast = v.n_fast;
        p.n_mini = v.n_mini;
        p.N_f = v.N_f;
        p.N_m = v.N_m;
        p.n_gen = v.n_gen;
        p.gen_chunk = v.gen_chunk;
    } else if (fast) {
        // fast tiles: keys and values packed; mini tiles: the rest in 16-token tiles
        p.n_fast = k->T_v / tok;
        p.n_mini = cdiv(k->n_sink, 16) + (k->T_k - p.n_fast * tok) / 16 + cdiv(k->n_kres, 16);
        p.N_f = (int64_t)U * p.n_fast;
        p.N_m = (int64_t)U * p.n_mini;
        split_pools(p.N_f, p.n_fast, p.N_m, p.n_mini, wpc, nsm, p.C_f, p.C_m, p.n_fast ? U : 0, p.n_mini ? U : 0);
    } else {
        // generic chunks of the whole sequence (CUDA cores)
        p.n_gen = L;
        const double kGen = 1.0;
        double best = 1e300;
        const int64_t gmax = std::max<int64_t>(32, cdiv(L, 32) * 32);
        int64_t cands[40];
        int nc = 0;
        for (int64_t ch = 32; ch <= 256 && ch < gmax; ch += 32) cands[nc++] = ch;
        for (int64_t ch = 512; ch < gmax && nc < 39; ch *= 2) cands[nc++] = ch;
        cands[nc++] = gmax;
        for (int ci = 0; ci < nc; ci++) {
            const int64_t chunk = cands[ci];
            const int64_t ngc = cdiv(L, chunk);
            const int64_t cg = cdiv((int64_t)U * ngc, wpc);
            if (cg > 4 * (int64_t)nsm && chunk < gmax) continue;
            const double est = (double)cdiv(cg, nsm) * (double)std::min(chunk, L) * kGen + 1e-3 * cg;
            if (est < best) {
                best = est;
                p.C_g = (int)cg;
                p.n_gc = (int)ngc;
                p.gen_chunk = chunk;
            }
        }
    }
    if (!hit) {
        // slots per sequence
        int64_t max_slots = 0;
        for (int64_t u = 0; u < U; u++) {
            int64_t sl = pool_ctas_host(p.C_f, wpc, p.N_f, p.n_fast, u) +
                         pool_ctas_host(p.C_m, wpc, p.N_m, p.n_mini, u);
            if (p.n_gc > 0) sl += ((u + 1) * p.n_gc - 1) / wpc - (u * p.n_gc) / wpc + 1;
            max_slots = std::max(max_slots, sl);
        }
        // item indices of the tile pools stay 32-bit in the kernel
        const bool small = p.N_f < (1LL << 31) && p.N_m < (1LL << 31) && p.n_fast + p.n_mini < (1LL << 31) &&
                           (int64_t)p.U * p.n_gc < (1LL << 31);
        if (max_slots < 1 || max_slots > slot_bound(c) || p.C_f > max_pool_ctas(c) || p.C_m > max_pool_ctas(c) ||
            p.C_g > 4 * (int64_t)max_pool_ctas(c) || !small)
            return KVQ_ERR_UNSUPPORTED;
        p.max_slots = (int)max_slots;
        ce.key = key;
        ce.val = SchedVal{p.C_f, p.C_m, p.C_g, p.n_gc, p.max_slots, p.n_fast,
                          p.n_mini, p.N_f, p.N_m, p.n_gen, p.gen_chunk};
        ce.valid = true;
    }

    p.n_items = fast ? (int)(p.n_fast + p.n_mini) : p.n_gc;
    p.W_f = p.C_f * wpc;
    p.W_m = p.C_m * wpc;
    p.qN_f = p.W_f ? (int)(p.N_f / p.W_f) : 0;
    p.rN_f = p.W_f ? (int)(p.N_f % p.W_f) : 0;
    p.qN_m = p.W_m ? (int)(p.N_m / p.W_m) : 0;
    p.rN_m = p.W_m ? (int)(p.N_m % p.W_m) : 0;
    p.B = c->B;
    p.H_kv = c->H_kv;
    p.g = g;
    if (fast) {
        int sh = 0;
        while ((tok << sh) < c->G) sh++;
        p.tpp_shift = sh;
        sh = 0;
        while ((1 << sh) < c->G) sh++;
        p.g_shift = sh;
    }
    p.D = c->D;
    p.G = c->G;
    p.bits = c->bits;
    p.vbits = vbits_of(c);
    p.Gv = gv_of(c);
    p.v_tile = vtile_of(c);
    p.n_boost = kitty(c) ? c->n_boost : 0;
    p.kitty = kitty(c) ? 1 : 0;
    p.S_cap = c->S;
    p.cap_k = (int)cap_k(c);
    p.cap_v = (int)cap_v(c);
    p.R_local = kitty(c) ? c->R : 1;
    p.max_T = c->max_T;
    p.rope = c->rope;
    p.rope_base = c->rope_base > 0.0f ? c->rope_base : 10000.0f;
    p.nvfp4 = nvfp4(c) ? 1 : 0;
    p.nv_kms = p.nv_vms = (int)nvfp4_page_bytes(c);
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
    p.k_new = kn;
    p.v_new = vn;
    char *w = static_cast<char *>(ws);
    p.status = status_word ? status_word : reinterpret_cast<int32_t *>(w + wl.status);
    p.done = done;
    p.done_ctr = reinterpret_cast<unsigned int *>(w + wl.status + 16);  // in the status block
    p.slot_ctr = nullptr;  // dense caches: a CTA's slot follows from the schedule
    {
        const int64_t fresh = take_fresh(k);
        p.early_tiles = fast ? (int)std::min<int64_t>(p.n_fast, fresh / tok) : 0;
    }
    p.item_ctr = reinterpret_cast<unsigned long long *>(w + wl.item_ctr);
    p.partials = reinterpret_cast<float *>(w + wl.partials);
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

// The device address of page-locked host memory mapped into the current device's
// address space, or null (pageable memory, device memory, or no such mapping).
static const void *mapped_host(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

// Staging layout of kvq_decode_step_host: q, k_new, v_new, out, each 256-byte aligned.
static size_t step_io_part(size_t n) { return (n + 255) & ~(size_t)255; }

size_t kvq_step_io_bytes(const kvq_config *c) {
    if (kvq_config_check(c) != KVQ_OK) return 0;
    const size_t nq = (size_t)c->B * c->H_q * c->D * 2, nk = (size_t)c->B * c->H_kv * c->D * 2;
    return 2 * step_io_part(nq) + 2 * step_io_part(nk);
}

int kvq_decode_step_host(const kvq_config *c, kvq_cache *k, const uint16_t *q, const uint16_t *k_new,
                         const uint16_t *v_new, uint16_t *out, void *io, size_t io_bytes, void *ws,
                         size_t ws_bytes, int *flushed_k, int *flushed_v, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if (!k || !q || !k_new || !v_new || !out || !io || ((uintptr_t)io & 255)) return KVQ_ERR_INVALID_ARG;
    if (io_bytes < kvq_step_io_bytes(c)) return KVQ_ERR_WORKSPACE;
    const size_t nq = (size_t)c->B * c->H_q * c->D * 2, nk = (size_t)c->B * c->H_kv * c->D * 2;
    char *d = static_cast<char *>(io);
    uint16_t *dq = reinterpret_cast<uint16_t *>(d);
    uint16_t *dk = reinterpret_cast<uint16_t *>(d + step_io_part(nq));
    uint16_t *dv = reinterpret_cast<uint16_t *>(d + step_io_part(nq) + step_io_part(nk));
    uint16_t *dout = reinterpret_cast<uint16_t *>(d + step_io_part(nq) + 2 * step_io_part(nk));
    cudaStream_t st = (cudaStream_t)stream;
    // Page-locked host buffers mapped into the device's address space are read and
    // written by the kernels themselves (plain loads and stores; no bulk copy touches
    // them); other host memory goes through one cudaMemcpyAsync per buffer.
    const void *mq = mapped_host(q), *mk = mapped_host(k_new), *mv = mapped_host(v_new);
    void *mo = const_cast<void *>(mapped_host(out));
    const bool direct = mq && mk && mv && mo && aligned16(mq) && aligned16(mk) && aligned16(mv) && aligned16(mo);
    if (direct) {
        dq = static_cast<uint16_t *>(const_cast<void *>(mq));
        dk = static_cast<uint16_t *>(const_cast<void *>(mk));
        dv = static_cast<uint16_t *>(const_cast<void *>(mv));
        dout = static_cast<uint16_t *>(mo);
    } else if (cudaMemcpyAsync(dk, k_new, nk, cudaMemcpyDefault, st) != cudaSuccess ||
               cudaMemcpyAsync(dv, v_new, nk, cudaMemcpyDefault, st) != cudaSuccess ||
               cudaMemcpyAsync(dq, q, nq, cudaMemcpyDefault, st) != cudaSuccess) {
        return KVQ_ERR_CUDA;
    }
    if ((e = kvq_append_decode(c, k, dk, dv, dq, dout, ws, ws_bytes, nullptr, stream))) return e;
    if ((e = kvq_flush_group(c, k, flushed_k, flushed_v, stream))) return e;
    if (!direct && cudaMemcpyAsync(out, dout, nq, cudaMemcpyDefault, st) != cudaSuccess) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int kvq_decode_step_host_wait(const kvq_config *c, kvq_cache *k, const uint16_t *q, const uint16_t *k_new,
                              const uint16_t *v_new, uint16_t *out, unsigned int *done, void *ws, size_t ws_bytes,
                              int *flushed_k, int *flushed_v, void *stream) {
    int e = kvq_config_check(c);
    if (e) return e;
    if (!k || !q || !k_new || !v_new || !out || !done || ((uintptr_t)done & 3)) return KVQ_ERR_INVALID_ARG;
    const void *mq = mapped_host(q), *mk = mapped_host(k_new), *mv = mapped_host(v_new);
    void *mo = const_cast<void *>(mapped_host(out));
    unsigned int *md = static_cast<unsigned int *>(const_cast<void *>(mapped_host(done)));
    if (!mq || !mk || !mv || !mo || !md || !aligned16(mq) || !aligned16(mk) || !aligned16(mv) || !aligned16(mo))
        return KVQ_ERR_INVALID_ARG;
    __atomic_store_n(done, 0u, __ATOMIC_RELEASE);  // before the launch that counts into it
    if ((e = append_decode_impl(c, k, static_cast<const uint16_t *>(mk), static_cast<const uint16_t *>(mv),
                                static_cast<const uint16_t *>(mq), static_cast<uint16_t *>(mo), ws, ws_bytes,
                                nullptr, stream, md)))
        return e;
    if ((e = kvq_flush_group(c, k, flushed_k, flushed_v, stream))) return e;
    // Every sequence is combined by exactly one CTA, which counts it after its output
    // stores; the last one releases U to *done.  Spin on it, then (past a bound) fall
    // back to the stream.
    const unsigned int want = (unsigned int)units(c);
    const auto t0 = std::chrono::steady_clock::now();
    for (uint32_t spins = 0; __atomic_load_n(done, __ATOMIC_ACQUIRE) < want; spins++) {
        if ((spins & 1023u) == 1023u && std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(200)) {
            if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KVQ_ERR_CUDA;
            return __atomic_load_n(done, __ATOMIC_ACQUIRE) == want ? KVQ_OK : KVQ_ERR_DEVICE;
        }
    }
    return KVQ_OK;
}

}  // extern "C"

namespace kvq {
namespace host {

int decode_check_args(const kvq_config *c, const kvq_cache *k, const uint16_t *q, const uint16_t *out) {
    int e = kvq_config_check(c);
    if (e) return e;
    if ((e = check_cache_ptrs(c, k))) return e;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
    const int64_t L = k->n_sink + k->T_k + k->n_kres;
    const int64_t Lv = k->n_sink + k->T_v + k->n_vres + k->n_local;
    if (L < 1 || L != Lv) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

size_t decode_ws_counter_end(const kvq_config *c) { return ws_layout(c).partials; }

int decode_attn_status(const kvq_config *c, const kvq_cache *k, const uint16_t *q, uint16_t *out, void *ws,
                       size_t ws_bytes, void *stream, int32_t *status_word) {
    return decode_impl(c, k, q, out, ws, ws_bytes, stream, nullptr, nullptr, status_word);
}

}  // namespace host
}  // namespace kvq
