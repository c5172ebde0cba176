// kvq_paged.cu -- the C ABI of the paged cache (kvq_paged_* in include/kvq.h).
//
// Kitty Sec. 4.1 stores every quantization group of G tokens as a page, apart from the
// fp16 sink and residual buffers, after PagedAttention; the KIVI notes describe
// PagedAttention as cutting the cache into fixed blocks reached through a mapping
// table.  Here a physical page holds one group of all H_kv heads of one batch slot, the
// caller's page table maps (slot, logical page) to it, and every batch slot has its own
// length.  The host keeps a mirror of the device lengths and updates it at enqueue time,
// exactly as the kernels update the device copy.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "kvq.h"
#include "kvq_host.h"
#include "kvq_internal.h"

using namespace kvq;
using namespace kvq::host;

namespace {

// Per-sequence slot ids a paged decode may need (the CTAs of both pools touching one
// sequence, bounded by two waves) and the pool of partials.
inline int paged_smax() { return 2 * num_sms() + 8; }

struct PagedWs {
    size_t status, slot_ctr, item_ctr, seq_slots, partials, total;
    int smax;
    int64_t cap;  // partial slots: CTA slots of up to two waves + two per sequence
};

PagedWs paged_ws_layout(const kvq_config *c) {
    PagedWs w;
    const int64_t U = units(c);
    const size_t ctr = (size_t)cdiv(U * 4, 256) * 256;
    w.smax = paged_smax();
    w.cap = (int64_t)2 * num_sms() * 2 * 8 + 2 * U;
    w.status = 0;
    w.slot_ctr = 256;
    w.item_ctr = w.slot_ctr + ctr;
    w.seq_slots = w.item_ctr + 2 * ctr;
    w.partials = w.seq_slots + (size_t)cdiv(U * w.smax * 4, 256) * 256;
    w.total = w.partials + (size_t)w.cap * 4 * (c->D + 4) * 4;
    return w;
}

int paged_cfg_check(const kvq_config *c) {
    const int e = kvq_config_check(c);
    if (e) return e;
    if (kitty(c) || c->rope || !fast_supported(c) || c->B > KVQ_PAGED_MAX_B) return KVQ_ERR_UNSUPPORTED;
    if (c->max_T / c->G < 1) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

int64_t max_pages(const kvq_config *c) { return c->max_T / c->G; }

int check_paged(const kvq_config *c, const kvq_paged *pc) {
    int e = paged_cfg_check(c);
    if (e) return e;
    if (!pc || !pc->lens_host) return KVQ_ERR_INVALID_ARG;
    const void *need[] = {pc->k_codes, pc->k_meta, pc->v_codes, pc->v_meta, pc->page_table,
                          pc->k_res, pc->v_res, pc->lens};
    for (const void *p : need)
        if (!p || !aligned16(p)) return KVQ_ERR_INVALID_ARG;
    if (c->S > 0 && (!pc->k_sink || !pc->v_sink || !aligned16(pc->k_sink) || !aligned16(pc->v_sink)))
        return KVQ_ERR_INVALID_ARG;
    if (pc->n_pages < 0 || pc->n_pages > (int64_t)INT32_MAX) return KVQ_ERR_INVALID_ARG;
    for (int b = 0; b < c->B; b++) {
        const int32_t *l = pc->lens_host + 4 * b;
        if (l[3] != 0 && l[3] != 1) return KVQ_ERR_INVALID_ARG;
        if (!l[3]) continue;
        if (l[0] < 0 || l[0] > c->S || l[1] < 0 || l[1] % c->G || l[1] > c->max_T || l[2] < 0 || l[2] > c->R)
            return KVQ_ERR_INVALID_ARG;
    }
    return KVQ_OK;
}

PageMap page_map(const kvq_config *c, const kvq_paged *pc) {
    PageMap m;
    memset(&m, 0, sizeof(m));
    m.ptab = pc->page_table;
    m.ptab_stride = (int)max_pages(c);
    m.H_kv = c->H_kv;
    m.n_pages = pc->n_pages;
    m.status = pc->status;
    return m;
}

QuantKParams qk_paged(const kvq_config *c, const kvq_paged *pc) {
    QuantKParams p;
    memset(&p, 0, sizeof(p));
    p.max_T = c->max_T;
    p.D = c->D;
    p.G = c->G;
    p.k_codes = pc->k_codes;
    p.k_meta = pc->k_meta;
    p.status = pc->status;
    p.pm = page_map(c, pc);
    return p;
}

QuantVParams qv_paged(const kvq_config *c, const kvq_paged *pc) {
    QuantVParams p;
    memset(&p, 0, sizeof(p));
    p.max_T = c->max_T;
    p.D = c->D;
    p.G = c->G;
    p.Gv = gv_of(c);
    p.TV = vtile_of(c);
    p.v_codes = pc->v_codes;
    p.v_meta = pc->v_meta;
    p.status = pc->status;
    p.pm = page_map(c, pc);
    return p;
}

// Rows [r0, r0 + n) of a one-sequence source [H_kv][L0][D] -> rows [0, n) of batch
// slot b's buffer [U][rows][D].
cudaError_t copy_slot_rows(const kvq_config *c, const uint16_t *src, int64_t L0, int64_t r0, uint16_t *dst,
                           int64_t rows, int b, int64_t n, cudaStream_t st) {
    CopyRowsParams p;
    p.src = src;
    p.dst = dst + (size_t)b * c->H_kv * rows * c->D;
    p.src_rows = L0;
    p.src_r0 = r0;
    p.dst_rows = rows;
    p.dst_r0 = 0;
    p.n_rows = n;
    p.U = c->H_kv;
    p.D = c->D;
    return launch_copy_rows(p, st);
}

cudaError_t set_lens(const kvq_paged *pc, int b, int v0, int v1, int v2, int v3, cudaStream_t st) {
    SetLensParams p;
    p.lens = pc->lens;
    p.b = b;
    p.v0 = v0;
    p.v1 = v1;
    p.v2 = v2;
    p.v3 = v3;
    return launch_set_lens(p, st);
}

// CTAs of a pool (C CTAs of wpc warps, N items) that hold items [a, a + n).
int64_t ctas_touching(int64_t C, int wpc, int64_t N, int64_t a, int64_t n) {
    if (n == 0 || C == 0) return 0;
    const int64_t W = C * wpc;
    auto warp_of = [&](int64_t x) { return std::min(W - 1, ((x + 1) * W - 1) / N); };
    return warp_of(a + n - 1) / wpc - warp_of(a) / wpc + 1;
}

}  // namespace

extern "C" {

size_t kvq_paged_bytes(const kvq_config *c, int64_t n_pages, int which) {
    if (paged_cfg_check(c) != KVQ_OK || n_pages < 0) return 0;
    const size_t P = (size_t)n_pages, H = (size_t)c->H_kv, D = c->D, G = c->G, U = (size_t)units(c);
    switch (which) {
        case 0: return P * H * (G / kfpi(c)) * D * 4;
        case 3: return P * H * D * 4;
        case 4: return P * H * (D / vfpi(c)) * G * 4;
        case 5: return P * H * G * (D / gv_of(c)) * 4;
        case 6: return U * (size_t)c->S * D * 2;
        case 7: return U * (size_t)c->R * D * 2;
        case 8: return U * (size_t)c->R * D * 2;
        case 10: return (size_t)c->B * 16;
        case 11: return (size_t)c->B * (size_t)max_pages(c) * 4;
    }
    return 0;
}

int kvq_paged_init(const kvq_config *c, kvq_paged *pc, void *stream) {
    const int e = paged_cfg_check(c);
    if (e) return e;
    if (!pc || !pc->lens || !pc->lens_host) return KVQ_ERR_INVALID_ARG;
    memset(pc->lens_host, 0, (size_t)c->B * 16);
    return status_of(cudaMemsetAsync(pc->lens, 0, (size_t)c->B * 16, (cudaStream_t)stream));
}

int kvq_paged_prefill(const kvq_config *c, kvq_paged *pc, int b, const uint16_t *k, const uint16_t *v,
                      int64_t L0, void *stream) {
    int e = check_paged(c, pc);
    if (e) return e;
    if (b < 0 || b >= c->B || pc->lens_host[4 * b + 3]) return KVQ_ERR_INVALID_ARG;
    if (!k || !v || !aligned16(k) || !aligned16(v) || L0 < 1) return KVQ_ERR_INVALID_ARG;
    const int64_t ns = std::min<int64_t>(c->S, L0), rest = L0 - ns, T = rest / c->G * c->G, res = rest - T;
    if (T > c->max_T) return KVQ_ERR_CAPACITY;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t ce = cudaSuccess;
    if (ns > 0) ce = copy_slot_rows(c, k, L0, 0, pc->k_sink, c->S, b, ns, st);
    if (ce == cudaSuccess && ns > 0) ce = copy_slot_rows(c, v, L0, 0, pc->v_sink, c->S, b, ns, st);
    if (ce == cudaSuccess && T > 0) {
        QuantKParams p = qk_paged(c, pc);
        p.src = k;
        p.src_ustride = L0 * c->D;
        p.src_t0 = ns;
        p.n_pages = T / c->G;
        p.U = c->H_kv;
        p.pm.n_seq = 1;
        p.pm.seq[0] = (int16_t)b;
        p.pm.lp0[0] = 0;
        ce = launch_quant_k(p, c->bits, false, st);
        if (ce == cudaSuccess) {
            QuantVParams q = qv_paged(c, pc);
            q.src = v;
            q.src_ustride = L0 * c->D;
            q.src_t0 = ns;
            q.n_tok = T;
            q.tok0 = 0;
            q.U = c->H_kv;
            q.pm = p.pm;
            ce = launch_quant_v(q, vbits_of(c), st);
        }
    }
    if (ce == cudaSuccess && res > 0) ce = copy_slot_rows(c, k, L0, ns + T, pc->k_res, c->R, b, res, st);
    if (ce == cudaSuccess && res > 0) ce = copy_slot_rows(c, v, L0, ns + T, pc->v_res, c->R, b, res, st);
    if (ce == cudaSuccess) ce = set_lens(pc, b, (int)ns, (int)T, (int)res, 1, st);
    if (ce != cudaSuccess) return KVQ_ERR_CUDA;
    int32_t *l = pc->lens_host + 4 * b;
    l[0] = (int32_t)ns;
    l[1] = (int32_t)T;
    l[2] = (int32_t)res;
    l[3] = 1;
    return KVQ_OK;
}

int kvq_paged_append(const kvq_config *c, kvq_paged *pc, const uint16_t *kn, const uint16_t *vn, void *stream) {
    int e = check_paged(c, pc);
    if (e) return e;
    if (!kn || !vn || !aligned16(kn) || !aligned16(vn)) return KVQ_ERR_INVALID_ARG;
    for (int b = 0; b < c->B; b++) {
        const int32_t *l = pc->lens_host + 4 * b;
        if (l[3] && l[0] >= c->S && l[2] >= c->R) return KVQ_ERR_CAPACITY;
    }
    PagedAppendParams p;
    p.k_new = kn;
    p.v_new = vn;
    p.k_sink = pc->k_sink;
    p.v_sink = pc->v_sink;
    p.k_res = pc->k_res;
    p.v_res = pc->v_res;
    p.lens = pc->lens;
    p.status = pc->status;
    p.B = c->B;
    p.H_kv = c->H_kv;
    p.D = c->D;
    p.S = c->S;
    p.R = c->R;
    if (launch_paged_append(p, (cudaStream_t)stream) != cudaSuccess) return KVQ_ERR_CUDA;
    for (int b = 0; b < c->B; b++) {
        int32_t *l = pc->lens_host + 4 * b;
        if (!l[3]) continue;
        if (l[0] < c->S) l[0]++;
        else l[2]++;
    }
    return KVQ_OK;
}

int kvq_paged_flush_plan(const kvq_config *c, const kvq_paged *pc, int32_t *seqs, int *n) {
    int e = check_paged(c, pc);
    if (e) return e;
    if (!n) return KVQ_ERR_INVALID_ARG;
    int k = 0;
    for (int b = 0; b < c->B; b++) {
        const int32_t *l = pc->lens_host + 4 * b;
        if (l[3] && l[2] == c->R) {
            if (seqs) seqs[k] = b;
            k++;
        }
    }
    *n = k;
    return KVQ_OK;
}

int kvq_paged_flush(const kvq_config *c, kvq_paged *pc, int *n_flushed, void *stream) {
    int e = check_paged(c, pc);
    if (e) return e;
    std::vector<int> list;
    for (int b = 0; b < c->B; b++) {
        const int32_t *l = pc->lens_host + 4 * b;
        if (l[3] && l[2] == c->R) {
            if ((int64_t)l[1] + c->R > c->max_T) return KVQ_ERR_CAPACITY;
            list.push_back(b);
        }
    }
    cudaStream_t st = (cudaStream_t)stream;
    for (size_t i0 = 0; i0 < list.size(); i0 += kMaxListSeq) {
        const int n = (int)std::min<size_t>(kMaxListSeq, list.size() - i0);
        QuantKParams p = qk_paged(c, pc);
        p.src = pc->k_res;
        p.src_ustride = (int64_t)c->R * c->D;
        p.src_t0 = 0;
        p.n_pages = c->R / c->G;
        p.U = n * c->H_kv;
        p.pm.n_seq = n;
        p.pm.src_by_seq = 1;
        for (int i = 0; i < n; i++) {
            const int b = list[i0 + i];
            p.pm.seq[i] = (int16_t)b;
            p.pm.lp0[i] = pc->lens_host[4 * b + 1] / c->G;
        }
        QuantVParams q = qv_paged(c, pc);
        q.src = pc->v_res;
        q.src_ustride = (int64_t)c->R * c->D;
        q.src_t0 = 0;
        q.n_tok = c->R;
        q.tok0 = 0;
        q.U = p.U;
        q.pm = p.pm;
        p.pm.lens = pc->lens;  // the key kernel commits T += R, n_res = 0 of each slot
        if (launch_quant_v(q, vbits_of(c), st) != cudaSuccess) return KVQ_ERR_CUDA;
        if (launch_quant_k(p, c->bits, false, st) != cudaSuccess) return KVQ_ERR_CUDA;
        for (int i = 0; i < n; i++) {
            int32_t *l = pc->lens_host + 4 * list[i0 + i];
            l[1] += c->R;
            l[2] = 0;
        }
    }
    if (n_flushed) *n_flushed = (int)list.size();
    return KVQ_OK;
}

int kvq_paged_release(const kvq_config *c, kvq_paged *pc, int b, void *stream) {
    int e = check_paged(c, pc);
    if (e) return e;
    if (b < 0 || b >= c->B) return KVQ_ERR_INVALID_ARG;
    if (set_lens(pc, b, 0, 0, 0, 0, (cudaStream_t)stream) != cudaSuccess) return KVQ_ERR_CUDA;
    memset(pc->lens_host + 4 * b, 0, 16);
    return KVQ_OK;
}

size_t kvq_paged_workspace_bytes(const kvq_config *c) {
    if (paged_cfg_check(c) != KVQ_OK) return 0;
    return paged_ws_layout(c).total;
}

int kvq_paged_decode_attn(const kvq_config *c, const kvq_paged *pc, const uint16_t *q, uint16_t *out, void *ws,
                          size_t ws_bytes, void *stream) {
    int e = check_paged(c, pc);
    if (e) return e;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
    const PagedWs wl = paged_ws_layout(c);
    if (!ws || !aligned16(ws) || ws_bytes < wl.total) return KVQ_ERR_WORKSPACE;

    const int B = c->B, H = c->H_kv, U = (int)units(c), nsm = num_sms();
    const int tok = 256 / c->bits;
    const int wpc = decode_warps_per_cta(c->bits, vbits_of(c), false, 0, true);
    // items per batch slot: packed tiles and 16-token fp16 tiles
    std::vector<int64_t> nf(B), nm(B);
    int64_t Sf = 0, Sm = 0, uf = 0, um = 0;
    for (int b = 0; b < B; b++) {
        const int32_t *l = pc->lens_host + 4 * b;
        nf[b] = l[3] ? l[1] / tok : 0;
        nm[b] = l[3] ? cdiv(l[0], 16) + cdiv(l[2], 16) : 0;
        Sf += nf[b];
        Sm += nm[b];
        uf += nf[b] ? H : 0;
        um += nm[b] ? H : 0;
    }
    const int64_t N_f = H * Sf, N_m = H * Sm;
    if (N_f + N_m == 0) return KVQ_OK;  // no active sequence
    if (N_f >= (1LL << 31) || N_m >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;

    DecodeParams p;
    memset(&p, 0, sizeof(p));
    p.U = U;
    p.wpc = wpc;
    split_pools(N_f, N_f, N_m, N_m, wpc, nsm, p.C_f, p.C_m, uf, um);
    if (p.C_f + p.C_m > 2 * nsm || wpc > 8) return KVQ_ERR_UNSUPPORTED;
    // slot ids per sequence: the CTAs of both pools that hold its items
    int64_t max_slots = 0, af = 0, am = 0;
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            const int64_t sl = ctas_touching(p.C_f, wpc, N_f, H * af + h * nf[b], nf[b]) +
                               ctas_touching(p.C_m, wpc, N_m, H * am + h * nm[b], nm[b]);
            max_slots = std::max(max_slots, sl);
        }
        af += nf[b];
        am += nm[b];
    }
    if (max_slots > wl.smax) return KVQ_ERR_UNSUPPORTED;
    p.smax = wl.smax;
    p.mid_base = (p.C_f + p.C_m) * 2 * wpc;
    p.max_slots = p.mid_base + 2 * U;  // pool ids in use: CTA slots, then two per sequence
    if (p.max_slots > wl.cap) return KVQ_ERR_UNSUPPORTED;
    p.n_fast = N_f;
    p.n_mini = N_m;
    p.N_f = N_f;
    p.N_m = N_m;
    p.W_f = p.C_f * wpc;
    p.W_m = p.C_m * wpc;
    p.qN_f = p.W_f ? (int)(N_f / p.W_f) : 0;
    p.rN_f = p.W_f ? (int)(N_f % p.W_f) : 0;
    p.qN_m = p.W_m ? (int)(N_m / p.W_m) : 0;
    p.rN_m = p.W_m ? (int)(N_m % p.W_m) : 0;
    p.B = B;
    p.H_kv = H;
    p.g = c->H_q / c->H_kv;
    int sh = 0;
    while ((tok << sh) < c->G) sh++;
    p.tpp_shift = sh;
    sh = 0;
    while ((1 << sh) < c->G) sh++;
    p.g_shift = sh;
    p.D = c->D;
    p.G = c->G;
    p.bits = c->bits;
    p.vbits = vbits_of(c);
    p.Gv = gv_of(c);
    p.v_tile = vtile_of(c);
    p.S_cap = c->S;
    p.cap_k = c->R;
    p.cap_v = c->R;
    p.R_local = 1;
    p.max_T = c->max_T;
    p.k_codes = pc->k_codes;
    p.k_meta = pc->k_meta;
    p.v_codes = pc->v_codes;
    p.v_meta = pc->v_meta;
    p.k_sink = pc->k_sink;
    p.v_sink = pc->v_sink;
    p.k_res = pc->k_res;
    p.v_res = pc->v_res;
    p.q = q;
    p.out = out;
    p.ptab = pc->page_table;
    p.ptab_stride = (int)max_pages(c);
    p.n_pages = pc->n_pages;
    p.lens = pc->lens;
    char *w = static_cast<char *>(ws);
    p.status = reinterpret_cast<int32_t *>(w + wl.status);
    p.slot_ctr = reinterpret_cast<int32_t *>(w + wl.slot_ctr);
    p.item_ctr = reinterpret_cast<unsigned long long *>(w + wl.item_ctr);
    p.seq_slots = reinterpret_cast<int32_t *>(w + wl.seq_slots);
    p.partials = reinterpret_cast<float *>(w + wl.partials);
    return status_of(launch_decode(p, true, (cudaStream_t)stream));
}

int kvq_paged_read_status(const kvq_paged *pc, void *ws, int32_t *dev_status, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    int32_t acc = 0, v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
    int32_t *words[2] = {static_cast<int32_t *>(ws), pc ? pc->status : nullptr};
    for (int32_t *wd : words) {
        if (!wd) continue;
        if (cudaMemcpy(&v, wd, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
        acc |= v;
        if (v && cudaMemset(wd, 0, 4) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    if (dev_status) *dev_status = acc;
    return acc ? KVQ_ERR_DEVICE : KVQ_OK;
}

}  // extern "C"
