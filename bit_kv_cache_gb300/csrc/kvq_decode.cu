// kvq_decode.cu -- single-query / GQA decode attention over the packed KV cache.
//
//   out[b][h] = softmax_t( q[b][h] . K_t / sqrt(D) ) . V_t
// with K_t, V_t dequantized as code*scale + min in registers (KIVI notes, Step 3/4:
// the kernel consumes packed codes plus scales and never writes an fp16 copy of
// the cache; BitDecoding Sec. II: softmax(Q D(K')^T) D(V')).
//
// Work split (flash-decoding style): each sequence (b, h_kv) is cut into tiles of
// TOK tokens; warps own disjoint token ranges and keep an online-softmax state
// (running max m, sum l, unnormalized output o) in log2 units.  A CTA merges its
// warps' states in shared memory into one partial; the last CTA of a sequence (an
// atomic ticket, no spin-wait) combines the partials with the log-sum-exp rule and
// writes fp16 out.
//
// Tensor-core tiles (all g <= 4 query heads of a KV head at once in one mma N=8
// tile -- the BitDecoding query transformation, Sec. V-A):
//   QK:  S[token][col] += Kcodes[token][ch] * q'[ch][col],  q' = q * scale_k * log2e/sqrt(D)
//        split in fp16 hi (column 2h) and lo (column 2h+1) parts of head h, so the
//        folded query keeps 22 significant bits
//        plus a per-head constant sum_ch q*min_k (keys are per-channel, so the
//        scale folds into q and the min into a constant; one page = one group).
//   PV:  O[ch][head] += Vcodes[ch][token] * p'[token][head],  p' = p * scale_v(token)
//        plus sum_t p*min_v(token) per head (values are per-token).
// The code operand is built from the packed words with one AND per two codes:
// a 2-bit (4-bit) code c sitting in the low 10 bits of a 16-bit half is the fp16
// subnormal c * 2^(k-24) (k = its bit offset), exactly representable, so the
// tensor core multiplies exact integer codes; the 2^k factor is a constant per
// mma (row set) and is removed in fp32 afterwards.  ldmatrix delivers each packed
// word to exactly one lane; the mma row <-> token (or channel) map is chosen so
// that a lane's words hold all of its rows (keys: row g <-> token 16g+j of the
// tile; values: row g <-> channel 16g+j), so nothing is loaded twice.
// Packed tiles stream global -> shared with cp.async.bulk on a per-warp
// double-buffered mbarrier pipeline.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
__host__ __device__ __forceinline__ int64_t kvq_min64(int64_t a, int64_t b) { return a < b ? a : b; }
}  // namespace kvq

#include "kvq_decode_fast.cuh"

namespace kvq {

constexpr int KVQ_DEV_BAD_STATE_BIT = 2;

// Per-warp shared memory of the generic-only kernel: [partial][q buffer fp16 [8][D]].
__host__ __device__ inline int gen_warp_bytes(int D) { return (part_bytes(D) + 8 * D * 2 + 127) & ~127; }

// ---------------------------------------------------------------------------------
// Generic path: one token per lane for QK, one token per step for PV (CUDA cores,
// fp32).  Handles sink, fp16 buffers and packed tokens of any layout the fast path
// does not take.  State: m[h], l[h] (lane-partial), o[h][DPL] for the lane's
// channels lane*DPL .. lane*DPL+DPL-1.
// ---------------------------------------------------------------------------------
template <int DPL>
struct GenState {
    float m[8], l[8], o[8][DPL];
};

__device__ __forceinline__ void load_k8(const DecodeParams &p, int u, int64_t tl, int d, float (&kv)[8]) {
    const int D = p.D;
    if (tl < p.n_sink) {
        uint4 w = *reinterpret_cast<const uint4 *>(p.k_sink + ((size_t)u * p.S_cap + tl) * D + d);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 f = unpack_half2(ww[i]);
            kv[2 * i] = f.x;
            kv[2 * i + 1] = f.y;
        }
        return;
    }
    int64_t tk = tl - p.n_sink;
    if (tk < p.T_k) {
        const int kb = p.kitty ? 2 : p.bits, fpi = 32 / kb;
        const int64_t page = tk / p.G;
        const int32_t *wp = p.k_codes + ((size_t)u * (p.max_T / fpi) + tk / fpi) * D + d;
        const uint32_t *mp = reinterpret_cast<const uint32_t *>(p.k_meta) +
                             ((size_t)u * (p.max_T / p.G) + page) * D + d;
        const int sh = kb * (int)(tk % fpi);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t code = ((uint32_t)wp[i] >> sh) & ((1u << kb) - 1);
            if (p.kitty && p.n_boost) {
                int slot = p.k_bidx[((size_t)u * (p.max_T / p.G) + page) * D + d + i];
                if (slot < p.n_boost) {
                    uint32_t h = (uint32_t)p.k_hi[((size_t)u * (p.max_T / 16) + tk / 16) * p.n_boost + slot];
                    code |= ((h >> (2 * (tk % 16))) & 3u) << 2;
                }
            }
            float2 sm = unpack_half2(mp[i]);
            kv[i] = (float)code * sm.x + sm.y;
        }
        return;
    }
    int64_t r = tk - p.T_k;
    uint4 w = *reinterpret_cast<const uint4 *>(p.k_res + ((size_t)u * p.cap_k + r) * D + d);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 f = unpack_half2(ww[i]);
        kv[2 * i] = f.x;
        kv[2 * i + 1] = f.y;
    }
}

template <int DPL>
__device__ __forceinline__ void load_v(const DecodeParams &p, int u, int64_t tl, int d, float (&vv)[DPL]) {
    const int D = p.D;
    const uint16_t *row = nullptr;
    if (tl < p.n_sink) {
        row = p.v_sink + ((size_t)u * p.S_cap + tl) * D;
    } else {
        int64_t tv = tl - p.n_sink;
        if (tv < p.T_v) {
            const int fpi = 32 / p.bits;
            const int64_t page = tv / p.G, tin = tv % p.G;
#pragma unroll
            for (int i = 0; i < DPL; i++) {
                const int dd = d + i;
                uint32_t w = (uint32_t)p.v_codes[(((size_t)u * (p.max_T / p.G) + page) * (D / fpi) + dd / fpi) * p.G + tin];
                uint32_t code = (w >> (p.bits * (dd % fpi))) & ((1u << p.bits) - 1);
                float2 sm = unpack_half2(reinterpret_cast<const uint32_t *>(p.v_meta)[((size_t)u * p.max_T + tv) * (D / p.Gv) + dd / p.Gv]);
                vv[i] = (float)code * sm.x + sm.y;
            }
            return;
        }
        int64_t r = tv - p.T_v;
        if (r < p.n_vres) {
            row = p.v_res + ((size_t)u * p.cap_v + r) * D;
        } else {
            int64_t slot = (p.local_head + (r - p.n_vres)) % p.R_local;
            row = p.v_local + ((size_t)u * p.R_local + slot) * D;
        }
    }
#pragma unroll
    for (int i = 0; i < DPL; i++) vv[i] = h2f(row[d + i]);
}

template <int DPL>
__device__ void generic_range(const DecodeParams &p, int u, const uint16_t *q_w, int64_t a, int64_t b,
                              GenState<DPL> &st) {
    const int lane = threadIdx.x & 31, D = p.D, g = p.g;
    const float C = kLog2e * rsqrtf((float)D);
    for (int64_t base = a; base < b; base += 32) {
        const int64_t j = base + lane;
        const bool valid = j < b;
        const int64_t tl = j < p.n_sink ? j : j + p.n_fast * (p.bits == 2 ? 128 : 64);
        float z[8];
#pragma unroll
        for (int h = 0; h < 8; h++) z[h] = 0.f;
        if (valid) {
            for (int d = 0; d < D; d += 8) {
                float kv[8];
                load_k8(p, u, tl, d, kv);
#pragma unroll
                for (int h = 0; h < 8; h++) {
                    if (h < g) {
                        const uint4 qq = *reinterpret_cast<const uint4 *>(q_w + h * D + d);
                        const float2 q0 = unpack_half2(qq.x), q1 = unpack_half2(qq.y);
                        const float2 q2 = unpack_half2(qq.z), q3 = unpack_half2(qq.w);
                        z[h] += q0.x * kv[0] + q0.y * kv[1] + q1.x * kv[2] + q1.y * kv[3] +
                                q2.x * kv[4] + q2.y * kv[5] + q3.x * kv[6] + q3.y * kv[7];
                    }
                }
            }
        }
        float pz[8];
#pragma unroll
        for (int h = 0; h < 8; h++) {
            if (h >= g) {
                pz[h] = 0.f;
                continue;
            }
            float zz = valid ? z[h] * C : -INFINITY;
            float mx = zz;
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mnew = fmaxf(st.m[h], mx);
            const float alpha = exp2f(st.m[h] - mnew);  // m = -inf initially -> 0
            st.m[h] = mnew;
            st.l[h] *= alpha;
#pragma unroll
            for (int i = 0; i < DPL; i++) st.o[h][i] *= alpha;
            pz[h] = valid ? exp2f(zz - mnew) : 0.f;
            st.l[h] += pz[h];
        }
        const int nt = (int)kvq_min64(32, b - base);
        for (int tt = 0; tt < nt; tt++) {
            const int64_t jj = base + tt;
            const int64_t tlv = jj < p.n_sink ? jj : jj + p.n_fast * (p.bits == 2 ? 128 : 64);
            float vv[DPL];
            load_v<DPL>(p, u, tlv, lane * DPL, vv);
#pragma unroll
            for (int h = 0; h < 8; h++) {
                if (h < g) {
                    const float ph = __shfl_sync(0xffffffffu, pz[h], tt);
#pragma unroll
                    for (int i = 0; i < DPL; i++) st.o[h][i] += ph * vv[i];
                }
            }
        }
    }
}

// Writes a warp's state as a partial [8][D+2] (o[0..D), m at D, l at D+1).
template <int DPL>
__device__ void generic_store(const DecodeParams &p, const GenState<DPL> &st, float *part) {
    const int lane = threadIdx.x & 31, D = p.D;
#pragma unroll
    for (int h = 0; h < 8; h++) {
        float l = st.l[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
        for (int i = 0; i < DPL; i++) part[h * prow(D) + lane * DPL + i] = st.o[h][i];
        if (lane == 0) {
            part[h * prow(D) + D] = st.m[h];
            part[h * prow(D) + D + 1] = l;
        }
    }
}

// ---------------------------------------------------------------------------------
// Schedule arithmetic (closed forms, identical on host and device).
// A pool of W = wpc * C warps cuts the sequence-major list of N = U * n items into
// ranges [a_k, a_{k+1}), a_k = floor(k * N / W).
// ---------------------------------------------------------------------------------
struct Pool {
    int64_t n, N, W;
    int c0;  // first CTA of the pool in the grid
    int C;
};
__device__ __forceinline__ int64_t pool_a(const Pool &P, int64_t k) { return k * P.N / P.W; }
__device__ __forceinline__ int64_t pool_warp_of(const Pool &P, int64_t x) {
    const int64_t k = ((x + 1) * P.W - 1) / P.N;
    return k < P.W - 1 ? k : P.W - 1;
}
// CTAs of the pool that hold items of sequence u (first via *first).
__device__ __forceinline__ int pool_ctas(const Pool &P, int wpc, int u, int *first) {
    if (P.n == 0 || P.C == 0) {
        *first = 0;
        return 0;
    }
    const int f = (int)(pool_warp_of(P, (int64_t)u * P.n) / wpc);
    const int l = (int)(pool_warp_of(P, (int64_t)(u + 1) * P.n - 1) / wpc);
    *first = f;
    return l - f + 1;
}
__device__ __forceinline__ int gen_ctas(const DecodeParams &p, int u, int *first) {
    if (p.n_gc == 0) {
        *first = 0;
        return 0;
    }
    const int f = (int)(((int64_t)u * p.n_gc) / p.wpc);
    const int l = (int)(((int64_t)(u + 1) * p.n_gc - 1) / p.wpc);
    *first = f;
    return l - f + 1;
}

__device__ __forceinline__ void load_q_gen(const DecodeParams &p, int u, uint16_t *q_w) {
    const int lane = threadIdx.x & 31, D = p.D;
    for (int i = lane; i < D; i += 32) {  // 8 heads x D halves in uint4 chunks
        const int h = (i * 8) / D, d = (i * 8) % D;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < p.g) v = *reinterpret_cast<const uint4 *>(p.q + ((size_t)u * p.g + h) * D + d);
        *reinterpret_cast<uint4 *>(q_w + h * D + d) = v;
    }
    __syncwarp();
}

// Weight tables of the merge and combine phases: behind warp 0's partial in a fast
// kernel (its slots are free once the tiles are done), else behind the warp regions.
constexpr int kGenTabFloats = 7168;
template <int BITS, bool KITTY, bool FAST, int NW>
__host__ __device__ inline int tab_offset(const DecodeParams &p) {
    if (FAST) return part_bytes(p.D);
    return NW * gen_warp_bytes(p.D);
}
template <int BITS, bool KITTY, bool FAST>
__host__ __device__ inline int tab_capacity(int n_boost, int D) {
    if (FAST) return (WarpSmem<BITS>(KITTY, n_boost).total - part_bytes(D)) / 4;
    return kGenTabFloats;
}

// ---------------------------------------------------------------------------------
// The kernel.  FAST: CTAs [0, C_f) fast warps, [C_f, C_f + C_m) mini warps.
// Otherwise: generic warps only.
// ---------------------------------------------------------------------------------
template <int BITS, bool KITTY, bool FAST, int DPL, int NW>
__global__ void __launch_bounds__(NW * 32, 1) decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_seg[NW][2];  // sequence of each warp segment (-1: none)
    __shared__ int s_last[24];    // sequences this CTA must combine
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, D = p.D, g = p.g;
    const int wbytes = FAST ? WarpSmem<BITS>(KITTY, p.n_boost).total : gen_warp_bytes(D);
    unsigned char *wbase = smem + warp * wbytes;
    float *part = reinterpret_cast<float *>(wbase);  // the warp's last partial, [8][D+2]
    int seg0 = -1, seg1 = -1;
    const Pool PF{p.n_fast, p.N_f, (int64_t)p.wpc * p.C_f, 0, p.C_f};
    const Pool PM{p.n_mini, p.N_m, (int64_t)p.wpc * p.C_m, p.C_f, p.C_m};
    int pool = 2;  // 0 fast, 1 mini, 2 generic
    if (FAST) pool = c < p.C_f ? 0 : 1;

    if (FAST) {
        const Pool &P = pool == 0 ? PF : PM;
        const int64_t k = (int64_t)(c - P.c0) * p.wpc + warp;
        const int64_t x0 = pool_a(P, k), x1 = pool_a(P, k + 1);
        // a warp range touches at most two sequences; a first segment followed by a
        // second one is parked in global scratch, the last one stays in shared memory
        int64_t x = x0;
        int nseg = 0;
        FastWarp<BITS, KITTY> fw(p, wbase);
        MiniWarp<BITS, KITTY> mw(p, wbase, 0);
        if (x < x1) {
            if (pool == 0) fw.init_bars();
            else mw.init_bars();
        }
        while (x < x1 && nseg < 2) {
            const int u = (int)(x / P.n);
            const int64_t e = kvq_min64(x1, (int64_t)(u + 1) * P.n);
            const bool more = e < x1;
            float *dst = more ? p.scratch + ((size_t)c * NW + warp) * (part_bytes(D) / 4) : part;
            if (pool == 0) fw.run(u, x - (int64_t)u * P.n, e - (int64_t)u * P.n, dst);
            else mw.run(u, x - (int64_t)u * P.n, e - (int64_t)u * P.n, dst);
            if (more) seg0 = u;
            else seg1 = u;
            x = e;
            nseg++;
        }
    } else {
        // ---- generic warp: one chunk of one sequence ----
        const int64_t j = (int64_t)c * p.wpc + warp;
        GenState<DPL> st;
#pragma unroll
        for (int h = 0; h < 8; h++) {
            st.m[h] = -INFINITY;
            st.l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; i++) st.o[h][i] = 0.f;
        }
        if (p.n_gc > 0 && j < (int64_t)p.U * p.n_gc) {
            const int u = (int)(j / p.n_gc);
            const int64_t a = (j % p.n_gc) * p.gen_chunk;
            const int64_t b = kvq_min64(a + p.gen_chunk, p.n_gen);
            uint16_t *q_w = reinterpret_cast<uint16_t *>(wbase + part_bytes(D));
            load_q_gen(p, u, q_w);
            generic_range<DPL>(p, u, q_w, a, b, st);
            generic_store<DPL>(p, st, part);
            seg1 = u;
        }
    }
    if (lane == 0) {
        s_seg[warp][0] = seg0;
        s_seg[warp][1] = seg1;
    }
    __syncthreads();

    // ---- merge the warps of this CTA per sequence, publish, take a ticket ----
    // Phase 1 (one thread per (sequence, head)): the running max over the warp
    // partials of that sequence and each partial's weight exp2(m - M).  Phase 2: a
    // flat loop over (sequence, head, channel) with independent loads.
    int ulo = 0x7fffffff, uhi = -1;
    for (int w = 0; w < NW; w++)
        for (int e = 0; e < 2; e++)
            if (s_seg[w][e] >= 0) {
                ulo = min(ulo, s_seg[w][e]);
                uhi = max(uhi, s_seg[w][e]);
            }
    if (uhi < 0) return;
    const int nu = uhi - ulo + 1;
    if (nu > 24) {  // impossible with the host schedule; never index past s_last
        if (tid == 0) report(p.status, KVQ_DEV_BAD_STATE_BIT);
        return;
    }
    const int wb = wbytes / 4;  // floats between warp partials in shared memory
    const float *wpart = reinterpret_cast<const float *>(smem);
    const int R = prow(D);
    // weight tables (merge: [nu*g][2*NW] + [nu*g][2]; combine: [nl*g][max_slots]) in
    // shared memory the tiles no longer use (host checks the capacity)
    float *wtab = reinterpret_cast<float *>(smem + tab_offset<BITS, KITTY, FAST, NW>(p));
    __shared__ int s_slot[24];
    auto src_of = [&](int w, int e) -> const float * {
        return e == 0 ? p.scratch + ((size_t)c * NW + w) * (part_bytes(D) / 4) : wpart + w * wb;
    };
    for (int pi = tid; pi < nu * g; pi += blockDim.x) {
        const int u = ulo + pi / g, h = pi % g;
        float M = -INFINITY;
        for (int w = 0; w < NW; w++)
            for (int e = 0; e < 2; e++)
                if (s_seg[w][e] == u) M = fmaxf(M, src_of(w, e)[h * R + D]);
        float L = 0.f;
        for (int w = 0; w < NW; w++)
            for (int e = 0; e < 2; e++) {
                float f = 0.f;
                if (s_seg[w][e] == u) {
                    const float mw = src_of(w, e)[h * R + D];
                    if (mw != -INFINITY) f = exp2f(mw - M);
                    L = fmaf(src_of(w, e)[h * R + D + 1], f, L);
                }
                wtab[pi * 2 * NW + 2 * w + e] = f;
            }
        wtab[nu * g * 2 * NW + pi * 2] = M;
        wtab[nu * g * 2 * NW + pi * 2 + 1] = L;
        if (h == 0) {
            int ff, fm, fg;
            const int nf = pool_ctas(PF, p.wpc, u, &ff);
            pool_ctas(PM, p.wpc, u, &fm);
            if (!FAST) gen_ctas(p, u, &fg);
            s_slot[u - ulo] = !FAST ? c - fg : (pool == 0 ? c - ff : nf + (c - p.C_f - fm));
        }
    }
    __syncthreads();
    for (int i = tid; i < nu * g * (D / 4); i += blockDim.x) {
        const int pi = i / (D / 4), d = 4 * (i % (D / 4));
        const int ul = pi / g, h = pi % g, u = ulo + ul;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < NW; w++)
            for (int e = 0; e < 2; e++) {
                const float f = wtab[pi * 2 * NW + 2 * w + e];
                if (f != 0.f) {
                    const float4 v = *reinterpret_cast<const float4 *>(src_of(w, e) + h * R + d);
                    acc.x = fmaf(v.x, f, acc.x);
                    acc.y = fmaf(v.y, f, acc.y);
                    acc.z = fmaf(v.z, f, acc.z);
                    acc.w = fmaf(v.w, f, acc.w);
                }
            }
        float *gpart = p.partials + ((size_t)u * p.max_slots + s_slot[ul]) * g * R + h * R;
        *reinterpret_cast<float4 *>(gpart + d) = acc;
        if (d == 0) {
            gpart[D] = wtab[nu * g * 2 * NW + pi * 2];
            gpart[D + 1] = wtab[nu * g * 2 * NW + pi * 2 + 1];
        }
    }
    // Publish: the CTA barrier orders every thread's partial stores before the
    // GPU-scope release fence of the ticket thread of each sequence; the acquire
    // fence after the ticket orders the combine's reads of the other CTAs' slots.
    __syncthreads();
    if (tid < nu) {
        const int u = ulo + tid;
        int f0;
        const int n = pool_ctas(PF, p.wpc, u, &f0) + pool_ctas(PM, p.wpc, u, &f0) + (FAST ? 0 : gen_ctas(p, u, &f0));
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        s_last[tid] = (atomicAdd(&p.tickets[u], 1) == n - 1);
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    __syncthreads();

    // ---- the last CTA of a sequence: log-sum-exp combine of its slots ----
    // Phase 1 (one thread per (sequence, head)): weights w_c = exp2(m_c - M) / L of the
    // slots; phase 2: out = sum_c w_c o_c over (sequence, head, channel).
    __shared__ int s_lu[24];
    if (tid == 0) {
        int n = 0;
        for (int k = 0; k < nu; k++)
            if (s_last[k]) s_lu[n++] = ulo + k;
    }
    int nl = 0;
    for (int k = 0; k < nu; k++) nl += s_last[k] ? 1 : 0;
    __syncthreads();
    if (nl == 0) return;
    const int ms = p.max_slots;
    float *ctab = wtab;  // [nl * g][ms] weights (phase 2 of the merge is done)
    __shared__ int s_ns[24];
    for (int pi = tid; pi < nl * g; pi += blockDim.x) {
        const int u = s_lu[pi / g], h = pi % g;
        int f0;
        const int ns = pool_ctas(PF, p.wpc, u, &f0) + pool_ctas(PM, p.wpc, u, &f0) + (FAST ? 0 : gen_ctas(p, u, &f0));
        if (h == 0) s_ns[pi / g] = ns;
        const float *up = p.partials + (size_t)u * ms * g * R + h * R;
        float M = -INFINITY;
        for (int cc = 0; cc < ns; cc++) M = fmaxf(M, __ldcg(up + (size_t)cc * g * R + D));
        float L = 0.f;
        for (int cc = 0; cc < ns; cc++) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(up + (size_t)cc * g * R + D));
            const float f = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            L = fmaf(ml.y, f, L);
            ctab[pi * ms + cc] = f;
        }
        const float inv = 1.0f / L;
        for (int cc = 0; cc < ns; cc++) ctab[pi * ms + cc] *= inv;
    }
    __syncthreads();
    for (int i = tid; i < nl * g * (D / 4); i += blockDim.x) {
        const int pi = i / (D / 4), d = 4 * (i % (D / 4));
        const int u = s_lu[pi / g], h = pi % g, ns = s_ns[pi / g];
        const float *up = p.partials + (size_t)u * ms * g * R + h * R + d;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int cc = 0; cc < ns; cc++) {
            const float f = ctab[pi * ms + cc];
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(up + (size_t)cc * g * R));
            O.x = fmaf(v.x, f, O.x);
            O.y = fmaf(v.y, f, O.y);
            O.z = fmaf(v.z, f, O.z);
            O.w = fmaf(v.w, f, O.w);
        }
        uint2 hv;
        hv.x = pack_half2(O.x, O.y);
        hv.y = pack_half2(O.z, O.w);
        *reinterpret_cast<uint2 *>(p.out + ((size_t)u * g + h) * D + d) = hv;
    }
    __syncthreads();
    if (tid < nl) p.tickets[s_lu[tid]] = 0;
}

// ---------------------------------------------------------------------------------
int decode_warps_per_cta(int bits, bool kitty, int n_boost, bool fast) {
    if (!fast) return 8;
    const int w = bits == 2 ? WarpSmem<2>(kitty, n_boost).total : WarpSmem<4>(kitty, n_boost).total;
    return w * 8 <= 227 * 1024 ? 8 : 6;
}

size_t decode_smem_bytes(int bits, bool kitty, int n_boost, int D, bool fast) {
    const int nw = decode_warps_per_cta(bits, kitty, n_boost, fast);
    if (fast) return (size_t)nw * (bits == 2 ? WarpSmem<2>(kitty, n_boost).total : WarpSmem<4>(kitty, n_boost).total);
    return (size_t)nw * gen_warp_bytes(D) + kGenTabFloats * 4;
}

int decode_table_floats(int bits, bool kitty, int n_boost, int D, bool fast) {
    if (!fast) return kGenTabFloats;
    if (bits == 2) return kitty ? tab_capacity<2, true, true>(n_boost, D) : tab_capacity<2, false, true>(n_boost, D);
    return tab_capacity<4, false, true>(n_boost, D);
}

template <int BITS, bool KITTY, bool FAST, int DPL, int NW>
static cudaError_t launch_one(const DecodeParams &p, cudaStream_t st) {
    const size_t smem = decode_smem_bytes(BITS, KITTY, p.n_boost, p.D, FAST);
    auto k = decode_kernel<BITS, KITTY, FAST, DPL, NW>;
    // The dynamic shared-memory limit is raised once per device to the most any
    // configuration of this instantiation asks for (the opt-in maximum).
    static int raised[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !raised[dev]) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 1024);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) raised[dev] = 1;
    }
    if (smem > (size_t)(227 * 1024)) return cudaErrorInvalidValue;
    k<<<(unsigned)(p.C_f + p.C_m + p.C_g), NW * 32, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams &p, bool fast, cudaStream_t st) {
    if (fast) {
        if (p.kitty) {
            if (p.wpc == 8) return launch_one<2, true, true, 4, 8>(p, st);
            return launch_one<2, true, true, 4, 6>(p, st);
        }
        if (p.bits == 2) return launch_one<2, false, true, 4, 8>(p, st);
        return launch_one<4, false, true, 4, 8>(p, st);
    }
    switch (p.D) {
        case 64: return launch_one<2, false, false, 2, 8>(p, st);
        case 128: return launch_one<2, false, false, 4, 8>(p, st);
        case 256: return launch_one<2, false, false, 8, 8>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvq
