// kvq_decode.cuh -- single-query / GQA decode attention over the packed KV cache
// (the kernel template and its launchers; instantiated by kvq_decode.cu for dense
// caches and by kvq_decode_paged.cu for paged ones).
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
#pragma once

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
    if (tk < p.T_k && p.nvfp4) {  // NVFP4: 8 codes of token tk, e4m3 scale of their block, page scale
        const uint8_t *codes = reinterpret_cast<const uint8_t *>(p.k_codes);
        const uint8_t *rec = reinterpret_cast<const uint8_t *>(p.k_meta) +
                             ((size_t)u * (p.max_T / p.G) + tk / p.G) * p.nv_kms;
        // key page [D/32][G][16]: channels d .. d+7 of token tk are 4 bytes of its group row
        const uint32_t w = *reinterpret_cast<const uint32_t *>(
            codes + ((size_t)u * (p.max_T / p.G) + tk / p.G) * ((size_t)p.G * D / 2) +
            ((size_t)(d / 32) * p.G + tk % p.G) * 16 + (d % 32) / 2);
        const float S = *reinterpret_cast<const float *>(rec);
        const float s = unpack_half2(e4m3x2_to_f16x2(rec[16 + (tk % p.G) * (D / 16) + d / 16])).x * S;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 f = unpack_half2(e2m1x2_to_f16x2((w >> (8 * i)) & 0xFFu));
            kv[2 * i] = f.x * s;
            kv[2 * i + 1] = f.y * s;
        }
        return;
    }
    if (tk < p.T_k) {
        const int kb = p.kitty ? 2 : p.bits, fpi = 32 / kb;
        const int64_t page = tk / p.G;
        // word row tk / fpi, row (tk % G) / fpi of its page: channel c at kword_pos(c, row)
        const int32_t *wp = p.k_codes + ((size_t)u * (p.max_T / fpi) + tk / fpi) * D;
        const int kr = (int)((tk % p.G) / fpi);
        const uint32_t *mp = reinterpret_cast<const uint32_t *>(p.k_meta) +
                             ((size_t)u * (p.max_T / p.G) + page) * D + d;
        const int sh = kb * (int)(tk % fpi);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t code = ((uint32_t)wp[kword_pos(d + i, kr)] >> sh) & ((1u << kb) - 1);
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
        if (tv < p.T_v && p.nvfp4) {  // NVFP4 values: codes of channels d.., scales of their blocks
            // value page [G/32][D][16]: token t of channel c is nibble t & 1 of byte (t % 32) / 2
            const int64_t t = tv % p.G;
            const uint8_t *codes = reinterpret_cast<const uint8_t *>(p.v_codes) +
                                   ((size_t)u * (p.max_T / p.G) + tv / p.G) * ((size_t)p.G * D / 2) +
                                   (size_t)(t / 32) * D * 16 + (t % 32) / 2;
            const uint8_t *rec = reinterpret_cast<const uint8_t *>(p.v_meta) +
                                 ((size_t)u * (p.max_T / p.G) + tv / p.G) * p.nv_vms;
            const float S = *reinterpret_cast<const float *>(rec);
            const uint8_t *sc = rec + 16 + ((tv % p.G) / 16) * D;
#pragma unroll
            for (int i = 0; i < DPL; i++) {
                const float2 f = unpack_half2(e2m1x2_to_f16x2(codes[(d + i) * 16]));
                vv[i] = ((t & 1) ? f.y : f.x) * unpack_half2(e4m3x2_to_f16x2(sc[d + i])).x * S;
            }
            return;
        }
        if (tv < p.T_v) {
            const int fpi = 32 / p.vbits, TV = p.v_tile;
            const int64_t page = tv / p.G, tin = tv % p.G;
            // the value tile of token tin within the page, position vword_pos there
            const int32_t *vt = p.v_codes + ((size_t)u * (p.max_T / p.G) + page) * (size_t)(D / fpi) * p.G +
                                (size_t)(tin / TV) * (D / fpi) * TV;
            const int j = (int)(tin % TV);
#pragma unroll
            for (int i = 0; i < DPL; i++) {
                const int dd = d + i;
                uint32_t w = (uint32_t)vt[(dd / fpi) * TV + vword_pos(j, dd / fpi, TV)];
                uint32_t code = (w >> (p.vbits * (dd % fpi))) & ((1u << p.vbits) - 1);
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

template <int DPL, bool RP = false>
__device__ void generic_range(const DecodeParams &p, int u, const uint16_t *q_w, int64_t a, int64_t b,
                              GenState<DPL> &st, const float *rt = nullptr) {
    const int lane = threadIdx.x & 31, D = p.D, g = p.g;
    const float C = kLog2e * rsqrtf((float)D);
    for (int64_t base = a; base < b; base += 32) {
        const int64_t j = base + lane;
        const bool valid = j < b;
        const int64_t tl = j < p.n_sink ? j : j + p.n_fast * (256 / p.bits);
        float z[8];
#pragma unroll
        for (int h = 0; h < 8; h++) z[h] = 0.f;
        if (valid) {
            for (int d = 0; d < D; d += 8) {
                float kv[8];
                load_k8(p, u, tl, d, kv);
                if (RP) {  // pre-RoPE keys: pairs (d + 2i, d + 2i + 1) turn by tl * theta
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int pr = d / 2 + i;
                        const float2 cs = rope_cs((float)tl, rt[kRopeHi + pr], rt[kRopeLo + pr]);
                        const float ka = kv[2 * i], kb = kv[2 * i + 1];
                        kv[2 * i] = fmaf(ka, cs.x, -kb * cs.y);
                        kv[2 * i + 1] = fmaf(ka, cs.y, kb * cs.x);
                    }
                }
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
            const int64_t tlv = jj < p.n_sink ? jj : jj + p.n_fast * (256 / p.bits);
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
// Schedule arithmetic.  A pool of W warps cuts the sequence-major list of N items
// (n per sequence) into ranges [a_k, a_{k+1}), a_k = floor(k * N / W), evaluated as
// k * (N / W) + floor(k * (N % W) / W) so that it stays in 32-bit values (the host
// checks N < 2^31).
// ---------------------------------------------------------------------------------
struct Pool32 {
    int n, qN, rN, W;
};
__device__ __forceinline__ int pool_a(const Pool32 &P, int k) {
    if (P.W < 46341) return k * P.qN + (int)((unsigned)(k * P.rN) / (unsigned)P.W);  // k * rN < W^2 < 2^31
    return k * P.qN + (int)(((long long)k * P.rN) / P.W);
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

// CTA (within its pool of W warps, wpc per CTA, N items) of the warp that owns item x:
// the largest k with floor(k N / W) <= x.
__device__ __forceinline__ long long cta_of_item(long long W, long long N, long long x, int wpc) {
    const long long k = ((x + 1) * W - 1) / N;
    return (k < W - 1 ? k : W - 1) / wpc;
}

// Slot of this CTA's partial of sequence u (dense caches): its rank among the CTAs that
// hold items of u, fast pool first.  Every CTA between a sequence's first and last one
// in a pool holds some of its items (the host schedule), so the slots of u are 0 .. its
// CTA count - 1, and the combine adds them in a fixed order: the result does not depend
// on the order in which CTAs finish.
__device__ __forceinline__ int dense_slot(const DecodeParams &p, int u, bool tile_kernel) {
    const long long c = blockIdx.x;
    if (!tile_kernel) return (int)(c - ((long long)u * p.n_gc) / p.wpc);
    long long flo = 0, nf = 0;
    if (p.n_fast > 0) {
        flo = cta_of_item(p.W_f, p.N_f, (long long)u * p.n_fast, p.wpc);
        nf = cta_of_item(p.W_f, p.N_f, (long long)(u + 1) * p.n_fast - 1, p.wpc) - flo + 1;
    }
    if (c >= p.C_m) return (int)((c - p.C_m) - flo);
    return (int)(nf + c - cta_of_item(p.W_m, p.N_m, (long long)u * p.n_mini, p.wpc));
}

// Completion count of a blocking host step (DecodeParams::done): one thread of a CTA
// that combined n sequences, after the CTA's output stores were fenced at system
// scope, adds n to the device counter; the CTA that brings it to U resets it and
// releases U to the host word.
__device__ __forceinline__ void count_done(const DecodeParams &p, unsigned int n) {
    unsigned int before;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(before) : "l"(p.done_ctr), "r"(n) : "memory");
    if (before + n == (unsigned int)p.U) {
        *p.done_ctr = 0u;
        asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p.done), "r"((unsigned int)p.U) : "memory");
    }
}
__device__ __forceinline__ unsigned long long atom_add_acq_rel_gpu(unsigned long long *ptr, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(ptr), "l"(v) : "memory");
    return old;
}

// ---------------------------------------------------------------------------------
// The kernel.  FAST: CTAs [0, C_m) mini warps, [C_m, C_m + C_f) fast warps.
// Otherwise: generic warps only, one chunk each.
//
// Epilogue, per sequence u that a CTA holds items of:
//   1. merge: the CTA's warp partials of u (shared memory) -> one partial, written to
//      slot s of u in global memory: the CTA's rank among the CTAs holding items of u
//      (dense caches), or a slot id of the CTA listed under u (paged caches);
//   2. publish: one acquire-release atomic adds the CTA's item count of u to a
//      per-sequence item counter; the CTA that completes the count of all items
//      combines (no CTA ever waits for another);
//   3. combine: log-sum-exp of the slots in slot order -> fp16 out; the combining CTA
//      resets the counters to zero for the next call.
// ---------------------------------------------------------------------------------
// theta_j (hi, lo), passed by value to the pre-RoPE kernels (the first kRopeArgFloats
// of their shared-memory tables); the other kernels take an empty argument.
struct RopeTab {
    float v[kRopeArgFloats];
};
template <bool RP>
struct RopeArg {};
template <>
struct RopeArg<true> {
    RopeTab t;
};

// A unit of sequence u in a pool: the pool's items [s0, s0 + n) are u's.
struct Seg {
    int u, s0, n;
};
// Dense caches: n items per sequence.  Paged: pf[b] = items of batch slots before b
// (one count per slot, the same for each of its H_kv heads); x < H_kv * pf[B].
template <bool PG>
__device__ __forceinline__ Seg seg_of(const DecodeParams &p, const Pool32 &P, const int *pf, int x) {
    Seg r;
    if (!PG) {
        r.u = x / P.n;
        r.s0 = r.u * P.n;
        r.n = P.n;
        return r;
    }
    int lo = 0, hi = p.B;  // the last b with H_kv * pf[b] <= x; H_kv * pf[B] > x
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.H_kv * pf[mid] <= x) lo = mid;
        else hi = mid;
    }
    const int nb = pf[lo + 1] - pf[lo], base = p.H_kv * pf[lo];  // nb > 0
    const int h = (x - base) / nb;
    r.u = lo * p.H_kv + h;
    r.s0 = base + h * nb;
    r.n = nb;
    return r;
}

// Partial of slot c of sequence u: dense [U][max_slots][g][D+4]; paged, the slot id list
// of u into a pool of [4][D+4] partials.
template <bool PG>
__device__ __forceinline__ const float *slot_ptr(const DecodeParams &p, int u, int c, int h) {
    const int R = prow(p.D);
    if (!PG) return p.partials + (((size_t)u * p.max_slots + c) * p.g + h) * R;
    const int id = __ldcg(p.seq_slots + (size_t)u * p.smax + c);
    return p.partials + ((size_t)id * 4 + h) * R;
}

// out[u][h][d .. d+3] = sum_c exp2(m_c - M) o_c / sum_c exp2(m_c - M) l_c over the ns
// slots of u: one pass with a running maximum, eight slots at a time (their loads go
// out together, then the chunk's maximum rescales the running sums once).
template <bool PG>
__device__ void combine_item(const DecodeParams &p, int u, int ns, int h, int d) {
    const int D = p.D;
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < ns; c0 += 8) {
        const float *sp[8];
#pragma unroll
        for (int j = 0; j < 8; j++) sp[j] = c0 + j < ns ? slot_ptr<PG>(p, u, c0 + j, h) : nullptr;
        float2 ml[8];
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            ml[j] = make_float2(-INFINITY, 0.f);
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sp[j]) {
                ml[j] = __ldcg(reinterpret_cast<const float2 *>(sp[j] + D));
                v[j] = __ldcg(reinterpret_cast<const float4 *>(sp[j] + d));
            }
        }
        float Mn = M;
#pragma unroll
        for (int j = 0; j < 8; j++) Mn = fmaxf(Mn, ml[j].x);
        if (Mn == -INFINITY) continue;
        const float r = M == -INFINITY ? 0.f : ex2(M - Mn);
        L *= r;
        O.x *= r;
        O.y *= r;
        O.z *= r;
        O.w *= r;
        M = Mn;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float f = ml[j].x == -INFINITY ? 0.f : ex2(ml[j].x - M);
            L = fmaf(ml[j].y, f, L);
            O.x = fmaf(v[j].x, f, O.x);
            O.y = fmaf(v[j].y, f, O.y);
            O.z = fmaf(v[j].z, f, O.z);
            O.w = fmaf(v[j].w, f, O.w);
        }
    }
    const float inv = 1.0f / L;
    uint2 hv;
    hv.x = pack_half2(O.x * inv, O.y * inv);
    hv.y = pack_half2(O.z * inv, O.w * inv);
    *reinterpret_cast<uint2 *>(p.out + ((size_t)u * p.g + h) * D + d) = hv;
}

// Paged caches: a segment holding all of u's items of one pool, published by the unit
// that computed it (its partial is already in pool slot `id`).  The warp that completes
// u's item count combines u itself.
static __device__ void publish_whole(const DecodeParams &p, int u, int cnt, int id, int n_items) {
    const int lane = threadIdx.x & 31;
    __syncwarp();  // every lane's partial stores precede lane 0's release
    unsigned long long before = 0;
    if (lane == 0) {
        const int k = atomicAdd(&p.slot_ctr[u], 1);
        if (k < p.smax) p.seq_slots[(size_t)u * p.smax + k] = id;
        else report(p.status, KVQ_DEV_BAD_STATE_BIT);
        before = atom_add_acq_rel_gpu(&p.item_ctr[u], ((unsigned long long)cnt << 32) | 1u);
    }
    before = __shfl_sync(0xffffffffu, before, 0);
    if ((int)(before >> 32) + cnt != n_items) return;
    const int ns = min((int)(before & 0xffffffffu) + 1, p.smax);
    const int D4 = p.D / 4;
    for (int i = lane; i < p.g * D4; i += 32) combine_item<true>(p, u, ns, i / D4, 4 * (i % D4));
    if (p.done) __threadfence_system();
    __syncwarp();
    if (lane == 0) {
        p.slot_ctr[u] = 0;
        p.item_ctr[u] = 0;
        if (p.done) count_done(p, 1u);
    }
}

template <int KB, int VB, bool KITTY, bool FAST, bool PAIR, int DPL, int NW, bool PG, bool RP, bool F4 = false>
__global__ void __launch_bounds__(NW * 32, 1) decode_kernel(const DecodeParams p, const RopeArg<RP> ra) {
    // Work units: a warp, or with PAIR (tile kernels) a warp pair -- query warp and
    // value warp -- that shares one region of shared memory.
    constexpr int NU = PAIR ? NW / 2 : NW;
    // A CTA merges up to 2 * NU sequences, and lanes 16.. of its last warp take their
    // slots: one lane per sequence.
    static_assert(2 * NU <= 16, "more merged sequences than slot-taking lanes");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_seg[NU][2];   // sequence of the first / last segment of each unit (-1: none)
    __shared__ int s_cnt[NU][2];   // items of those segments
    // the CTA merges at most the first and last sequence of each unit range
    __shared__ int s_slot[2 * NU]; // this CTA's slot (dense) or slot id (paged) in its i-th sequence
    __shared__ int s_lu[2 * NU];   // sequences this CTA combines
    __shared__ int s_ns[2 * NU];   // their slot counts
    __shared__ int s_fl[2 * NU];   // paged: first and last sequence of each unit range
    __shared__ int s_ml[2 * NU];   // paged: the CTA's merged sequences, ascending
    __shared__ int s_nl, s_nm;
    // The next decode launch in the stream may start as this kernel's CTAs leave.
    griddep_launch_dependents();
    // The paged cache's prologue reads device lengths that preceding work writes.
    if (FAST && PG) griddep_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = PAIR ? warp >> 1 : warp, role = PAIR ? warp & 1 : 0;
    const int D = p.D, g = p.g;
    const int wbytes = FAST ? WarpSmem(KB, VB, KITTY, p.n_boost).total : gen_warp_bytes(D);
    const int part0_off = FAST ? WarpSmem(KB, VB, KITTY, p.n_boost).part0 : 0;
    unsigned char *wbase = smem + unit * wbytes;
    int seg0 = -1, seg1 = -1, cnt0 = 0, cnt1 = 0;
    constexpr bool RG = FAST && PG;  // paged cache: per-sequence item counts
    int *s_pf = reinterpret_cast<int *>(smem + NU * wbytes);  // paged: [B + 1] fast items before slot b
    int *s_pm = s_pf + (p.B + 1);                             // paged: [B + 1] mini items before slot b
    float *s_rt = reinterpret_cast<float *>(smem + NU * wbytes);  // pre-RoPE: the tables (never paged)
    if constexpr (RP) {
        for (int i = tid; i < kRopeArgFloats; i += NW * 32) s_rt[i] = ra.t.v[i];
        __syncthreads();
        if (FAST) {  // the in-row turns of the packed tiles: k theta_j for k = 2m, 2m + 1
            for (int i = tid; i < 8 * 64; i += NW * 32) {
                const int m = i >> 6, j = i & 63;
                const float th = s_rt[kRopeHi + j], tl = s_rt[kRopeLo + j];
                const float k0 = (float)(2 * m), k1 = k0 + 1.f;
                float s0, c0, s1, c1;
                sincosf(fmaf(k0, th, k0 * tl), &s0, &c0);
                sincosf(fmaf(k1, th, k1 * tl), &s1, &c1);
                reinterpret_cast<float4 *>(s_rt + kRopeCS)[i] = make_float4(c0, c1, s0, s1);
                reinterpret_cast<float2 *>(s_rt + kRopeNS)[i] = make_float2(-s0, -s1);
            }
            __syncthreads();
        }
    }

    if (RG && warp == 0) {
        // per-slot item counts from the device lengths, then an exclusive scan
        const int per = (p.B + 31) / 32, b0 = lane * per;
        int sf = 0, sm = 0;
        for (int i = 0; i < per; i++) {
            const int b = b0 + i;
            if (b < p.B) {
                const int4 ln = __ldg(reinterpret_cast<const int4 *>(p.lens) + b);
                const int nf = ln.w ? (int)(((int64_t)ln.y * p.bits) >> 8) : 0;
                const int nm = ln.w ? (ln.x + 15) / 16 + (ln.z + 15) / 16 : 0;
                s_pf[b + 1] = nf;  // counts first, prefix below
                s_pm[b + 1] = nm;
                sf += nf;
                sm += nm;
            }
        }
        int ef = sf, em = sm;  // inclusive scan of the lane sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tf = __shfl_up_sync(0xffffffffu, ef, o), tm = __shfl_up_sync(0xffffffffu, em, o);
            if (lane >= o) {
                ef += tf;
                em += tm;
            }
        }
        ef -= sf;
        em -= sm;
        for (int i = 0; i < per; i++) {
            const int b = b0 + i;
            if (b < p.B) {
                ef += s_pf[b + 1];
                em += s_pm[b + 1];
                s_pf[b + 1] = ef;
                s_pm[b + 1] = em;
            }
        }
        if (lane == 0) {
            s_pf[0] = 0;
            s_pm[0] = 0;
        }
    }
    if (RG) __syncthreads();

    // The CTA's sequences ulo .. ulo + nu - 1 follow from its item range.  Their slots
    // are taken now (lanes of warp 0); the atomics' latency hides behind the tiles.
    // The grid holds the mini pool's CTAs first: their work is short, and under a
    // programmatic dependent launch the first CTAs are the first to get SMs.
    const bool fastpool = FAST && (int)blockIdx.x >= p.C_m;
    const Pool32 P = fastpool ? Pool32{(int)p.n_fast, p.qN_f, p.rN_f, p.W_f}
                              : Pool32{(int)p.n_mini, p.qN_m, p.rN_m, p.W_m};
    const int *pfx = fastpool ? s_pf : s_pm;
    const int kc = ((int)blockIdx.x - (fastpool ? p.C_m : 0)) * p.wpc;
    int ulo, nu;
    if (RG) {
        // merged sequences: first and last of each unit range, ascending and distinct
        if (tid < 2 * p.wpc) {
            const int k = kc + (tid >> 1);
            const int x = (tid & 1) ? pool_a(P, k + 1) - 1 : pool_a(P, k);
            s_fl[tid] = seg_of<RG>(p, P, pfx, x).u;
        }
        __syncthreads();
        if (tid < 2 * p.wpc) {
            const int v = s_fl[tid];
            if (tid == 0 || v != s_fl[tid - 1]) {
                int pos = 0;
                for (int j = 1; j <= tid; j++) pos += s_fl[j] != s_fl[j - 1];
                s_ml[pos] = v;
            }
            if (tid == 0) {
                int n = 1;
                for (int j = 1; j < 2 * p.wpc; j++) n += s_fl[j] != s_fl[j - 1];
                s_nm = n;
            }
        }
        __syncthreads();
        ulo = 0;
        nu = s_nm;
    } else {
        int a0, a1, n;
        if (FAST) {
            a0 = pool_a(P, kc);
            a1 = pool_a(P, kc + p.wpc);
            n = P.n;
        } else {
            a0 = (int)blockIdx.x * p.wpc;
            a1 = min(a0 + p.wpc, p.U * p.n_gc);
            n = p.n_gc;
        }
        if (a1 <= a0) return;  // no items (never with the host schedule)
        ulo = a0 / n;
        nu = (a1 - 1) / n - ulo + 1;
    }
    if (nu > 2 * NU) {  // impossible with the host schedule; never index past the tables
        if (tid == 0) report(p.status, KVQ_DEV_BAD_STATE_BIT);
        return;
    }
    // sequence of the CTA's i-th merged entry; items of sequence u in both pools
    auto seq_at = [&](int i) { return RG ? s_ml[i] : ulo + i; };
    auto items_of = [&](int u) {
        if (!RG) return p.n_items;
        const int b = u / p.H_kv;
        return (s_pf[b + 1] - s_pf[b]) + (s_pm[b + 1] - s_pm[b]);
    };
    // The slots are taken by lanes 16.. of the last warp, which issue no copies and no
    // release fences, so nothing waits for the paged cache's atomics before the epilogue.
    const int slot_lane = tid - (NW * 32 - 16);
    int my_slot = 0;
    auto take_slot = [&]() {
        const int u = seq_at(slot_lane);
        if (!RG) return dense_slot(p, u, FAST);
        const int k = atomicAdd(&p.slot_ctr[u], 1);
        const int id = (int)blockIdx.x * (2 * NU) + slot_lane;  // the CTA's own pool slots
        if (k < p.smax) p.seq_slots[(size_t)u * p.smax + k] = id;
        else report(p.status, KVQ_DEV_BAD_STATE_BIT);
        return id;
    };

    if (FAST) {
        const int k = kc + unit;
        int x = pool_a(P, k);
        const int x1 = pool_a(P, k + 1);
        // The first segment of a unit range (if another follows) keeps its partial in
        // the unit's part0 area, the last one in the (then idle) tile region.  A
        // paged range may cross more sequences: a segment between the first and the
        // last holds all of its sequence's items of this pool, and its unit writes it
        // to its own pool slot and publishes it alone.
        // one object per unit for all its segments: each keeps its mbarrier phases
        PairWarp<KB, VB, KITTY, RG, RP> pw(p, wbase);
        MiniWarp<KB, VB, KITTY, RG, RP> mw(p, wbase, 0);
        F4Warp<RG> fw(p, wbase);
        pw.rt = s_rt;
        mw.rt = s_rt;
        if (role == 0) pw.init_bars();  // all of the unit's mbarriers (mini units use four)
        if (PAIR) asm volatile("bar.sync %0, 64;" ::"r"(1 + unit) : "memory");  // the pair's partner
        if (slot_lane >= 0 && slot_lane < nu) my_slot = take_slot();
        // Before the wait for the preceding kernel in the stream: the first copies of a
        // packed-tile warp's first segment, when those tiles lie in pages that no
        // library call has written since this cache's previous decode (p.early_tiles).
        bool pre = false;
        if (!PAIR && !F4 && !RG && fastpool && x < x1) {
            const Seg sg = seg_of<RG>(p, P, pfx, x);
            const int a = x - sg.s0, b = min(x1, sg.s0 + sg.n) - sg.s0;
            if (a + min(b - a, 2) <= p.early_tiles) {
                pw.start(sg.u, a, b);
                pre = true;
            }
        }
        if (!RG) griddep_wait();
        // mini units: the first warp of a pair runs the 16-token tiles alone
        const bool active = fastpool || role == 0;
        const int writer = (PAIR && fastpool) ? 1 : 0;  // the warp that writes the partial
        for (int e = 0; (RG || e < 2) && x < x1; e++) {  // dense ranges: at most two sequences
            const Seg sg = seg_of<RG>(p, P, pfx, x);
            const int u = sg.u;
            const int end = min(x1, sg.s0 + sg.n);
            const bool last = end == x1, whole = RG && e > 0 && !last;
            const int id = p.mid_base + (fastpool ? 0 : p.U) + u;
            float *dst = whole ? p.partials + (size_t)id * 4 * prow(D)
                               : reinterpret_cast<float *>(wbase + (last ? 0 : part0_off));
            if (F4 && fastpool) {
                fw.run(u, x - sg.s0, end - sg.s0, dst);
            } else if (fastpool) {
                if (!PAIR) pw.run(u, x - sg.s0, end - sg.s0, dst, pre && e == 0);
                else if (role == 0) pw.run_q(u, x - sg.s0, end - sg.s0);
                else pw.run_p(u, x - sg.s0, end - sg.s0, dst);
            } else if (active) {
                mw.run(u, x - sg.s0, end - sg.s0, dst);
            }
            if (RG && whole) {
                if (role == writer) publish_whole(p, u, end - x, id, items_of(u));
            } else if (!last) {
                seg0 = u;
                cnt0 = end - x;
            } else {
                seg1 = u;
                cnt1 = end - x;
            }
            x = end;
        }
    } else {
        // ---- generic warp: one chunk of one sequence ----
        griddep_wait();
        if (slot_lane >= 0 && slot_lane < nu) my_slot = take_slot();
        const int64_t j = (int64_t)blockIdx.x * p.wpc + warp;
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
            generic_range<DPL, RP>(p, u, q_w, a, b, st, s_rt);
            generic_store<DPL>(p, st, reinterpret_cast<float *>(wbase));
            seg1 = u;
            cnt1 = 1;
        }
    }
    if (lane == 0 && role == 0) {
        s_seg[unit][0] = seg0;
        s_seg[unit][1] = seg1;
        s_cnt[unit][0] = cnt0;
        s_cnt[unit][1] = cnt1;
    }
    if (slot_lane >= 0 && slot_lane < nu) s_slot[slot_lane] = my_slot;
    __syncthreads();

    // ---- merge: one float4 of (sequence, head, channels) per thread and step ----
    const int R = prow(D), D4 = D / 4;
    auto src_of = [&](int w, int e) -> const float * {
        return reinterpret_cast<const float *>(smem + w * wbytes + (e == 0 ? part0_off : 0));
    };
    for (int i = tid; i < nu * g * D4; i += NW * 32) {
        const int pi = i / D4, d = 4 * (i - pi * D4);
        const int ul = pi / g, h = pi - ul * g, u = seq_at(ul);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NU; w++)
#pragma unroll
            for (int e = 0; e < 2; e++)
                if (s_seg[w][e] == u) M = fmaxf(M, src_of(w, e)[h * R + D]);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NU; w++)
#pragma unroll
            for (int e = 0; e < 2; e++)
                if (s_seg[w][e] == u) {
                    const float *s = src_of(w, e) + h * R;
                    const float mw = s[D];
                    const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
                    L = fmaf(s[D + 1], f, L);
                    const float4 v = *reinterpret_cast<const float4 *>(s + d);
                    acc.x = fmaf(v.x, f, acc.x);
                    acc.y = fmaf(v.y, f, acc.y);
                    acc.z = fmaf(v.z, f, acc.z);
                    acc.w = fmaf(v.w, f, acc.w);
                }
        const int slot = s_slot[ul];
        if (slot < p.max_slots) {
            float *gp = RG ? p.partials + ((size_t)slot * 4 + h) * R
                           : p.partials + (((size_t)u * p.max_slots + slot) * g + h) * R;
            *reinterpret_cast<float4 *>(gp + d) = acc;
            if (d == 0) *reinterpret_cast<float2 *>(gp + D) = make_float2(M, L);
        } else if (d == 0) {
            report(p.status, KVQ_DEV_BAD_STATE_BIT);
        }
    }
    // ---- publish: the barrier orders every thread's partial stores before the
    // release of the item-counter atomic; its acquire orders the combine's reads ----
    __syncthreads();
    if (tid == 0) s_nl = 0;
    __syncthreads();
    if (tid < nu) {
        const int u = seq_at(tid);
        int items = 0;
#pragma unroll
        for (int w = 0; w < NU; w++)
#pragma unroll
            for (int e = 0; e < 2; e++)
                if (s_seg[w][e] == u) items += s_cnt[w][e];
        // item counter: items merged in the high word, CTAs arrived in the low word
        const unsigned long long before = atom_add_acq_rel_gpu(&p.item_ctr[u], ((unsigned long long)items << 32) | 1u);
        if ((int)(before >> 32) + items == items_of(u)) {  // every CTA of u has arrived: it took
            const int k = atomicAdd(&s_nl, 1);              // its slot before its arrival
            s_lu[k] = u;
            s_ns[k] = (int)(before & 0xffffffffu) + 1;
        }
    }
    __syncthreads();
    const int nl = s_nl;
    if (nl == 0) return;

    // ---- combine: out = sum_c exp2(m_c - M) o_c / sum_c exp2(m_c - M) l_c ----
    for (int i = tid; i < nl * g * D4; i += NW * 32) {
        const int pi = i / D4, d = 4 * (i - pi * D4);
        const int lk = pi / g, h = pi - lk * g;
        combine_item<RG>(p, s_lu[lk], min(s_ns[lk], RG ? p.smax : p.max_slots), h, d);
    }
    if (p.done) __threadfence_system();  // this thread's output stores, before the count
    __syncthreads();
    if (tid < nl) {
        if (RG) p.slot_ctr[s_lu[tid]] = 0;
        p.item_ctr[s_lu[tid]] = 0;
    }
    if (p.done && tid == 0) count_done(p, (unsigned int)nl);
}

// ---------------------------------------------------------------------------------
// Dynamic shared memory of a CTA: the 227 KB per block less 4 KB kept for the kernel's
// static shared memory and the paged / pre-RoPE extras.
constexpr int kSmemMax = 227 * 1024 - 4096;

// Units (warps, or warp pairs) per CTA of a tile kernel: as many of 8, 6, 4 as fit.
constexpr int tile_units(int kb, int vb, bool kitty, int n_boost) {
    const int w = WarpSmem(kb, vb, kitty, n_boost).total;
    return w * 8 <= kSmemMax ? 8 : w * 6 <= kSmemMax ? 6 : 4;
}
// Tile kernels on warp pairs (query warp + value warp per unit): 4-bit keys.
constexpr bool tile_pair(int kb, int vb) { return kb == 4 && vb == 4; }

// theta_j = base^(-2j/D) of (D, base) in double, kept as a two-float hi + lo (computed
// once per (D, base) on the host).
static const RopeTab &rope_tables(int D, float base) {
    static thread_local RopeTab tab;
    static thread_local int tD = -1;
    static thread_local float tb = -1.f;
    if (tD != D || tb != base) {
        for (int i = 0; i < kRopeArgFloats; i++) tab.v[i] = 0.f;
        for (int j = 0; j < D / 2 && j < 128; j++) {
            const double th = pow((double)base, -2.0 * (double)j / (double)D);
            const float hi = (float)th;
            tab.v[kRopeHi + j] = hi;
            tab.v[kRopeLo + j] = (float)(th - (double)hi);
        }
        tD = D;
        tb = base;
    }
    return tab;
}

template <int KB, int VB, bool KITTY, bool FAST, bool PAIR, int DPL, int NW, bool PG = false, bool RP = false,
          bool F4 = false>
static cudaError_t launch_one(const DecodeParams &p, cudaStream_t st) {
    size_t smem = decode_smem_bytes(KB, VB, KITTY, p.n_boost, p.D, FAST);
    if (PG) smem += (size_t)(p.B + 1) * 8;  // paged: per-slot item prefixes
    if (RP) smem += kRopeFloats * 4;        // pre-RoPE: the tables
    auto k = decode_kernel<KB, VB, KITTY, FAST, PAIR, DPL, NW, PG, RP, F4>;
    // The dynamic shared-memory limit is raised once per device to the most any
    // configuration of this instantiation can ask for: the opt-in maximum less the
    // kernel's static shared memory.
    static int raised[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !raised[dev]) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) raised[dev] = 1;
    }
    if (smem > (size_t)kSmemMax) return cudaErrorInvalidValue;
    RopeArg<RP> ra;
    if constexpr (RP) ra.t = rope_tables(p.D, p.rope_base);
    // Programmatic dependent launch: the kernel's CTAs may start while the preceding
    // kernel in the stream finishes; every read of data that kernel may write waits
    // for it (griddep_wait in the kernel).
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(p.C_f + p.C_m + p.C_g));
    lc.blockDim = dim3(NW * 32);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&lc, k, p, ra);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// KIVI tiles of key width KB and value width VB; p.wpc == tile_units(KB, VB).
// Pre-RoPE tiles run on single warps (their QK is on the CUDA cores).
template <int KB, int VB, bool PG, bool RP = false>
static cudaError_t launch_tiles(const DecodeParams &p, cudaStream_t st) {
    constexpr int U = tile_units(KB, VB, false, 0);
    constexpr bool PAIR = tile_pair(KB, VB) && !RP;
    if (p.wpc != U) return cudaErrorInvalidValue;
    return launch_one<KB, VB, false, true, PAIR, 4, PAIR ? 2 * U : U, PG, RP>(p, st);
}

// Key / value width pair of a tile launch -> its instantiation.
template <bool PG, bool RP = false>
static cudaError_t launch_tiles_any(const DecodeParams &p, cudaStream_t st) {
    switch (p.bits * 16 + p.vbits) {
        case 2 * 16 + 2: return launch_tiles<2, 2, PG, RP>(p, st);
        case 2 * 16 + 4: return launch_tiles<2, 4, PG, RP>(p, st);
        case 2 * 16 + 8: return launch_tiles<2, 8, PG, RP>(p, st);
        case 4 * 16 + 2: return launch_tiles<4, 2, PG, RP>(p, st);
        case 4 * 16 + 4: return launch_tiles<4, 4, PG, RP>(p, st);
        case 4 * 16 + 8: return launch_tiles<4, 8, PG, RP>(p, st);
        case 8 * 16 + 2: return launch_tiles<8, 2, PG, RP>(p, st);
        case 8 * 16 + 4: return launch_tiles<8, 4, PG, RP>(p, st);
        case 8 * 16 + 8: return launch_tiles<8, 8, PG, RP>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvq
