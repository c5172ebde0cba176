// kvq_quant.cu -- quantize/pack kernels (keys per channel, values per token, Kitty
// key pages), plus the row-copy and token-append kernels of the cache.
//
// The quantizer is the min-max asymmetric one of the KIVI notes (Step 1):
//   scale = fp16( (max - min) / (2^b - 1) ),  code = clamp(rint((x - min) / scale))
// with min/max exact in fp16, the scale computed in fp32 (IEEE division) and
// rounded to fp16, the code computed in fp32 with IEEE division and
// round-half-to-even, a zero scale giving code 0, and signed zeros of min/max
// taken as +0.  Codes are packed 32/b per int32, element j at bit b*j (KIVI
// notes, Step 2, pack_tensor).
//
// Division without a divide per element: r = (x - min) * rcp(scale) differs from
// the correctly rounded quotient q = fl(d / scale) by at most 3 ulp-relative
// (|r - q| <= 2^-22 * |q|), so rint(r) == rint(q) whenever r is farther than
// 2^-11 from a half-integer (for |q| <= 2^10; larger quotients clamp to max_int on
// both sides).  Only those near-tie elements redo the IEEE division (__fdiv_rn),
// which makes every code identical to the one the plain definition gives.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// Group parameters from exact fp16 min/max (as fp32 values).
struct GroupQ {
    float mn, s, inv, maxf;
    uint16_t s16, mn16;
    bool zero;
};

__device__ __forceinline__ GroupQ make_group(float mn, float mx, int max_int) {
    GroupQ g;
    if (mn == 0.0f) mn = 0.0f;  // -0 -> +0
    if (mx == 0.0f) mx = 0.0f;
    float range = __fsub_rn(mx, mn);
    float s32 = __fdiv_rn(range, (float)max_int);
    __half sh = __float2half_rn(s32);
    g.s16 = __half_as_ushort(sh);
    g.mn16 = __half_as_ushort(__float2half_rn(mn));  // exact: mn is an fp16 value
    g.mn = mn;
    g.s = __half2float(sh);
    g.zero = (g.s == 0.0f);
    g.inv = g.zero ? 0.0f : __frcp_rn(g.s);
    g.maxf = (float)max_int;
    return g;
}

__device__ __forceinline__ uint32_t quant_code(float x, const GroupQ &g) {
    float d = __fsub_rn(x, g.mn);  // >= 0
    float r = __fmul_rn(d, g.inv);
    float k = rintf(r);
    if (fabsf(__fsub_rn(r, k)) > 0.5f - 0x1p-11f) k = rintf(__fdiv_rn(d, g.s));
    k = fminf(k, g.maxf);
    return g.zero ? 0u : (uint32_t)k;
}

// |x| * 2^24 of an fp16 value as an exact integer.
__device__ __forceinline__ unsigned long long abs_units(uint32_t h) {
    uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0) return m;
    return (unsigned long long)(m | 0x400u) << (e - 1);
}

// ------------------------------------------------------------------------------
// Fast quantizer.  r = (x - mn) * rcp(s) in fp32 (x - mn is exact: both are fp16
// values); t = r + 1.5 * 2^23 rounds r to the nearest integer, ties to even, into
// the low mantissa bits (0 <= r < 2^22): its bits are 0x4B400000 + rint(r), clamped
// to 0x4B400000 + max_int as integers.  A zero scale has rcp 0, so every code is 0.
// Each thread tracks max |r - rint(r)|; one that comes within 2^-14 of a
// half-integer redoes its block with quant_code (IEEE division), so the codes are
// those of the plain definition: |r - q| <= 1.5 * 2^-23 * q for the correctly
// rounded quotient q, below 2^-14 for q < 128, and larger quotients are clamped to
// max_int by both.  A word accumulates t * 2^(b pos) by integer multiply-add and
// subtracts 0x4B400000 * sum 2^(b pos) once (mod 2^32), which leaves the packed codes.
// ------------------------------------------------------------------------------
constexpr uint32_t kMagicBits = 0x4B400000u;  // 1.5 * 2^23
constexpr float kTieMargin = 0.5f - 0x1p-14f;

// fp32 pairs (Blackwell's f32x2 arithmetic): each lane of the pair rounds exactly as
// the scalar operation, so the pair forms give the same bits, in half the instructions.
__device__ __forceinline__ uint64_t pk2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t sub_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// qbits for two elements at once: h is a half2 of two fp16 values whose groups have
// (min, rcp(scale)) = mn2, inv2.  Returns the two clamped magic-biased codes; em
// tracks the largest distance to a rounding tie.
__device__ __forceinline__ void qbits2(uint32_t h, uint64_t mn2, uint64_t inv2, uint32_t lim, uint32_t &c0,
                                       uint32_t &c1, float &em) {
    const uint64_t mg2 = 0x4B4000004B400000ull;  // (1.5 * 2^23, 1.5 * 2^23)
    const float2 f = unpack_half2(h);
    const uint64_t r = mul_x2(sub_x2(pk2(f.x, f.y), mn2), inv2);
    const uint64_t t = add_x2(r, mg2);
    const float2 e = up2(sub_x2(r, sub_x2(t, mg2)));
    em = fmaxf(em, fmaxf(fabsf(e.x), fabsf(e.y)));
    const float2 tf = up2(t);
    c0 = min(__float_as_uint(tf.x), lim);
    c1 = min(__float_as_uint(tf.y), lim);
}

// 0x4B400000 * sum_{j < n} 2^(b j)  (mod 2^32): the offset a word of n codes picks up.
__host__ __device__ constexpr uint32_t magic_sum(int b, int n) {
    uint32_t s = 0;
    for (int j = 0; j < n; j++) s += kMagicBits << (b * j);
    return s;
}

// ------------------------------------------------------------------------------
// Page map (see PageMap): source unit and destination page index of grid unit u.
// ------------------------------------------------------------------------------
__device__ __forceinline__ int map_src_unit(const PageMap &m, int u) {
    if (!m.ptab) return u;
    const int i = u / m.H_kv, h = u - i * m.H_kv;
    return m.src_by_seq ? (int)m.seq[i] * m.H_kv + h : h;
}
// page index of page pg of the call (dense: pg0 + pg of unit u's region)
__device__ __forceinline__ int64_t map_dst_page(const PageMap &m, int64_t max_T, int G, int64_t pg0, int u,
                                                int64_t pg) {
    if (!m.ptab) return (int64_t)u * (max_T / G) + pg0 + pg;
    const int i = u / m.H_kv, h = u - i * m.H_kv;
    int64_t e = m.ptab[(size_t)m.seq[i] * m.ptab_stride + m.lp0[i] + pg];
    if (e < 0 || e >= m.n_pages) {
        report(m.status, 2 /*KVQ_DEV_BAD_STATE*/);
        e = 0;
    }
    return e * m.H_kv + h;
}

// The row copies of unit u carried by a quant launch: CTA `col` of the rc.cols copying
// CTAs of that unit takes every rc.cols-th 16-byte chunk of each copy.
__device__ __forceinline__ void row_copies(const RowCopies &rc, int D, int u, int64_t col) {
    const int cpr = D >> 3;  // chunks per row
#pragma unroll
    for (int j = 0; j < kMaxRowCopies; j++) {
        if (j >= rc.n) break;
        const RowCopy &c = rc.c[j];
        const int64_t total = c.n_rows * cpr;
        const uint4 *s = reinterpret_cast<const uint4 *>(c.src + ((size_t)u * c.src_rows + c.src_r0) * D);
        uint4 *d = reinterpret_cast<uint4 *>(c.dst + ((size_t)u * c.dst_rows + c.dst_r0) * D);
        for (int64_t i = col * blockDim.x + threadIdx.x; i < total; i += (int64_t)rc.cols * blockDim.x)
            d[i] = __ldg(s + i);
    }
}

// ------------------------------------------------------------------------------
// Keys: one CTA per page of G tokens.  Thread (pair pr, slice sl) holds channels
// 2pr, 2pr+1 for TPS consecutive tokens in registers; min/max (and, for Kitty, the
// channel scores) are combined across slices in shared memory.
// ------------------------------------------------------------------------------
template <int BITS, bool KITTY, int TPS>
__global__ void __launch_bounds__(256) quant_k_kernel(QuantKParams p) {
    constexpr int FPI = KITTY ? 16 : 32 / BITS;  // codes per word of the (low) plane
    constexpr int CB = KITTY ? 2 : BITS;          // bits per code in that plane
    constexpr int NW = TPS / FPI;                 // words per channel per thread
    extern __shared__ __align__(16) unsigned char smem[];
    const int D = p.D, pairs = D >> 1, S = p.slices;
    float *s_min = reinterpret_cast<float *>(smem);           // [S][D]
    float *s_max = s_min + S * D;                             // [S][D]
    unsigned long long *s_score =
        reinterpret_cast<unsigned long long *>(s_max + S * D);  // [S][D] (Kitty)
    int *s_slot = reinterpret_cast<int *>(s_score + (KITTY ? S * D : 0));  // [D]
    if (blockIdx.x >= p.rc.x0) {
        row_copies(p.rc, D, blockIdx.y, blockIdx.x - p.rc.x0);
        return;
    }

    const int tid = threadIdx.x, pr = tid % pairs, sl = tid / pairs;
    const bool active = sl < S;
    const int u = blockIdx.y;
    const int64_t pg = blockIdx.x;
    const int d0 = 2 * pr;
    if (p.pm.lens && tid == 0 && pg == 0 && u % p.pm.H_kv == 0) {  // paged flush: commit the lengths
        const int i = u / p.pm.H_kv;
        int32_t *ln = p.pm.lens + 4 * (size_t)p.pm.seq[i];
        ln[1] = (int32_t)((p.pm.lp0[i] + p.n_pages) * p.G);
        ln[2] = 0;
    }

    uint32_t x[TPS];
    if (active) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(
            p.src + (size_t)map_src_unit(p.pm, u) * p.src_ustride + (size_t)(p.src_t0 + pg * p.G + sl * TPS) * D) +
                              pr;
#pragma unroll
        for (int i = 0; i < TPS; i++) x[i] = __ldg(src + (size_t)i * pairs);
        __half2 lo = *reinterpret_cast<__half2 *>(&x[0]), hi = lo;
#pragma unroll
        for (int i = 1; i < TPS; i++) {
            __half2 v = *reinterpret_cast<__half2 *>(&x[i]);
            lo = __hmin2(lo, v);
            hi = __hmax2(hi, v);
        }
        float2 fl = __half22float2(lo), fh = __half22float2(hi);
        s_min[sl * D + d0] = fl.x;
        s_min[sl * D + d0 + 1] = fl.y;
        s_max[sl * D + d0] = fh.x;
        s_max[sl * D + d0 + 1] = fh.y;
        if (KITTY) {
            unsigned long long a0 = 0, a1 = 0;
#pragma unroll
            for (int i = 0; i < TPS; i++) {
                a0 += abs_units(x[i] & 0xffffu);
                a1 += abs_units(x[i] >> 16);
            }
            s_score[sl * D + d0] = a0;
            s_score[sl * D + d0 + 1] = a1;
        }
    }
    __syncthreads();
    if (KITTY) {
        // Boost selection (Kitty, Sec. 3.2): the n_boost channels with the largest
        // sum |k| over the page; equal scores go to the lower channel index; slots in
        // ascending channel order, sentinel n_boost+1 otherwise.
        if (tid < D) {
            unsigned long long sc = 0;
            for (int s = 0; s < S; s++) sc += s_score[s * D + tid];
            s_score[tid] = sc;  // slice 0 row now holds the page score
        }
        __syncthreads();
        bool boosted = false;
        if (tid < D) {
            unsigned long long sc = s_score[tid];
            int rank = 0;
            for (int e = 0; e < D; e++) {
                unsigned long long o = s_score[e];
                rank += (o > sc) || (o == sc && e < tid);
            }
            boosted = rank < p.n_boost;
            s_slot[tid] = boosted ? 1 : 0;
        }
        __syncthreads();
        int slot = 0;
        if (tid < D) {
            for (int e = 0; e < tid; e++) slot += s_slot[e];
        }
        __syncthreads();
        if (tid < D) s_slot[tid] = boosted ? slot : p.n_boost + 1;
        __syncthreads();
    }
    if (!active) return;

    GroupQ gq[2];
    int slot[2] = {0, 0};
#pragma unroll
    for (int c = 0; c < 2; c++) {
        float mn = s_min[d0 + c], mx = s_max[d0 + c];
        for (int s = 1; s < S; s++) {
            mn = fminf(mn, s_min[s * D + d0 + c]);
            mx = fmaxf(mx, s_max[s * D + d0 + c]);
        }
        int max_int = (1 << BITS) - 1;
        if (KITTY) {
            slot[c] = s_slot[d0 + c];
            max_int = slot[c] < p.n_boost ? 15 : 3;
        }
        gq[c] = make_group(mn, mx, max_int);
    }

    const int64_t page = map_dst_page(p.pm, p.max_T, p.G, p.pg0, u, pg);  // page index
    const int64_t wrow0 = page * (p.G / FPI) + sl * NW;  // first word row of this thread
    uint2 *dst = reinterpret_cast<uint2 *>(p.k_codes);   // channel pairs; in-page order kword_pos
#pragma unroll
    for (int wi = 0; wi < NW; wi++) {
        uint32_t w0 = 0, w1 = 0, h0 = 0, h1 = 0;
#pragma unroll
        for (int j = 0; j < FPI; j++) {
            __half2 v = *reinterpret_cast<__half2 *>(&x[wi * FPI + j]);
            float2 f = __half22float2(v);
            uint32_t c0 = quant_code(f.x, gq[0]), c1 = quant_code(f.y, gq[1]);
            w0 |= (c0 & ((1u << CB) - 1)) << (CB * j);
            w1 |= (c1 & ((1u << CB) - 1)) << (CB * j);
            if (KITTY) {
                h0 |= (c0 >> 2) << (2 * j);
                h1 |= (c1 >> 2) << (2 * j);
            }
        }
        dst[(size_t)(wrow0 + wi) * pairs + (kword_pos(d0, sl * NW + wi) >> 1)] = make_uint2(w0, w1);
        if (KITTY) {
            int32_t *hp = p.k_hi + (size_t)(wrow0 + wi) * p.n_boost;
            if (slot[0] < p.n_boost) hp[slot[0]] = (int32_t)h0;
            if (slot[1] < p.n_boost) hp[slot[1]] = (int32_t)h1;
        }
    }
    if (sl == 0) {
        uint2 m;
        m.x = (uint32_t)gq[0].s16 | ((uint32_t)gq[0].mn16 << 16);
        m.y = (uint32_t)gq[1].s16 | ((uint32_t)gq[1].mn16 << 16);
        reinterpret_cast<uint2 *>(p.k_meta + (size_t)page * D * 2)[pr] = m;
        if (KITTY) {
            uint8_t *bi = p.k_bidx + (size_t)page * D;
            bi[d0] = (uint8_t)slot[0];
            bi[d0 + 1] = (uint8_t)slot[1];
        }
    }
}

// ------------------------------------------------------------------------------
// Keys, KIVI, D = G = 128: one CTA per page, 16 tokens per warp.  Lane l of warp w
// holds channels 4 l .. 4 l + 3 of tokens 16 w .. 16 w + 15 (each warp load reads one
// 256-byte token row).  Channel min / max reduce over the lane's tokens in registers
// and over the warps in shared memory, where threads 0..127 form one channel's group
// each.  Every lane then quantizes its 64 values with the fp32-pair quantizer and
// packs its four channels' codes along tokens into whole words; each word row leaves
// as one 16-byte store (four channels are one chunk of the kword_pos order).  A token
// that came near a rounding tie has its four codes recomputed with quant_code.
// (Measured against it: warps that own 16 channels of all 128 tokens, with no CTA
// barrier, reading 32-byte sectors of 8 rows: 5% slower; a persistent CTA that
// prefetches the next page with cp.async while it quantizes: 10% slower.)
// ------------------------------------------------------------------------------
__device__ __forceinline__ GroupQ group_from_meta(uint32_t m, int max_int) {
    GroupQ g;
    g.s16 = (uint16_t)(m & 0xffffu);
    g.mn16 = (uint16_t)(m >> 16);
    g.mn = h2f(g.mn16);
    g.s = h2f(g.s16);
    g.zero = (g.s == 0.0f);
    g.inv = g.zero ? 0.0f : __frcp_rn(g.s);
    g.maxf = (float)max_int;
    return g;
}

// The exact codes of one token's four channels (x: two half2 words; m: their
// (scale, min) words).  Out of line: the rare near-tie path stays out of the unrolled
// loop, whose code would otherwise outgrow the instruction cache.
__device__ __noinline__ uint4 exact_codes4(uint2 x, uint4 m, int max_int) {
    const float2 f01 = unpack_half2(x.x), f23 = unpack_half2(x.y);
    return make_uint4(quant_code(f01.x, group_from_meta(m.x, max_int)), quant_code(f01.y, group_from_meta(m.y, max_int)),
                      quant_code(f23.x, group_from_meta(m.z, max_int)), quant_code(f23.y, group_from_meta(m.w, max_int)));
}

template <int BITS>
__global__ void __launch_bounds__(256, 4) quant_k_rows(QuantKParams p) {
    constexpr int D = 128, FPI = 32 / BITS, NWR = 16 / FPI;  // word rows per warp
    constexpr int MAXI = (1 << BITS) - 1;
    __shared__ __align__(16) uint16_t s_lo[8][D], s_hi[8][D];  // per warp: channel min / max (fp16)
    __shared__ __align__(16) float s_mn[D], s_inv[D];
    __shared__ __align__(16) uint32_t s_meta[D];
    if (blockIdx.x >= p.rc.x0) {
        row_copies(p.rc, D, blockIdx.y, blockIdx.x - p.rc.x0);
        return;
    }
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int u = blockIdx.y;
    const int64_t pg = blockIdx.x;
    if (p.pm.lens && tid == 0 && pg == 0 && u % p.pm.H_kv == 0) {  // paged flush: commit the lengths
        const int i = u / p.pm.H_kv;
        int32_t *ln = p.pm.lens + 4 * (size_t)p.pm.seq[i];
        ln[1] = (int32_t)((p.pm.lp0[i] + p.n_pages) * p.G);
        ln[2] = 0;
    }
    const uint2 *src = reinterpret_cast<const uint2 *>(
        p.src + (size_t)map_src_unit(p.pm, u) * p.src_ustride + (size_t)(p.src_t0 + pg * 128 + 16 * w) * D) + lane;
    uint2 x[16];
#pragma unroll
    for (int j = 0; j < 16; j++) x[j] = __ldg(src + (size_t)j * (D / 4));
    {
        __half2 lo0 = *reinterpret_cast<const __half2 *>(&x[0].x), hi0 = lo0;
        __half2 lo1 = *reinterpret_cast<const __half2 *>(&x[0].y), hi1 = lo1;
#pragma unroll
        for (int j = 1; j < 16; j++) {
            const __half2 a = *reinterpret_cast<const __half2 *>(&x[j].x);
            const __half2 b = *reinterpret_cast<const __half2 *>(&x[j].y);
            lo0 = __hmin2(lo0, a);
            hi0 = __hmax2(hi0, a);
            lo1 = __hmin2(lo1, b);
            hi1 = __hmax2(hi1, b);
        }
        reinterpret_cast<uint2 *>(&s_lo[w][0])[lane] =
            make_uint2(*reinterpret_cast<uint32_t *>(&lo0), *reinterpret_cast<uint32_t *>(&lo1));
        reinterpret_cast<uint2 *>(&s_hi[w][0])[lane] =
            make_uint2(*reinterpret_cast<uint32_t *>(&hi0), *reinterpret_cast<uint32_t *>(&hi1));
    }
    __syncthreads();
    const int64_t page = map_dst_page(p.pm, p.max_T, p.G, p.pg0, u, pg);
    if (tid < D) {  // channel tid's group over the page
        float mn = h2f(s_lo[0][tid]), mx = h2f(s_hi[0][tid]);
#pragma unroll
        for (int ww = 1; ww < 8; ww++) {
            mn = fminf(mn, h2f(s_lo[ww][tid]));
            mx = fmaxf(mx, h2f(s_hi[ww][tid]));
        }
        const GroupQ g = make_group(mn, mx, MAXI);
        s_mn[tid] = g.mn;
        s_inv[tid] = g.inv;
        const uint32_t m = (uint32_t)g.s16 | ((uint32_t)g.mn16 << 16);
        s_meta[tid] = m;
        reinterpret_cast<uint32_t *>(p.k_meta + (size_t)page * D * 2)[tid] = m;
    }
    __syncthreads();
    const float4 mn4 = reinterpret_cast<const float4 *>(s_mn)[lane];
    const float4 in4 = reinterpret_cast<const float4 *>(s_inv)[lane];
    const uint64_t mn01 = pk2(mn4.x, mn4.y), mn23 = pk2(mn4.z, mn4.w);
    const uint64_t in01 = pk2(in4.x, in4.y), in23 = pk2(in4.z, in4.w);
    constexpr uint32_t lim = kMagicBits + MAXI;
    uint32_t wd[NWR][4];
#pragma unroll
    for (int r = 0; r < NWR; r++)
#pragma unroll
        for (int c = 0; c < 4; c++) wd[r][c] = 0u;
#pragma unroll
    for (int j = 0; j < 16; j++) {
        uint32_t a0, a1, a2, a3;
        float em = 0.f;
        qbits2(x[j].x, mn01, in01, lim, a0, a1, em);
        qbits2(x[j].y, mn23, in23, lim, a2, a3, em);
        if (em > kTieMargin) {  // near a half-integer: this token's exact quotients
            const uint4 e = exact_codes4(x[j], reinterpret_cast<const uint4 *>(s_meta)[lane], MAXI);
            a0 = kMagicBits + e.x;
            a1 = kMagicBits + e.y;
            a2 = kMagicBits + e.z;
            a3 = kMagicBits + e.w;
        }
        const uint32_t m = 1u << (BITS * (j % FPI));
        wd[j / FPI][0] += a0 * m;
        wd[j / FPI][1] += a1 * m;
        wd[j / FPI][2] += a2 * m;
        wd[j / FPI][3] += a3 * m;
    }
    const int64_t row0 = page * (128 / FPI) + w * NWR;  // first word row of this warp
#pragma unroll
    for (int r = 0; r < NWR; r++) {
        const uint32_t off = magic_sum(BITS, FPI);
        const int R = w * NWR + r;
        *reinterpret_cast<uint4 *>(p.k_codes + (size_t)(row0 + r) * D + kword_pos(4 * lane, R)) =
            make_uint4(wd[r][0] - off, wd[r][1] - off, wd[r][2] - off, wd[r][3] - off);
    }
}

// ------------------------------------------------------------------------------
// Values: one thread per token; the whole row (ND x 8 halves) sits in registers.
// ------------------------------------------------------------------------------
template <int BITS, int ND, int GV>
__global__ void __launch_bounds__(128) quant_v_kernel(QuantVParams p) {
    constexpr int FPI = 32 / BITS, D = ND * 8, NWORD = D / FPI;
    static_assert(GV % FPI == 0 && D % GV == 0, "whole words per value group");
    const int u = blockIdx.y;
    if (blockIdx.x >= p.rc.x0) {
        row_copies(p.rc, D, u, blockIdx.x - p.rc.x0);
        return;
    }
    const int64_t tl = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // token within call
    if (tl >= p.n_tok) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(
        p.src + (size_t)map_src_unit(p.pm, u) * p.src_ustride + (size_t)(p.src_t0 + tl) * D);
    uint32_t xw[D / 2];  // the token's row as half2 words
#pragma unroll
    for (int i = 0; i < ND; i++) {
        uint4 v = __ldg(src + i);
        xw[4 * i] = v.x;
        xw[4 * i + 1] = v.y;
        xw[4 * i + 2] = v.z;
        xw[4 * i + 3] = v.w;
    }
    // tok0 is a multiple of G: page tl / G of the call, token tl % G within it
    const int64_t page = map_dst_page(p.pm, p.max_T, p.G, p.tok0 / p.G, u, tl / p.G), tin = tl % p.G;
    // value tile of token tin and its position j there (in-page order vword_pos)
    const int TV = p.TV, j = (int)(tin % TV);
    int32_t *vc = p.v_codes + ((size_t)page * NWORD) * p.G + (size_t)(tin / TV) * NWORD * TV;
    uint32_t *vm = reinterpret_cast<uint32_t *>(p.v_meta) + ((size_t)page * p.G + tin) * (D / GV);
#pragma unroll
    for (int g0 = 0; g0 < D; g0 += GV) {
        __half2 lo = *reinterpret_cast<const __half2 *>(&xw[g0 / 2]), hi = lo;
#pragma unroll
        for (int i = 1; i < GV / 2; i++) {
            __half2 v = *reinterpret_cast<const __half2 *>(&xw[g0 / 2 + i]);
            lo = __hmin2(lo, v);
            hi = __hmax2(hi, v);
        }
        float mn = fminf(__low2float(lo), __high2float(lo));
        float mx = fmaxf(__low2float(hi), __high2float(hi));
        GroupQ g = make_group(mn, mx, (1 << BITS) - 1);
        vm[g0 / GV] = (uint32_t)g.s16 | ((uint32_t)g.mn16 << 16);
#pragma unroll
        for (int wi = g0 / FPI; wi < (g0 + GV) / FPI; wi++) {
            uint32_t w = 0;
#pragma unroll
            for (int j = 0; j < FPI; j += 2) {
                float2 f = unpack_half2(xw[(wi * FPI + j) / 2]);
                w |= quant_code(f.x, g) << (BITS * j);
                w |= quant_code(f.y, g) << (BITS * (j + 1));
            }
            vc[(size_t)wi * TV + vword_pos(j, wi, TV)] = (int32_t)w;
        }
    }
}

// ------------------------------------------------------------------------------
// Values, D = Gv = 128: one CTA per 128 tokens, 16 tokens per warp.  Lane (tq, c) of
// warp w holds tokens 16 w + 8 g + tq (g = 0, 1) and of each the 8-channel chunks
// c, c + 4, c + 8, c + 12 (a warp load reads 64 contiguous bytes of 8 rows).  A
// token's min / max reduces over its 4 lanes by two shuffles, and each of them forms
// the token's group itself.  Codes pack along channels (2-bit words pair the chunks of
// lanes c and c ^ 1) and are staged in shared memory, so that each word row of a value
// tile leaves as contiguous stores (16-byte chunks in the tile's in-page order).
// ------------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ void quant_v_chunk(const QuantVParams &p, int u, int64_t tl0, const uint16_t *src) {
    static_assert(BITS == 2 || BITS == 4, "2- or 4-bit values");
    constexpr int D = 128, FPI = 32 / BITS, NWORD = D / FPI;
    __shared__ __align__(16) uint32_t s_codes[NWORD][128];
    __shared__ __align__(16) uint32_t s_meta[128];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, tq = lane >> 2, c = lane & 3;
    uint4 x[2][4];
#pragma unroll
    for (int g = 0; g < 2; g++)
#pragma unroll
        for (int i = 0; i < 4; i++)
            x[g][i] = reinterpret_cast<const uint4 *>(src + (size_t)(16 * w + 8 * g + tq) * D)[c + 4 * i];
    constexpr uint32_t lim = kMagicBits + (1u << BITS) - 1;
#pragma unroll
    for (int g = 0; g < 2; g++) {
        const int tt = 16 * w + 8 * g + tq;
        __half2 lo = *reinterpret_cast<const __half2 *>(&x[g][0].x), hi = lo;
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int k = (i == 0 ? 1 : 0); k < 4; k++) {
                const uint32_t wk = (&x[g][i].x)[k];
                const __half2 v = *reinterpret_cast<const __half2 *>(&wk);
                lo = __hmin2(lo, v);
                hi = __hmax2(hi, v);
            }
        float a = fminf(__low2float(lo), __high2float(lo)), b = fmaxf(__low2float(hi), __high2float(hi));
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
            b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
        }
        const GroupQ gr = make_group(a, b, (1 << BITS) - 1);
        if (c == 0) s_meta[tt] = (uint32_t)gr.s16 | ((uint32_t)gr.mn16 << 16);
        const uint64_t mn2 = pk2(gr.mn, gr.mn), inv2 = pk2(gr.inv, gr.inv);
#pragma unroll
        for (int i = 0; i < 4; i++) {  // chunk c + 4 i: channels 8 (c + 4 i) .. + 7
            uint32_t part = 0;
            float emax = 0.f;
#pragma unroll
            for (int k = 0; k < 4; k++) {
                uint32_t c0, c1;
                qbits2((&x[g][i].x)[k], mn2, inv2, lim, c0, c1, emax);
                part += c0 * (1u << (BITS * (2 * k)));
                part += c1 * (1u << (BITS * (2 * k + 1)));
            }
            part -= magic_sum(BITS, 8);
            if (emax > kTieMargin) {  // near a half-integer in this chunk: the exact path
                part = 0;
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float2 f = unpack_half2((&x[g][i].x)[k]);
                    part |= quant_code(f.x, gr) << (BITS * (2 * k));
                    part |= quant_code(f.y, gr) << (BITS * (2 * k + 1));
                }
            }
            if (BITS == 2) {  // 16 channels per word: chunks 2m (lane c even) and 2m + 1
                const uint32_t nb = __shfl_xor_sync(0xffffffffu, part, 1);
                if ((c & 1) == 0) s_codes[(c + 4 * i) >> 1][tt] = part | (nb << 16);
            } else {
                s_codes[c + 4 * i][tt] = part;
            }
        }
    }
    __syncthreads();
    // 128 tokens within one page (G is a multiple of 128 here, tok0 a multiple of G)
    const int64_t page = map_dst_page(p.pm, p.max_T, p.G, p.tok0 / p.G, u, tl0 / p.G), tin0 = tl0 % p.G;
    for (int i = tid; i < NWORD * 32; i += 256) {
        const int m = i >> 5, q4 = i & 31;
        const uint4 v = *reinterpret_cast<const uint4 *>(&s_codes[m][4 * q4]);
        // tokens tt .. tt + 3 of the page: value tile tt / TV, position vword_pos there
        const int TV = p.TV, tt = (int)tin0 + 4 * q4, tile = tt / TV, j = tt - tile * TV;
        *reinterpret_cast<uint4 *>(p.v_codes + (size_t)page * NWORD * p.G + ((size_t)tile * NWORD + m) * TV +
                                   vword_pos(j, m, TV)) = v;
    }
    if (tid < 32)
        reinterpret_cast<uint4 *>(reinterpret_cast<uint32_t *>(p.v_meta) + (size_t)page * p.G + tin0)[tid] =
            *reinterpret_cast<const uint4 *>(&s_meta[4 * tid]);
}

// One CTA per 128 value tokens, reading its rows straight from global memory; five
// CTAs per SM (48 registers) hide more of the loads' latency than four.
template <int BITS>
__global__ void __launch_bounds__(256, 5) quant_v_rows(QuantVParams p) {
    const int u = blockIdx.y;
    if (blockIdx.x >= p.rc.x0) {
        row_copies(p.rc, 128, u, blockIdx.x - p.rc.x0);
        return;
    }
    const int64_t tl0 = (int64_t)blockIdx.x * 128;
    quant_v_chunk<BITS>(p, u, tl0,
                        p.src + (size_t)map_src_unit(p.pm, u) * p.src_ustride + (size_t)(p.src_t0 + tl0) * 128);
}

// ------------------------------------------------------------------------------
// Row copies between [U][*][D] fp16 buffers (prefill split, flush bookkeeping).
// ------------------------------------------------------------------------------
__global__ void copy_rows_kernel(CopyRowsParams p) {
    const int64_t chunks = (int64_t)p.n_rows * (p.D / 8);
    const int64_t total = chunks * p.U;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t u = i / chunks, r = i % chunks;
        int64_t row = r / (p.D / 8), c = r % (p.D / 8);
        const uint4 *s = reinterpret_cast<const uint4 *>(
            p.src + ((size_t)u * p.src_rows + p.src_r0 + row) * p.D) + c;
        uint4 *d = reinterpret_cast<uint4 *>(p.dst + ((size_t)u * p.dst_rows + p.dst_r0 + row) * p.D) + c;
        *d = *s;
    }
}

// One new token per sequence: key row -> k_dst[k_row]; value row -> v_dst[v_row],
// after moving v_dst's old row to v_evict[evict_row] when evict_row >= 0 (Kitty
// local window full: the oldest value leaves the window for the Q-buffer).
__global__ void append_kernel(AppendParams p) {
    const int64_t chunks = p.D / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= chunks * p.U) return;
    const int64_t u = i / chunks, c = i % chunks;
    const uint4 *kn = reinterpret_cast<const uint4 *>(p.k_new + (size_t)u * p.D) + c;
    const uint4 *vn = reinterpret_cast<const uint4 *>(p.v_new + (size_t)u * p.D) + c;
    uint4 *kd = reinterpret_cast<uint4 *>(p.k_dst + ((size_t)u * p.k_rows + p.k_row) * p.D) + c;
    uint4 *vd = reinterpret_cast<uint4 *>(p.v_dst + ((size_t)u * p.v_rows + p.v_row) * p.D) + c;
    *kd = *kn;
    if (p.evict_row >= 0) {
        uint4 *ev = reinterpret_cast<uint4 *>(p.v_evict + ((size_t)u * p.evict_rows + p.evict_row) * p.D) + c;
        *ev = *vd;
    }
    *vd = *vn;
}

// ------------------------------------------------------------------------------
// NVFP4 pages (BitDecoding notes, Sec. V-D: Blackwell's native mxfp4 / nvfp4
// formats).  One CTA per page of G tokens: the fp16 page is staged in shared memory,
// its amax gives the page scale S = amax / 2688 (6 * 448); every block of 16 elements
// along the contracted dimension (a key's channels, a value's tokens) gets the e4m3
// scale of (amax_block / 6) / S and its elements the e2m1 codes of x / (s * S), both
// by the hardware conversions (nearest even, saturating); IEEE divisions throughout.
// Code bytes pair the two elements one mma register takes: keys leave as [D/32][G][16]
// (byte = channels 2i, 2i+1 of a token, low nibble first), values as [G/32][D][16]
// (byte = tokens 2m, 2m+1 of a channel).
// ------------------------------------------------------------------------------
template <bool VALUES>
__global__ void __launch_bounds__(256) nvfp4_page_kernel(QuantNvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int G = p.G, D = p.D, tid = threadIdx.x;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);             // [G][D] fp16
    uint8_t *cs = smem + (size_t)G * D * 2;                        // codes: keys [G][D/2], values [D][G/2]
    uint8_t *ss = cs + (size_t)G * D / 2;                          // block scales
    __shared__ float s_red[8];
    const int u = blockIdx.y;
    const int64_t pg = blockIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.src + (size_t)u * p.src_ustride +
                                                       (size_t)(p.src_t0 + pg * G) * D);
    const int n16 = G * D / 8;  // uint4 chunks of the page
    float amax = 0.f;
    for (int i = tid; i < n16; i += 256) {
        const uint4 v = __ldg(src + i);
        reinterpret_cast<uint4 *>(xs)[i] = v;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float2 f = unpack_half2(w[k]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((tid & 31) == 0) s_red[tid >> 5] = amax;
    __syncthreads();
    float pmax = s_red[0];
#pragma unroll
    for (int w = 1; w < 8; w++) pmax = fmaxf(pmax, s_red[w]);
    const float S = __fdiv_rn(pmax, 2688.0f);
    auto xval = [&](int t, int c) { return __half2float(__ushort_as_half(xs[t * D + c])); };
    // one 16-element block: its scale code and the divisor d = s * S (0: all codes 0)
    auto block_scale = [&](float bmax, uint32_t &sc) {
        if (S == 0.0f) {
            sc = 0;
            return 0.0f;
        }
        sc = f32_to_e4m3(__fdiv_rn(__fdiv_rn(bmax, 6.0f), S));
        const float sd = unpack_half2(e4m3x2_to_f16x2(sc)).x;
        return __fmul_rn(sd, S);
    };
    if (!VALUES) {
        // task = (token t, channel block b): 16 channels, 8 code bytes, 1 scale
        for (int i = tid; i < G * (D / 16); i += 256) {
            const int t = i / (D / 16), b = i - t * (D / 16);
            float bmax = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++) bmax = fmaxf(bmax, fabsf(xval(t, 16 * b + k)));
            uint32_t sc;
            const float d = block_scale(bmax, sc);
            uint32_t lo = 0, hi = 0;
            if (d != 0.0f) {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(xval(t, 16 * b + 2 * k + 1), d),
                                                          __fdiv_rn(xval(t, 16 * b + 2 * k), d));
                    if (k < 4) lo |= byte << (8 * k);
                    else hi |= byte << (8 * (k - 4));
                }
            }
            *reinterpret_cast<uint2 *>(cs + (size_t)t * (D / 2) + 8 * b) = make_uint2(lo, hi);
            ss[t * (D / 16) + b] = (uint8_t)sc;
        }
    } else {
        // task = (token block tb, channel c): 16 tokens, 8 code bytes, 1 scale
        for (int i = tid; i < (G / 16) * D; i += 256) {
            const int tb = i / D, c = i - tb * D;
            float bmax = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++) bmax = fmaxf(bmax, fabsf(xval(16 * tb + k, c)));
            uint32_t sc;
            const float d = block_scale(bmax, sc);
            uint32_t lo = 0, hi = 0;
            if (d != 0.0f) {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(xval(16 * tb + 2 * k + 1, c), d),
                                                          __fdiv_rn(xval(16 * tb + 2 * k, c), d));
                    if (k < 4) lo |= byte << (8 * k);
                    else hi |= byte << (8 * (k - 4));
                }
            }
            *reinterpret_cast<uint2 *>(cs + (size_t)c * (G / 2) + 8 * tb) = make_uint2(lo, hi);
            ss[tb * D + c] = (uint8_t)sc;
        }
    }
    __syncthreads();
    const int64_t page = p.pg0 + pg;
    uint4 *dc = reinterpret_cast<uint4 *>(p.codes + ((size_t)u * (p.max_T / G) + (size_t)page) * ((size_t)G * D / 2));
    if (!VALUES) {  // chunk i = (group i / G, token i % G) <- staging row token, bytes 16 group ..
        for (int i = tid; i < G * D / 32; i += 256) {
            const int grp = i / G, t = i - grp * G;
            dc[i] = *reinterpret_cast<const uint4 *>(cs + (size_t)t * (D / 2) + 16 * grp);
        }
    } else {        // chunk i = (token group i / D, channel i % D) <- staging row channel, bytes 16 tg ..
        for (int i = tid; i < G * D / 32; i += 256) {
            const int tg = i / D, c = i - tg * D;
            dc[i] = *reinterpret_cast<const uint4 *>(cs + (size_t)c * (G / 2) + 16 * tg);
        }
    }
    uint8_t *rec = p.meta + ((size_t)u * (p.max_T / G) + page) * p.ms;
    const int nsc = G * D / 16;
    for (int i = tid; i < nsc / 16; i += 256)
        reinterpret_cast<uint4 *>(rec + 16)[i] = reinterpret_cast<const uint4 *>(ss)[i];
    if (tid == 0) *reinterpret_cast<float4 *>(rec) = make_float4(S, 0.f, 0.f, 0.f);
}

// Paged append: CTA b moves the new key and value rows of batch slot b's H_kv heads
// into its sink (while not full) or residual, at the slot's device lengths, and
// advances them.  Only this CTA reads or writes lens[b].
__global__ void paged_append_kernel(PagedAppendParams p) {
    const int b = blockIdx.x;
    int32_t *ln = p.lens + 4 * (size_t)b;
    __shared__ int s_ns, s_nr, s_act;
    if (threadIdx.x == 0) {
        s_ns = ln[0];
        s_nr = ln[2];
        s_act = ln[3];
    }
    __syncthreads();
    if (!s_act) return;
    const bool to_sink = s_ns < p.S;
    if (!to_sink && s_nr >= p.R) {  // never with the host's capacity check
        if (threadIdx.x == 0) report(p.status, 2 /*KVQ_DEV_BAD_STATE*/);
        return;
    }
    const int chunks = p.D / 8, total = p.H_kv * chunks;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int h = i / chunks, c = i - h * chunks;
        const size_t u = (size_t)b * p.H_kv + h;
        const uint4 kn = reinterpret_cast<const uint4 *>(p.k_new + u * p.D)[c];
        const uint4 vn = reinterpret_cast<const uint4 *>(p.v_new + u * p.D)[c];
        uint16_t *kd = to_sink ? p.k_sink + (u * p.S + s_ns) * p.D : p.k_res + (u * p.R + s_nr) * p.D;
        uint16_t *vd = to_sink ? p.v_sink + (u * p.S + s_ns) * p.D : p.v_res + (u * p.R + s_nr) * p.D;
        reinterpret_cast<uint4 *>(kd)[c] = kn;
        reinterpret_cast<uint4 *>(vd)[c] = vn;
    }
    if (threadIdx.x == 0) {
        if (to_sink) ln[0] = s_ns + 1;
        else ln[2] = s_nr + 1;
    }
}

__global__ void set_lens_kernel(SetLensParams p) {
    int32_t *ln = p.lens + 4 * (size_t)p.b;
    ln[0] = p.v0;
    ln[1] = p.v1;
    ln[2] = p.v2;
    ln[3] = p.v3;
}

// ------------------------------------------------------------------------------
// Launchers
// ------------------------------------------------------------------------------
// CTAs per unit for the row copies of a quant launch: about one 16-byte chunk per
// thread of a 256-thread CTA, at most 64.
static int row_copy_cols(const RowCopies &rc, int D) {
    int64_t most = 0;
    for (int j = 0; j < rc.n; j++) most = most > rc.c[j].n_rows ? most : rc.c[j].n_rows;
    if (rc.n <= 0 || most <= 0) return 0;
    const int64_t cols = (most * (D / 8) + 255) / 256;
    return (int)(cols < 64 ? cols : 64);
}

template <int BITS, bool KITTY>
static cudaError_t launch_qk_tps(const QuantKParams &p, int tps, size_t smem, cudaStream_t st) {
    dim3 grid((unsigned)(p.n_pages + p.rc.cols), (unsigned)p.U);
    switch (tps) {
#define KVQ_TPS(T)                                                                        \
    case T:                                                                               \
        if (smem > 48 * 1024)                                                             \
            cudaFuncSetAttribute(quant_k_kernel<BITS, KITTY, T>,                          \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        quant_k_kernel<BITS, KITTY, T><<<grid, 256, smem, st>>>(p);                       \
        return cudaGetLastError();
        KVQ_TPS(16)
        KVQ_TPS(32)
        KVQ_TPS(64)
#undef KVQ_TPS
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant_k(const QuantKParams &p_in, int bits, bool kitty, cudaStream_t st) {
    QuantKParams p = p_in;
    if (p.n_pages <= 0) return cudaSuccess;
    const int fpi = kitty ? 16 : 32 / bits;
    const int pairs = p.D / 2;
    const int smax = 256 / pairs;
    // S slices of G/S tokens per thread: G/S one of 16, 32, 64 and whole words
    int S = 0;
    for (int s = smax < p.G ? smax : p.G; s >= 1 && S == 0; s--)
        if (p.G % s == 0 && (p.G / s == 16 || p.G / s == 32 || p.G / s == 64) && (p.G / s) % fpi == 0) S = s;
    if (S == 0) return cudaErrorInvalidValue;
    const int tps = p.G / S;
    p.slices = S;
    p.rc.x0 = p.n_pages;
    p.rc.cols = row_copy_cols(p.rc, p.D);
    if (!kitty && p.D == 128 && p.G == 128) {  // whole-word rows, fp32-pair quantizer
        dim3 grid((unsigned)(p.n_pages + p.rc.cols), (unsigned)p.U);
        if (bits == 2) quant_k_rows<2><<<grid, 256, 0, st>>>(p);
        else if (bits == 4) quant_k_rows<4><<<grid, 256, 0, st>>>(p);
        else if (bits == 8) quant_k_rows<8><<<grid, 256, 0, st>>>(p);
        else return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    size_t smem = (size_t)S * p.D * 8 + (kitty ? (size_t)S * p.D * 8 + (size_t)p.D * 4 : 0);
    if (kitty) return launch_qk_tps<2, true>(p, tps, smem, st);
    if (bits == 2) return launch_qk_tps<2, false>(p, tps, smem, st);
    if (bits == 4) return launch_qk_tps<4, false>(p, tps, smem, st);
    if (bits == 8) return launch_qk_tps<8, false>(p, tps, smem, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant_v(const QuantVParams &p_in, int bits, cudaStream_t st) {
    QuantVParams p = p_in;
    if (p.n_tok <= 0) return cudaSuccess;
    p.rc.x0 = (p.n_tok + 127) / 128;
    p.rc.cols = row_copy_cols(p.rc, p.D);
    const unsigned gx = (unsigned)(p.rc.x0 + p.rc.cols);
    if ((bits == 2 || bits == 4) && p.D == 128 && p.Gv == 128 && p.G % 128 == 0 && p.n_tok % 128 == 0 &&
        p.tok0 % 128 == 0) {
        dim3 grid(gx, (unsigned)p.U);
        if (bits == 2) quant_v_rows<2><<<grid, 256, 0, st>>>(p);
        else if (bits == 4) quant_v_rows<4><<<grid, 256, 0, st>>>(p);
        else return cudaErrorInvalidValue;
        return cudaGetLastError();
    }
    dim3 grid(gx, (unsigned)p.U);
#define KVQ_QV(B, N, GVV)                                          \
    if (bits == B && p.D == N * 8 && p.Gv == GVV) {                \
        quant_v_kernel<B, N, GVV><<<grid, 128, 0, st>>>(p);        \
        return cudaGetLastError();                                 \
    }
#define KVQ_QV_B(B)                                                        \
    KVQ_QV(B, 8, 32) KVQ_QV(B, 8, 64)                                      \
    KVQ_QV(B, 16, 32) KVQ_QV(B, 16, 64) KVQ_QV(B, 16, 128)                 \
    KVQ_QV(B, 32, 32) KVQ_QV(B, 32, 64) KVQ_QV(B, 32, 128) KVQ_QV(B, 32, 256)
    KVQ_QV_B(2)
    KVQ_QV_B(4)
    KVQ_QV_B(8)
#undef KVQ_QV_B
#undef KVQ_QV
    return cudaErrorInvalidValue;
}

cudaError_t launch_copy_rows(const CopyRowsParams &p, cudaStream_t st) {
    if (p.n_rows <= 0) return cudaSuccess;
    int64_t total = (int64_t)p.U * p.n_rows * (p.D / 8);
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    copy_rows_kernel<<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4(const QuantNvParams &p, bool values, cudaStream_t st) {
    if (p.n_pages <= 0) return cudaSuccess;
    const size_t smem = (size_t)p.G * p.D * 2 + (size_t)p.G * p.D / 2 + (size_t)p.G * p.D / 16;
    dim3 grid((unsigned)p.n_pages, (unsigned)p.U);
    auto k = values ? nvfp4_page_kernel<true> : nvfp4_page_kernel<false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    k<<<grid, 256, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_paged_append(const PagedAppendParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    paged_append_kernel<<<(unsigned)p.B, 128, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_set_lens(const SetLensParams &p, cudaStream_t st) {
    set_lens_kernel<<<1, 1, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t st) {
    int64_t total = (int64_t)p.U * (p.D / 8);
    append_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kvq
