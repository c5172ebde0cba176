// kvq_decode_fast.cuh -- tensor-core warps of the decode kernel (sm_103a, mma.sync
// m16n8k16 f16 -> f32).  Included by kvq_decode.cu only.
//
// FastWarp: packed tiles (TOK = 128 tokens at 2 bits, 64 at 4 bits) whose keys and
// values are both packed.  MiniWarp: 16-token tiles whose values are fp16 (sink,
// residual / Q-buffer / local window), with fp16 keys or, for Kitty, a packed key
// block.  Both keep the online-softmax state of head t in lane (g, t) and write one
// partial [8][D+2] (o[0..D), m, l; log2 units) per sequence segment.
//
// Conventions shared by both:
//  * Query heads g <= 4.  The QK B operand has 8 columns: column 2h carries the fp16
//    hi part of head h's folded query, column 2h+1 the fp16 lo part (the exact
//    residual), so each lane adds its two columns.  The folded query is
//    q * 2^-4 * scale_k, formed with HMUL2 / HFMA2 on exact fp16 inputs (22 bits);
//    log2(e)/sqrt(D) * 2^4 is applied to the fp32 logits.
//  * The per-page key-min term sum_d q_d * min_d of each head comes from one more
//    mma per 16-channel slab: A = the mins (all rows equal), B = q * 2^-4.
//  * A packed code c at bit offset k < 10 of a 16-bit half is the fp16 subnormal
//    c * 2^(k-24): one AND per two codes gives an exact mma operand; the 2^(24-k)
//    factor is applied to the fp32 results.
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQScale = 0.0625f;  // q is folded as q * 2^-4 (exact) to keep q*scale in fp16 range
constexpr int kSlots = 4;           // copy mbarriers per unit (fast: 2 key halves, 2 value halves)
constexpr int kBars = 9;            // + warp-pair handoff: p' full x2, p' empty x2, query side done

__host__ __device__ constexpr int hi_stride(int nb) { return nb * 4 + 16; }
// A warp / CTA partial: 8 head rows of prow(D) floats: o[0..D), m at D, l at D+1
// (rows padded to 16 bytes for vector access).
__host__ __device__ constexpr int prow(int D) { return D + 4; }
__host__ __device__ inline int part_bytes(int D) { return 8 * prow(D) * 4; }

// Code-width constants of the register extraction.  A packed word holds FPI codes of
// B bits; after split(), each 16-bit half of a register holds FPI/2 of them, and row
// set J of an mma reads code J of every half as an exact fp16 subnormal (code *
// 2^(B JJ - 24)) through one AND.  Codes above bit 9 of a half would reach the
// exponent field, so row sets J >= JDIRECT read a copy of the register shifted right
// by SH.
template <int B>
struct Codes {
    static constexpr int FPI = 32 / B;
    static constexpr int NJ = FPI / 2;                         // mma row sets per word: 8, 4 or 2
    static constexpr int JDIRECT = B == 2 ? 5 : B == 4 ? 2 : 1;
    static constexpr int SH = B == 2 ? 6 : 8;
    static constexpr uint32_t MASK0 = ((1u << B) - 1u) | (((1u << B) - 1u) << 16);
    template <int J>
    __device__ __forceinline__ static constexpr int jj() { return J < JDIRECT ? J : J - SH / B; }
};

// A packed tile: TOK tokens of keys (8 word rows of KB-bit codes, D channels) and of
// values (D / VFPI word rows of VB-bit codes, TOK tokens).  P is the token (and key
// channel) pairing of split(): a register pairs the values at offsets t and t + P of
// a 16-wide slab; it is chosen so that the two tokens of a lane's QK rows g and g+8
// (KFPI / 2 apart) land next to each other in the p' row.
template <int KB, int VB>
struct Tile {
    using K = Codes<KB>;
    using V = Codes<VB>;
    static constexpr int D = 128;
    static constexpr int TOK = 8 * K::FPI;                  // 128, 64 or 32 tokens
    static constexpr int P = KB == 2 ? 8 : 4;
    static constexpr bool P_ADJ = K::FPI / 2 == P;          // a lane's two p' values are adjacent
    static constexpr int K_STRIDE = D * 4;                  // key word row (chunks in kword_pos order)
    static constexpr int V_ROWS = D / V::FPI;               // value channel blocks: 8, 16 or 32
    static constexpr int V_STRIDE = TOK * 4;                // value word row (chunks in vword_pos order)
    static constexpr int NSET = V_ROWS / 8;                 // 1, 2 or 4 sets of 8 word rows
    static constexpr int TSLABS = TOK / 16;                 // 16-token slabs for PV
    static constexpr int PV_STEPS = TSLABS * NSET;          // one ldmatrix + split each
    // key half-stage
    static constexpr int OFF_K = 0;
    static constexpr int OFF_KM = 8 * K_STRIDE;             // (scale, min) per channel, 512 B
    static constexpr int OFF_HI = OFF_KM + D * 4;           // Kitty: 8 rows of hi_stride(nb), then D bytes of index
    // value half-stage
    static constexpr int OFF_V = 0;
    static constexpr int OFF_VM = V_ROWS * V_STRIDE;        // (scale, min) per token
    static constexpr int V_HALF = OFF_VM + TOK * 4;
    static constexpr int PROW = TOK + 8;                    // p' row (halves), padded
    static constexpr int PBUF = 4 * PROW * 2;               // one p' buffer: heads 0..3
};

constexpr int kMiniRow = 128 * 2 + 16;                 // padded fp16 row of the mini tiles
constexpr int kMiniHalf = 16 * kMiniRow;               // 16 fp16 rows

__host__ __device__ constexpr int round128(int x) { return (x + 127) & ~127; }
// The NVFP4 tiles' four stages (F4Warp) live in the 4-bit tile region.
constexpr int kF4Region = 2 * 4736 + 2 * 4608;

// Per-warp shared memory (fast and mini warps share one layout):
//   [tile region][p' buffer x2][q fp16 [4][128]][q' pairs [4 heads][8 slabs][4 lanes] x 8 B]
//   [slot index 64 B][mbarriers kBars x 8 B][pair handoff: stats [3][4], alpha [2][4] fp32]
//   [first-segment partial [4][D+4] fp32]
// The tile region holds, for a fast warp, two key halves (codes + (scale, min) per
// channel [+ Kitty planes]), two value-code halves and two value (scale, min) rows;
// for a mini warp, four 16-row halves.  After the tiles it holds the warp's partial.
struct WarpSmem {
    int ksz = 0, vsz = 0, vmsz = 0, mslot = 0, k0 = 0, v0 = 0, vm0 = 0, region = 0;
    int pbuf = 0, qraw = 0, qpair = 0, invb = 0, bars = 0, stats = 0, alpha = 0, part0 = 0, total = 0;
    // kb, vb: key and value code widths of the tile (2, 4 or 8)
    __host__ __device__ constexpr WarpSmem(int kb, int vb, bool kitty, int nb) {
        const int D = 128, tok = 256 / kb, v_rows = D * vb / 32;
        const int off_hi = 8 * D * 4 + D * 4, pbuf1 = 4 * (tok + 8) * 2;
        ksz = round128(off_hi + (kitty ? 8 * hi_stride(nb) + D : 0));
        vsz = round128(v_rows * tok * 4);
        vmsz = round128(tok * 4);
        const int mk = 1024 + ((4 * nb + 15) & ~15) + 128;  // mini packed-key block
        mslot = round128(kMiniHalf > mk ? kMiniHalf : mk);
        k0 = 0;
        v0 = 2 * ksz;
        vm0 = v0 + 2 * vsz;
        region = vm0 + 2 * vmsz;
        if (region < kSlots * mslot) region = kSlots * mslot;
        if (kb == 4 && vb == 4 && !kitty && region < kF4Region) region = kF4Region;
        pbuf = region;
        qraw = pbuf + 2 * pbuf1;
        qpair = qraw + 4 * 128 * 2;
        invb = qpair + 4 * 8 * 4 * 8;
        bars = invb + 64;
        stats = bars + 8 * 16;                      // m, l, mn of 4 heads
        alpha = stats + 12 * 4;                     // per p' buffer: rescale of 4 heads (+4 unused = 1)
        part0 = (alpha + 8 * 4 * 2 + 15) & ~15;     // partial of a first segment: 4 head rows
        total = round128(part0 + 4 * prow(128) * 4);
    }
};

// ---------------------------------------------------------------------------
// Shared pieces
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Channel of k index kk (0..3 = k 2t, 2t+1, 2t+8, 2t+9) of lane t in slab sl under
// the key k-mapping of split(): (t, t+8, t+4, t+12) for 2 bits, (t, t+4, t+8, t+12)
// for 4 bits, all + 16 sl.
template <int PS>
__device__ __forceinline__ int chan_of(int sl, int t, int kk) {  // kk: 0..3 = k 2t, 2t+1, 2t+8, 2t+9
    const int off[4] = {0, PS, PS == 8 ? 4 : 8, 12};
    return 16 * sl + t + off[kk];
}

// The g query heads of sequence u, 2 x 16 bytes per lane (heads >= g zero).  Loaded
// before a warp issues its first tile copies so that they are not queued behind them.
struct QRegs {
    uint4 v[2];
};
__device__ __forceinline__ QRegs load_q_regs(const DecodeParams &p, int u) {
    const int lane = threadIdx.x & 31;
    QRegs r;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int i = lane + 32 * j, h = i / 16, d = (i % 16) * 8;
        r.v[j] = make_uint4(0, 0, 0, 0);
        if (h < p.g) r.v[j] = __ldg(reinterpret_cast<const uint4 *>(p.q + ((size_t)u * p.g + h) * 128 + d));
    }
    return r;
}

// Stores the query into the warp's buffers:
//   qraw[h][ch] = q (fp16), heads >= g zero;
//   qpair[h][sl][t] = the two half2 (q * 2^-4) of lane t's channels in slab sl.
template <int PS>
__device__ void store_q_warp(const QRegs &qr, uint16_t *qraw, uint2 *qpair) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int i = lane + 32 * j, h = i / 16, d = (i % 16) * 8;
        *reinterpret_cast<uint4 *>(qraw + h * 128 + d) = qr.v[j];
    }
    __syncwarp();
    const uint32_t s4 = 0x2C002C00u;  // half2(2^-4, 2^-4)
    for (int i = lane; i < 4 * 8 * 4; i += 32) {
        const int h = i / 32, sl = (i / 4) % 8, t = i % 4;
        auto qh = [&](int kk) { return (uint32_t)qraw[h * 128 + chan_of<PS>(sl, t, kk)]; };
        uint2 w;
        w.x = hmul2(qh(0) | (qh(1) << 16), s4);
        w.y = hmul2(qh(2) | (qh(3) << 16), s4);
        qpair[i] = w;
    }
    __syncwarp();
}

// The QK B operand column of a lane: column 2h carries the fp16 hi part of head h's
// folded query, column 2h+1 the lo part.
struct ColConst {
    bool lo;
};
__device__ __forceinline__ ColConst col_const(bool lo_col) { return ColConst{lo_col}; }

// B operands of one 16-channel slab from the page's (scale, min) words kmA..kmD of
// channels chan_of(sl, t, 0..3): the folded query (hi or lo part by column) and
// q * 2^-4 for the min mma (zero in lo columns); A operand of the min mma.
//   hi column: t = fl16(q s);  lo column: fl16(t - q s), exact (fused) -- the residual
//   with its sign flipped, so a head's logit is (hi column) - (lo column).
struct SlabB {
    uint32_t b0, b1, c0, c1, am0, am1;
};
__device__ __forceinline__ SlabB slab_b(uint2 qp, uint32_t kmA, uint32_t kmB, uint32_t kmC, uint32_t kmD,
                                        const ColConst &cc) {
    SlabB r;
    const uint32_t s01 = prmt(kmA, kmB, 0x5410), s23 = prmt(kmC, kmD, 0x5410);
    const uint32_t t01 = hmul2(qp.x, s01), t23 = hmul2(qp.y, s23);
    if (cc.lo) {
        r.b0 = hfma2(qp.x ^ 0x80008000u, s01, t01);
        r.b1 = hfma2(qp.y ^ 0x80008000u, s23, t23);
        r.c0 = r.c1 = 0u;
    } else {
        r.b0 = t01;
        r.b1 = t23;
        r.c0 = qp.x;
        r.c1 = qp.y;
    }
    r.am0 = prmt(kmA, kmB, 0x7632);  // (min A, min B)
    r.am1 = prmt(kmC, kmD, 0x7632);  // (min C, min D)
    return r;
}

// 2^x with the hardware approximation (relative error about 2^-22; -inf gives 0).
// The softmax weights feed fp16 operands, so this is far below their rounding.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The lane's share of a 16-channel slab's B operands, prepared once per tile by
// prep_slabs(): lane (sl, t) turns the (scale, min) words of its channels chan_of(sl,
// t, 0..3) into {scales of channels 0, 1 | 2, 3; mins of 0, 1 | 2, 3} (half2 each), in
// place over the tile's (scale, min) row (32 lanes x 16 bytes = the row's 512 bytes).
template <int PS>
__device__ __forceinline__ void prep_slabs(unsigned char *km_row) {
    const int lane = threadIdx.x & 31, sl = lane >> 2, t = lane & 3;
    uint32_t *km = reinterpret_cast<uint32_t *>(km_row);
    const uint32_t a = km[chan_of<PS>(sl, t, 0)], b = km[chan_of<PS>(sl, t, 1)];
    const uint32_t c = km[chan_of<PS>(sl, t, 2)], d = km[chan_of<PS>(sl, t, 3)];
    __syncwarp();
    reinterpret_cast<uint4 *>(km_row)[lane] =
        make_uint4(prmt(a, b, 0x5410), prmt(c, d, 0x5410), prmt(a, b, 0x7632), prmt(c, d, 0x7632));
    __syncwarp();
}

__device__ __forceinline__ uint32_t lop_xor_and(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(r) : "r"(a), "r"(b), "r"(c));  // (a ^ b) & c
    return r;
}

__device__ __forceinline__ void issue_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    bulk_g2s(dst, src, bytes, bar);
}

// Lengths of sequence u: the call's (dense cache) or its batch slot's (paged cache:
// KIVI, keys and values packed alike, no local window).
struct SeqLen {
    int64_t n_sink, T_k, n_kres, T_v, n_vres, n_local, local_head, L, n_fast;
};
template <bool PG>
__device__ __forceinline__ SeqLen seq_len(const DecodeParams &p, int u) {
    SeqLen s;
    if (!PG) {
        s.n_sink = p.n_sink;
        s.T_k = p.T_k;
        s.n_kres = p.n_kres;
        s.T_v = p.T_v;
        s.n_vres = p.n_vres;
        s.n_local = p.n_local;
        s.local_head = p.local_head;
        s.L = p.L;
        s.n_fast = p.n_fast;
    } else {
        const int4 ln = __ldg(reinterpret_cast<const int4 *>(p.lens) + u / p.H_kv);
        s.n_sink = ln.x;
        s.T_k = s.T_v = ln.y;
        s.n_kres = s.n_vres = ln.z;
        s.n_local = 0;
        s.local_head = 0;
        s.L = (int64_t)ln.x + ln.y + ln.z;
        s.n_fast = ((int64_t)ln.y * p.bits) >> 8;  // tiles of 256 / bits tokens
    }
    return s;
}

// Page index (page-major buffers) of logical page j of sequence u.  Dense: u * max_T/G
// + j.  Paged: page_table row of u's batch slot, read 32 entries at a time into one
// register per lane; lookups are warp-wide (shuffles) and must be made by all lanes.
template <bool PG>
struct PageIds {
    int64_t dense0 = 0;
    __device__ void set(const DecodeParams &p, int u) { dense0 = (int64_t)u * (p.max_T / p.G); }
    __device__ __forceinline__ int64_t operator()(const DecodeParams &, int64_t j) const { return dense0 + j; }
};
template <>
struct PageIds<true> {
    const int32_t *row = nullptr;  // the slot's table row
    int64_t dense0 = 0;            // head h
    int base = 0, reg = 0;         // entries [base, base + 32) are in reg (lane j: base + j)
    __device__ void set(const DecodeParams &p, int u) {
        const int b = u / p.H_kv;
        dense0 = u - b * p.H_kv;
        row = p.ptab + (size_t)b * p.ptab_stride;
        base = -(1 << 30);  // nothing loaded
    }
    __device__ __forceinline__ int64_t operator()(const DecodeParams &p, int64_t j) {
        if (j < base || j >= base + 32) {
            base = (int)j;
            const int e = (int)j + (int)(threadIdx.x & 31);
            reg = e < p.ptab_stride ? __ldg(row + e) : 0;
            if (reg < 0 || reg >= p.n_pages) {  // a bad table entry reads page 0
                if (e < p.ptab_stride) report(p.status, 2 /*KVQ_DEV_BAD_STATE*/);
                reg = 0;
            }
        }
        return (int64_t)__shfl_sync(0xffffffffu, reg, (int)j - base) * p.H_kv + dense0;
    }
};

// Pre-RoPE keys (KVQuant notes, mechanism two).  The tables in shared memory:
//   - theta_j as a two-float hi + lo, 128 entries each (the kernel argument);
//   - for the packed tiles, the turns by k theta_j within a word row (k < 16, j < 64):
//     one float4 (cos, cos, sin, sin) of k = 2m, 2m + 1 per (m, j) at kRopeCS, and one
//     float2 of their negated sines at kRopeNS (index m * 64 + j).
constexpr int kRopeHi = 0, kRopeLo = 128, kRopeArgFloats = 256;
constexpr int kRopeCS = kRopeArgFloats, kRopeNS = kRopeCS + 8 * 64 * 4, kRopeFloats = kRopeNS + 8 * 64 * 2;

// (cos, sin) of pos * theta_j, the angle reduced modulo 2 pi: the product's rounding
// error is recovered with an FMA and 2 pi is subtracted in two parts (the Cody-Waite
// reduction), so the reduced angle stays within a few 1e-7 rad for any position
// below 2^24; then the sine and cosine of an angle in [-pi, pi].
__device__ __forceinline__ float2 rope_cs(float pos, float th_hi, float th_lo) {
    const float ph = pos * th_hi;
    const float pe = fmaf(pos, th_hi, -ph);  // pos * th_hi - ph, exactly
    const float pl = fmaf(pos, th_lo, pe);
    const float n = rintf(ph * 0.159154943091895336f);   // 1 / (2 pi)
    float r = fmaf(-n, 6.28318548202514648f, ph);         // 2 pi rounded to float
    r = fmaf(-n, -1.74845553146951720e-7f, r) + pl;       // 2 pi minus that
    float s, c;
    __sincosf(r, &s, &c);
    return make_float2(c, s);
}

// Packed fp32 pairs (Blackwell's f32x2 arithmetic): two lanes of fp32, each rounded as
// the scalar operation would be.
__device__ __forceinline__ uint64_t f2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2x(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------------------
// Packed tiles
// ---------------------------------------------------------------------------
template <int KB, int VB, bool KITTY, bool PG = false, bool RP = false>
struct FastWarp {
    using T = Tile<KB, VB>;
    using CK = typename T::K;
    using CV = typename T::V;
    const DecodeParams &p;
    unsigned char *wbase;
    WarpSmem L;
    int u, lane;
    uint64_t *bars;
    uint32_t phase = 0;    // bit s: parity of the next completion of slot s
    uint32_t pending = 0;  // bit s: slot s has copies in flight
    PageIds<PG> pid;       // page index of a logical page of sequence u
    const float *rt = nullptr;  // RP: the RoPE tables
    // Dense caches: this lane's copy of a key batch and of a value batch (codes rows,
    // the key (scale, min) row, Kitty planes) is at  base + (tile >> tpp_shift) * pstride
    // + (tile & tiles-per-page - 1) * tstride  (bytes), set per sequence by set_copies();
    // bytes == 0: no copy.  vm_base: the value (scale, min) rows of the sequence.
    struct CopyLane {
        const unsigned char *base;
        uint32_t pstride, tstride, dst, bytes;
    };
    CopyLane ck{};         // Kitty: this lane's high-plane row or boost-index copy
    // Dense caches: tile ti of sequence u (pages contiguous, whole tiles per page) has
    // its key codes at kc_base + ti * 8 D 4 bytes, its value codes at vc_base + ti *
    // V_ROWS TOK 4, its page's key (scale, min) row at km_base + (ti >> tpp_shift) * D 4
    // and its value (scale, min) at vm_base + ti * TOK 4; lane 0 issues those copies.
    const unsigned char *kc_base = nullptr, *km_base = nullptr, *vc_base = nullptr, *vm_base = nullptr;
    uint32_t k_total = 0;  // bytes of a key batch (without the first batch's value meta)
    // ldmatrix: the lane addresses row r = lane & 7 of a row set at logical 16-byte chunk
    // 4 sl + lane / 8 of slab sl, stored at chunk (4 sl + lane / 8) ^ r (kword_pos /
    // vword_pos): 128 (sl / 2) bytes + cx[sl & 1].
    uint32_t cx[2];

    __device__ FastWarp(const DecodeParams &pp, unsigned char *wb)
        : p(pp), wbase(wb), L(KB, VB, KITTY, pp.n_boost), u(0), lane(threadIdx.x & 31) {
        bars = reinterpret_cast<uint64_t *>(wbase + L.bars);
        cx[0] = 16u * (uint32_t)((lane >> 3) ^ (lane & 7));
        cx[1] = 16u * (uint32_t)((4 + (lane >> 3)) ^ (lane & 7));
    }
    __device__ __forceinline__ uint32_t chunk(int sl) const { return 128u * (uint32_t)(sl >> 1) + cx[sl & 1]; }
    __device__ unsigned char *kslot(int s) const { return wbase + L.k0 + s * L.ksz; }
    __device__ unsigned char *vslot(int s) const { return wbase + L.v0 + s * L.vsz; }
    __device__ unsigned char *vmslot(int s) const { return wbase + L.vm0 + s * L.vmsz; }

    __device__ void init_bars() {
        if (lane == 0) {
            for (int s = 0; s < kBars; s++) mbar_init(&bars[s], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }

    __device__ bool wait_slot(int s) {
        const bool ok = mbar_wait(&bars[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        pending &= ~(1u << s);
        return ok;
    }

    // Copies of sequence u (dense caches): lane 0 the tile's code rows, the page's key
    // (scale, min) row and the value blocks; Kitty lanes 10..17 the high-plane rows and
    // lane 18 the boost index.
    __device__ void set_copies() {
        const int64_t pg0 = (int64_t)u * (p.max_T / p.G);
        const int nb = KITTY ? p.n_boost : 0;
        kc_base = reinterpret_cast<const unsigned char *>(p.k_codes) + (size_t)pg0 * (p.G / CK::FPI) * T::D * 4;
        km_base = reinterpret_cast<const unsigned char *>(p.k_meta) + (size_t)pg0 * T::D * 4;
        vc_base = reinterpret_cast<const unsigned char *>(p.v_codes) + (size_t)pg0 * T::V_ROWS * p.G * 4;
        vm_base = reinterpret_cast<const unsigned char *>(p.v_meta) + (size_t)pg0 * p.G * 4;
        ck = CopyLane{nullptr, 0, 0, 0, 0};
        if (KITTY && nb > 0 && lane >= 10 && lane < 18) {
            const uint32_t row = nb * 4, page = (uint32_t)(p.G / 16) * row;
            ck = CopyLane{reinterpret_cast<const unsigned char *>(p.k_hi) + (size_t)pg0 * page + (lane - 10) * row,
                          page, 8 * row, (uint32_t)(T::OFF_HI + (lane - 10) * hi_stride(nb)), row};
        } else if (KITTY && lane == 18) {
            ck = CopyLane{reinterpret_cast<const unsigned char *>(p.k_bidx) + (size_t)pg0 * T::D, T::D, 0,
                          (uint32_t)(T::OFF_HI + 8 * hi_stride(nb)), T::D};
        }
        k_total = 8 * T::D * 4 + T::D * 4 + (KITTY ? 8 * nb * 4 + T::D : 0);
    }
    __device__ __forceinline__ const unsigned char *copy_src(const CopyLane &c, int64_t ti) const {
        return c.base + (size_t)(ti >> p.tpp_shift) * c.pstride + (size_t)(ti & ((1 << p.tpp_shift) - 1)) * c.tstride;
    }

    // Batch K(j): key codes and (scale, min) of tile t0 + j -> key half j & 1, barrier
    // j & 1; the first batch also brings the value (scale, min) of tile t0.
    __device__ void issue_kb(int64_t t0, int j) {
        if constexpr (!PG) {
            const int s = j & 1;
            const int64_t ti = t0 + j;
            pending |= 1u << s;
            unsigned char *st = kslot(s);
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[s], k_total + (j == 0 ? T::TOK * 4 : 0));
                issue_copy(st + T::OFF_K, kc_base + (size_t)ti * (8 * T::D * 4), 8 * T::D * 4, &bars[s]);
                issue_copy(st + T::OFF_KM, km_base + (size_t)(ti >> p.tpp_shift) * (T::D * 4), T::D * 4, &bars[s]);
                if (j == 0) issue_copy(vmslot(0), vm_base + (size_t)ti * (T::TOK * 4), T::TOK * 4, &bars[s]);
            }
            if (KITTY) {  // the high-plane rows after lane 0's expect-tx
                __syncwarp();
                if (ck.bytes) issue_copy(st + ck.dst, copy_src(ck, ti), ck.bytes, &bars[s]);
            }
            return;
        }
        const int s = j & 1;
        const int64_t ti = t0 + j;
        pending |= 1u << s;
        unsigned char *st = kslot(s);
        const int nb = KITTY ? p.n_boost : 0;
        const uint32_t bytes = 8 * T::D * 4 + T::D * 4 + (KITTY ? 8 * nb * 4 + T::D : 0) + (j == 0 ? T::TOK * 4 : 0);
        // tiles per page: a power of two; pg: page index, tin: tile within the page
        const int64_t pg = pid(p, ti >> p.tpp_shift), tin = ti & ((1 << p.tpp_shift) - 1);
        const int i = lane;
        if (i == 0) {
            mbar_arrive_expect_tx(&bars[s], bytes);
            issue_copy(st + T::OFF_K, p.k_codes + ((size_t)pg * (p.G / CK::FPI) + tin * 8) * T::D, 8 * T::D * 4,
                       &bars[s]);
            issue_copy(st + T::OFF_KM, p.k_meta + (size_t)pg * T::D * 2, T::D * 4, &bars[s]);
            if (j == 0)
                issue_copy(vmslot(0), p.v_meta + ((size_t)pg * p.G + tin * T::TOK) * 2, T::TOK * 4, &bars[s]);
        }
        if (KITTY) __syncwarp();  // the high-plane rows after lane 0's expect-tx
        if (KITTY && nb > 0 && i >= 10 && i < 18) {
            const int r = i - 10;
            issue_copy(st + T::OFF_HI + r * hi_stride(nb), p.k_hi + ((size_t)pg * (p.G / 16) + tin * 8 + r) * nb,
                       nb * 4, &bars[s]);
        } else if (KITTY && i == 18) {
            issue_copy(st + T::OFF_HI + 8 * hi_stride(nb), p.k_bidx + (size_t)pg * T::D, T::D, &bars[s]);
        }
    }

    // Batch V(j): value codes of tile t0 + j -> value half j & 1 and, if tile j + 1
    // exists, its value (scale, min) -> value-meta row (j + 1) & 1; barrier 2 + (j & 1).
    __device__ void issue_vb(int64_t t0, int j, int64_t n) {
        if constexpr (!PG) {
            const int s = 2 + (j & 1);
            const int64_t ti = t0 + j;
            const bool meta = j + 1 < n;
            pending |= 1u << s;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[s], T::V_ROWS * T::TOK * 4 + (meta ? T::TOK * 4 : 0));
                issue_copy(vslot(j & 1), vc_base + (size_t)ti * (T::V_ROWS * T::TOK * 4), T::V_ROWS * T::TOK * 4,
                           &bars[s]);
                if (meta) issue_copy(vmslot((j + 1) & 1), vm_base + (size_t)(ti + 1) * (T::TOK * 4), T::TOK * 4, &bars[s]);
            }
            return;
        }
        const int s = 2 + (j & 1);
        const int64_t ti = t0 + j;
        const bool meta = j + 1 < n;
        pending |= 1u << s;
        unsigned char *st = vslot(j & 1);
        const int tmask = (1 << p.tpp_shift) - 1;
        const int64_t pg = pid(p, ti >> p.tpp_shift), tin = ti & tmask;
        const int64_t pg1 = meta ? pid(p, (ti + 1) >> p.tpp_shift) : 0, off1 = ((ti + 1) & tmask) * T::TOK;
        if (lane == 0) {  // the tile's value rows: one block of the tile-major page
            mbar_arrive_expect_tx(&bars[s], T::V_ROWS * T::TOK * 4 + (meta ? T::TOK * 4 : 0));
            issue_copy(st, p.v_codes + ((size_t)pg * p.G + tin * T::TOK) * T::V_ROWS, T::V_ROWS * T::TOK * 4,
                       &bars[s]);
            if (meta) issue_copy(vmslot((j + 1) & 1), p.v_meta + ((size_t)pg1 * p.G + off1) * 2, T::TOK * 4, &bars[s]);
        }
    }

    // 4 A registers of row set J (code width of C) from the split words (rows g /
    // g+8, k pairs).
    template <typename C, int J>
    __device__ __forceinline__ static void frag(const uint32_t (&x)[4], const uint32_t (&xs)[4], uint32_t (&a)[4]) {
        constexpr uint32_t M = C::MASK0 << (32 / C::FPI * C::template jj<J>());
#pragma unroll
        for (int r = 0; r < 4; r++) a[r] = (J < C::JDIRECT ? x[r] : xs[r]) & M;
    }
    template <typename C, int J>
    __device__ __forceinline__ static constexpr float unscale() {
        return (float)(1u << (24 - 32 / C::FPI * C::template jj<J>()));
    }
    // ldmatrix words W0..W3 (segments c = 0..3) -> k-paired registers (k = 2t, 2t+1 |
    // 2t+8, 2t+9) for rows g (low halves) and g+8 (high halves); xs: x >> SH of C.
    template <typename C>
    __device__ __forceinline__ static void split(const uint32_t (&w)[4], uint32_t (&x)[4], uint32_t (&xs)[4]) {
        if (T::P == 8) {  // pairs (t, t+8) and (t+4, t+12)
            x[0] = prmt(w[0], w[2], 0x5410);
            x[1] = prmt(w[0], w[2], 0x7632);
            x[2] = prmt(w[1], w[3], 0x5410);
            x[3] = prmt(w[1], w[3], 0x7632);
        } else {          // pairs (t, t+4) and (t+8, t+12)
            x[0] = prmt(w[0], w[1], 0x5410);
            x[1] = prmt(w[0], w[1], 0x7632);
            x[2] = prmt(w[2], w[3], 0x5410);
            x[3] = prmt(w[2], w[3], 0x7632);
        }
#pragma unroll
        for (int r = 0; r < 4; r++) xs[r] = x[r] >> C::SH;
    }
    // S row sets of a key slab.  Z: the first slab of a tile, whose accumulators start
    // from zero.
    template <bool Z = false>
    __device__ __forceinline__ static void mma_sets(float (&acc)[CK::NJ][4], const uint32_t (&x)[4],
                                                    const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                                                      \
    if (J < CK::NJ) {                                                                  \
        frag<CK, J>(x, xs, a);                                                         \
        if (Z) mma_16816_z(acc[J % CK::NJ], a[0], a[1], a[2], a[3], b0, b1);           \
        else mma_16816(acc[J % CK::NJ], a[0], a[1], a[2], a[3], b0, b1);              \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }
    // O row sets of value channel set `set`.
    __device__ __forceinline__ static void mma_sets_o(float (&O)[8][4], int set, const uint32_t (&x)[4],
                                                      const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                                                  \
    if (J < CV::NJ) {                                                              \
        frag<CV, J>(x, xs, a);                                                     \
        mma_16816(O[set * CV::NJ + (J % CV::NJ)], a[0], a[1], a[2], a[3], b0, b1); \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }

    // One 16-channel slab of S = Kcodes . q' (+ the min mma) for the key half in st;
    // slab 0 starts the accumulators from zero.
    // KIVI tiles (not Kitty, keys as stored) prepare their slabs' scales and mins once
    // per tile (prep_slabs); Kitty's boost pass and the pre-RoPE path read the row as it
    // was copied.
    static constexpr bool kPrep = !KITTY && !RP;

    __device__ __forceinline__ void qk_slab(int sl, const unsigned char *st, float (&acc)[CK::NJ][4],
                                            float (&cm)[4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const uint2 qp = reinterpret_cast<const uint2 *>(wbase + L.qpair)[((gq >> 1) * 8 + sl) * 4 + t];
        uint32_t b0, b1, am0, am1, c0, c1;
        if constexpr (kPrep) {
            // hi column (even gq): fl16(q s); lo column: fl16(q s) - q s, the sign-flipped
            // exact residual, formed as fma(q * m, s, fl16(q s)) with m = 0 or -1 by column
            const uint4 sm = reinterpret_cast<const uint4 *>(st + T::OFF_KM)[sl * 4 + t];
            const uint32_t m = (gq & 1) ? 0xBC00BC00u : 0u;  // half2(-1, -1) or 0
            b0 = hfma2(hmul2(qp.x, m), sm.x, hmul2(qp.x, sm.x));
            b1 = hfma2(hmul2(qp.y, m), sm.y, hmul2(qp.y, sm.y));
            am0 = sm.z;
            am1 = sm.w;
            c0 = qp.x;  // the min mma: q in both columns of a head (only the hi one is read)
            c1 = qp.y;
        } else {
            const uint32_t *km = reinterpret_cast<const uint32_t *>(st + T::OFF_KM);
            const SlabB b = slab_b(qp, km[chan_of<T::P>(sl, t, 0)], km[chan_of<T::P>(sl, t, 1)],
                                   km[chan_of<T::P>(sl, t, 2)], km[chan_of<T::P>(sl, t, 3)],
                                   col_const((gq & 1) != 0));
            b0 = b.b0;
            b1 = b.b1;
            am0 = b.am0;
            am1 = b.am1;
            c0 = b.c0;
            c1 = b.c1;
        }
        if (sl == 0) mma_16816_z(cm, am0, am0, am1, am1, c0, c1);
        else mma_16816(cm, am0, am0, am1, am1, c0, c1);
        uint32_t w[4], x[4], xs[4];
        ldmatrix_x4(w, smem_u32(st + T::OFF_K) + (lane & 7) * T::K_STRIDE + chunk(sl));
        split<CK>(w, x, xs);
        if (sl == 0) mma_sets<true>(acc, x, xs, b0, b1);
        else mma_sets<false>(acc, x, xs, b0, b1);
    }

    // Kitty: S += hi-plane codes . (4 q') over the boosted slots.
    __device__ void qk_boost(const unsigned char *st, float (&acc)[CK::NJ][4]) const {
        static_assert(!KITTY || KB == 2, "Kitty planes are 2-bit");
        const int gq = lane >> 2, t = lane & 3, hq = gq >> 1;
        const int nb = p.n_boost;
        const uint32_t *km = reinterpret_cast<const uint32_t *>(st + T::OFF_KM);
        const uint8_t *bi = st + T::OFF_HI + 8 * hi_stride(nb);
        uint8_t *invb = wbase + L.invb;
        const uint16_t *qraw = reinterpret_cast<const uint16_t *>(wbase + L.qraw);
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int ch = lane * 4 + r;
            const int sl = bi[ch];
            if (sl < nb) invb[sl] = (uint8_t)ch;
        }
        __syncwarp();
        const uint32_t s4 = 0x44004400u;  // half2(4, 4): the high plane carries bits 2..3
        const uint32_t hb = smem_u32(st + T::OFF_HI) + (lane & 7) * hi_stride(nb) + 16 * (lane >> 3);
        for (int s2 = 0; s2 < nb / 16; s2++) {
            uint32_t km4[4], q2[2];
            uint16_t qv[4];
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
                const int ch = invb[chan_of<T::P>(s2, t, kk)] & (T::D - 1);
                km4[kk] = km[ch];
                qv[kk] = qraw[hq * 128 + ch];
            }
            q2[0] = hmul2((uint32_t)qv[0] | ((uint32_t)qv[1] << 16), 0x2C002C00u);
            q2[1] = hmul2((uint32_t)qv[2] | ((uint32_t)qv[3] << 16), 0x2C002C00u);
            q2[0] = hmul2(q2[0], s4);
            q2[1] = hmul2(q2[1], s4);
            const SlabB b = slab_b(make_uint2(q2[0], q2[1]), km4[0], km4[1], km4[2], km4[3], col_const((gq & 1) != 0));
            uint32_t w[4], x[4], xs[4];
            ldmatrix_x4(w, hb + 64 * s2);
            split<CK>(w, x, xs);
            mma_sets(acc, x, xs, b.b0, b.b1);
        }
        __syncwarp();
    }

    // One PV step: token slab sl / channel set `set` of the value half in st.
    __device__ __forceinline__ void pv_step(int step, const unsigned char *st, const uint16_t *pb,
                                            float (&O)[8][4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const int sl = step / T::NSET, set = step % T::NSET;
        uint2 bp = make_uint2(0u, 0u);
        if (gq < 4) bp = *reinterpret_cast<const uint2 *>(pb + gq * T::PROW + 16 * sl + 4 * t);
        uint32_t w[4], x[4], xs[4];
        ldmatrix_x4(w, smem_u32(st) + (set * 8 + (lane & 7)) * T::V_STRIDE + chunk(sl));
        split<CV>(w, x, xs);
        mma_sets_o(O, set, x, xs, bp.x, bp.y);
    }

    // Softmax of a tile, first part: logits z (log2 units) from the S accumulators,
    // the new running maximum, l and mn rescaled to it.  Returns the factors by which
    // O must be rescaled once the previous tile's PV is in (a0 / a1: columns 2t /
    // 2t+1); *grow tells whether any head's maximum rose.
    __device__ __forceinline__ void softmax_begin(const float (&acc)[CK::NJ][4], const float (&cm)[4],
                                                  float (&z)[CK::NJ][2], float &m, float &l, float &mn,
                                                  float &a0, float &a1, bool &grow) const {
        float a;
        softmax_begin_a(acc, cm, z, m, l, mn, a, grow);
        const int t = lane & 3;
        a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
        a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
    }
    // The same; `a` is the rescale factor of the lane's head (lane & 3).
    __device__ __forceinline__ void softmax_begin_a(const float (&acc)[CK::NJ][4], const float (&cm)[4],
                                                    float (&z)[CK::NJ][2], float &m, float &l, float &mn,
                                                    float &a, bool &grow) const {
        const float C = kLog2e * rsqrtf((float)T::D) / kQScale;
        const float cst = cm[0] * C;  // row g, column 2t: sum_d q_d min_d of head t
        float tm = -INFINITY;
#define KVQ_Z(J)                                                                        \
    if (J < CK::NJ) {                                                                   \
        const float f = unscale<CK, J>() * C;                                           \
        z[J % CK::NJ][0] = fmaf(acc[J % CK::NJ][0] - acc[J % CK::NJ][1], f, cst);       \
        z[J % CK::NJ][1] = fmaf(acc[J % CK::NJ][2] - acc[J % CK::NJ][3], f, cst);       \
        tm = fmaxf(tm, fmaxf(z[J % CK::NJ][0], z[J % CK::NJ][1]));                      \
    }
        KVQ_Z(0) KVQ_Z(1) KVQ_Z(2) KVQ_Z(3) KVQ_Z(4) KVQ_Z(5) KVQ_Z(6) KVQ_Z(7)
#undef KVQ_Z
        softmax_max(tm, m, l, mn, a, grow);
    }
    // The running maximum from the tile's maximum tm of the lane's head.
    __device__ __forceinline__ static void softmax_max(float tm, float &m, float &l, float &mn, float &a,
                                                       bool &grow) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
        const float nm = fmaxf(m, tm);
        a = ex2(m - nm);  // 0 while m is -inf
        grow = __any_sync(0xffffffffu, nm > m);
        m = nm;
        l *= a;
        mn *= a;
    }
    // The same from logits z already in log2 units (pre-RoPE path).
    __device__ __forceinline__ void softmax_begin_z(const float (&z)[CK::NJ][2], float &m, float &l, float &mn,
                                                    float &a0, float &a1, bool &grow) const {
        float tm = -INFINITY, a;
#pragma unroll
        for (int j = 0; j < CK::NJ; j++) tm = fmaxf(tm, fmaxf(z[j][0], z[j][1]));
        softmax_max(tm, m, l, mn, a, grow);
        const int t = lane & 3;
        a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
        a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
    }

    // Pre-RoPE keys (KVQuant notes, mechanism two): key t is dequantized in fp32, its
    // channel pair (2j, 2j+1) turned by t * theta_j and dotted with the query on the
    // CUDA cores.  Lane (g, t) takes word row g -- KFPI tokens at positions pos0 + k --
    // and the pairs j = t + 4i.  The turn by (pos0 + k) theta_j is split in two: the
    // query turns back by pos0 theta_j once per pair (q . R(a + b) k = (R(a)^T q) .
    // (R(b) k)), the key by k theta_j from the in-row table.  This call covers i in
    // [i0, i0 + n).
    //
    // Codes become floats with one LOP3 each: code c at bit offset o (o + KB <= 16) of
    // a word, OR-ed into the mantissa of 2^(23 - o), is the float 2^(23 - o) + c, so
    // one subtraction leaves c exactly.  Tokens of the upper half-word come from the
    // word shifted right by 16.
    __device__ __forceinline__ void qk_rope_part(const unsigned char *st, float pos0, int i0, int n,
                                                 float (&acc)[CK::FPI][4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const uint16_t *qraw = reinterpret_cast<const uint16_t *>(wbase + L.qraw);
        constexpr int HALF = CK::FPI / 2;
        constexpr uint32_t MASK = (1u << KB) - 1u;
        const float4 *tcs = reinterpret_cast<const float4 *>(rt + kRopeCS);
        const float2 *tns = reinterpret_cast<const float2 *>(rt + kRopeNS);
        // tokens 2k and 2k+1 of the lane's row share each f32x2 operation
        uint64_t *acc2 = reinterpret_cast<uint64_t *>(&acc[0][0]);  // [FPI/2][4]: (token 2k, 2k+1)
#pragma unroll
        for (int ii = 0; ii < 2; ii++) {
            if (ii >= n) break;
            const int pr = t + 4 * (i0 + ii);
            // words 2 pr, 2 pr + 1 of row gq: chunk pr / 2, stored at chunk (pr / 2) ^ gq
            const uint2 w = *reinterpret_cast<const uint2 *>(st + T::OFF_K + gq * T::K_STRIDE +
                                                             16 * ((pr >> 1) ^ gq) + 8 * (pr & 1));
            const uint2 km = *reinterpret_cast<const uint2 *>(st + T::OFF_KM + 8 * pr);
            const float2 sa = unpack_half2(km.x), sb = unpack_half2(km.y);  // (scale, min)
            const uint64_t SA = f2(sa.x, sa.x), MA = f2(sa.y, sa.y), SB = f2(sb.x, sb.x), MB = f2(sb.y, sb.y);
            // the query of each head turned back by pos0 theta_j
            const float2 cs = rope_cs(pos0, rt[kRopeHi + pr], rt[kRopeLo + pr]);
            uint64_t QA[4], QB[4];
#pragma unroll
            for (int h = 0; h < 4; h++) {
                const float2 qq = unpack_half2(*reinterpret_cast<const uint32_t *>(qraw + h * 128 + 2 * pr));
                const float a = fmaf(qq.x, cs.x, qq.y * cs.y), b = fmaf(qq.y, cs.x, -(qq.x * cs.y));
                QA[h] = f2(a, a);
                QB[h] = f2(b, b);
            }
            const uint32_t xs[2] = {w.x, w.x >> 16}, ys[2] = {w.y, w.y >> 16};
#pragma unroll
            for (int k = 0; k < CK::FPI; k += 2) {
                const int o0 = KB * (k % HALF), o1 = KB * ((k + 1) % HALF);
                const uint32_t e0 = (uint32_t)(150 - o0) << 23, e1 = (uint32_t)(150 - o1) << 23;
                const uint32_t sx = xs[k / HALF], sy = ys[k / HALF];
                const uint64_t MAGIC = f2(-__uint_as_float(e0), -__uint_as_float(e1));
                const uint64_t fa = add2(f2(__uint_as_float((sx & (MASK << o0)) | e0),
                                            __uint_as_float((sx & (MASK << o1)) | e1)), MAGIC);
                const uint64_t fb = add2(f2(__uint_as_float((sy & (MASK << o0)) | e0),
                                            __uint_as_float((sy & (MASK << o1)) | e1)), MAGIC);
                const uint64_t ka = fma2(fa, SA, MA), kb = fma2(fb, SB, MB);
                // turn by k theta_j: (ka, kb) -> (ka cos - kb sin, ka sin + kb cos)
                const float4 cs4 = tcs[(k / 2) * 64 + pr];
                const float2 ns2 = tns[(k / 2) * 64 + pr];
                const uint64_t C = f2(cs4.x, cs4.y), S = f2(cs4.z, cs4.w), NS = f2(ns2.x, ns2.y);
                const uint64_t ra = fma2(ka, C, mul2(kb, NS)), rb = fma2(ka, S, mul2(kb, C));
#pragma unroll
                for (int h = 0; h < 4; h++) acc2[(k / 2) * 4 + h] = fma2(QA[h], ra, fma2(QB[h], rb, acc2[(k / 2) * 4 + h]));
            }
        }
    }
    // The four lanes of a word row hold partial sums over their pairs for all heads:
    // a reduce-scatter leaves head t in lane t; z in log2 units, in the mma path's
    // layout (z[J][0] token KFPI g + J, z[J][1] token KFPI g + KFPI/2 + J).
    __device__ __forceinline__ void qk_rope_finish(float (&acc)[CK::FPI][4], float (&z)[CK::NJ][2]) const {
        const int t = lane & 3;
        const bool b2 = (t & 2) != 0, b1 = (t & 1) != 0;
        const float C = kLog2e * rsqrtf((float)T::D);
        float zt[CK::FPI];
        // acc holds (token 2k, token 2k+1) pairs per head: entry [2k + e][h] is at pair
        // (k, h), element e
        const float *af = &acc[0][0];
        auto A = [&](int tk, int h) { return af[((tk >> 1) * 4 + h) * 2 + (tk & 1)]; };
#pragma unroll
        for (int k = 0; k < CK::FPI; k++) {
            const float s0 = b2 ? A(k, 0) : A(k, 2), s1 = b2 ? A(k, 1) : A(k, 3);
            float k0 = b2 ? A(k, 2) : A(k, 0), k1 = b2 ? A(k, 3) : A(k, 1);
            k0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            k1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            const float s2 = b1 ? k0 : k1;
            float kk = b1 ? k1 : k0;
            kk += __shfl_xor_sync(0xffffffffu, s2, 1);
            zt[k] = kk * C;
        }
#pragma unroll
        for (int j = 0; j < CK::NJ; j++) {
            z[j][0] = zt[j];
            z[j][1] = zt[j + CK::FPI / 2];
        }
    }
    // The whole pre-RoPE QK of a key half: a rolled loop over groups of two pairs (the
    // unrolled form overflows the instruction cache).
    __device__ __forceinline__ void qk_rope(const unsigned char *st, float pos0, float (&acc)[CK::FPI][4],
                                            float (&z)[CK::NJ][2]) const {
        zero_acc(acc);
#pragma unroll 1
        for (int i0 = 0; i0 < T::D / 8; i0 += 2) qk_rope_part(st, pos0, i0, 2, acc);
        qk_rope_finish(acc, z);
    }
    __device__ __forceinline__ static void zero_acc(float (&acc)[CK::FPI][4]) {
#pragma unroll
        for (int k = 0; k < CK::FPI; k++)
#pragma unroll
            for (int h = 0; h < 4; h++) acc[k][h] = 0.f;
    }

    // Position of tile token tk in a p' row: the k index of the PV B operand under the
    // pairing of split() (slab tk / 16; segment c = (tk % 16) / 4 and lane t = tk % 4
    // of the ldmatrix words).
    __device__ __forceinline__ static int ppos(int tk) {
        const int c = (tk >> 2) & 3, cp = T::P == 8 ? ((c & 1) << 1) | (c >> 1) : c;
        return 16 * (tk >> 4) + 4 * (tk & 3) + cp;
    }

    // Softmax of a tile, row set j: p = exp2(z - m) of the lane's two tokens (rows g
    // and g+8: tokens KFPI g + j and KFPI g + KFPI/2 + j), their sums, and p' = p *
    // scale_v into the tile's p' buffer.
    // The value (scale, min) words of the lane's tokens KFPI g .. KFPI g + KFPI - 1,
    // 16 bytes at a time.
    __device__ __forceinline__ void load_vm(const unsigned char *vms, uint32_t (&vm)[CK::FPI]) const {
        const uint4 *src = reinterpret_cast<const uint4 *>(vms) + (CK::FPI / 4) * (lane >> 2);
#pragma unroll
        for (int i = 0; i < CK::FPI / 4; i++) {
            const uint4 w = src[i];
            vm[4 * i] = w.x;
            vm[4 * i + 1] = w.y;
            vm[4 * i + 2] = w.z;
            vm[4 * i + 3] = w.w;
        }
    }
    __device__ __forceinline__ void softmax_chunk(int j, const float (&z)[CK::NJ][2], const uint32_t (&vm)[CK::FPI],
                                                  uint16_t *pb, float m, float &l, float &mn) const {
        const int gq = lane >> 2, t = lane & 3;
        const int tk0 = CK::FPI * gq + j, tk1 = tk0 + CK::FPI / 2;
        const float2 sm0 = unpack_half2(vm[j]), sm1 = unpack_half2(vm[j + CK::FPI / 2]);
        const float p0 = ex2(z[j][0] - m), p1 = ex2(z[j][1] - m);
        l += p0 + p1;
        mn = fmaf(p0, sm0.y, fmaf(p1, sm1.y, mn));
        uint16_t *row = pb + t * T::PROW;
        if (T::P_ADJ) {
            *reinterpret_cast<uint32_t *>(row + ppos(tk0)) = pack_half2(p0 * sm0.x, p1 * sm1.x);
        } else {
            row[ppos(tk0)] = __half_as_ushort(__float2half_rn(p0 * sm0.x));
            row[ppos(tk1)] = __half_as_ushort(__float2half_rn(p1 * sm1.x));
        }
    }

    __device__ __forceinline__ void zero(float (&a)[CK::NJ][4], float (&cm)[4]) const {
#pragma unroll
        for (int j = 0; j < CK::NJ; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) a[j][e] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; e++) cm[e] = 0.f;
    }

    // Tiles [t0, t1) of sequence uu; writes the warp's partial [4][D+4] to `part`.
    // Software pipeline, iteration i: PV of tile i interleaved slab by slab with QK of
    // tile i+1, then the softmax of tile i+1 (its p' goes to the other p' buffer; O is
    // rescaled only if a head's running maximum rose).
    // Copies: batch K(j) = key codes + (scale, min) of tile j -> key half j&1 (barrier
    // j&1); batch V(j) = value codes of j + value (scale, min) of j+1 -> value half
    // j&1, meta row (j+1)&1 (barrier 2 + j&1).  Both are issued two tiles ahead, each
    // into a buffer whose previous contents the warp has just finished reading.
    // The first copies of tiles [t0, t1) of sequence uu: batches K(0), V(0), K(1).
    __device__ void start(int uu, int64_t t0, int64_t t1) {
        u = uu;
        pid.set(p, uu);
        if (!PG) set_copies();
        issue_kb(t0, 0);
        issue_vb(t0, 0, t1 - t0);
        if (t1 - t0 > 1) issue_kb(t0, 1);
    }

    // started: start(uu, t0, t1) has issued the first copies already (before the
    // kernel's wait for the preceding kernel in the stream).
    __device__ void run(int uu, int64_t t0, int64_t t1, float *part, bool started = false) {
        u = uu;
        pid.set(p, uu);
        const int64_t n = t1 - t0;
        const QRegs qr = load_q_regs(p, u);  // its loads go out before the first copies
        if (!started) start(uu, t0, t1);
        store_q_warp<T::P>(qr, reinterpret_cast<uint16_t *>(wbase + L.qraw),
                            reinterpret_cast<uint2 *>(wbase + L.qpair));
        uint16_t *pb0 = reinterpret_cast<uint16_t *>(wbase + L.pbuf);
        for (int i = lane; i < 4 * T::PROW; i += 32)  // both p' buffers (2 x 4 rows)
            reinterpret_cast<uint32_t *>(pb0)[i] = 0u;
        __syncwarp();
        float m = -INFINITY, l = 0.f, mn = 0.f;
        float O[8][4];
#pragma unroll
        for (int o = 0; o < 8; o++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[o][e] = 0.f;
        float acc[CK::NJ][4], cm[4];
        float z[CK::NJ][2];
        float accr[RP ? CK::FPI : 1][4];  // RP: per-token partial dot products
        // RP: position of the lane's first token in tile i
        auto rpos = [&](int64_t i) { return (float)(p.n_sink + (t0 + i) * T::TOK + CK::FPI * (lane >> 2)); };
        bool ok = true;

        // prologue: QK(0), softmax(0) (the value (scale, min) of tile 0 came with K(0))
        ok &= wait_slot(0);
        if (kPrep) prep_slabs<T::P>(kslot(0) + T::OFF_KM);
        if (RP) {
            qk_rope(kslot(0), rpos(0), reinterpret_cast<float (&)[CK::FPI][4]>(accr), z);
        } else {
#pragma unroll
            for (int sl = 0; sl < 8; sl++) qk_slab(sl, kslot(0), acc, cm);
            if (KITTY && p.n_boost > 0) qk_boost(kslot(0), acc);
        }
        {
            float a0, a1;
            bool grow;
            if (RP) softmax_begin_z(z, m, l, mn, a0, a1, grow);
            else softmax_begin(acc, cm, z, m, l, mn, a0, a1, grow);
            uint32_t vm[CK::FPI];
            load_vm(vmslot(0), vm);
#pragma unroll
            for (int j = 0; j < CK::NJ; j++) softmax_chunk(j, z, vm, pb0, m, l, mn);
        }
        __syncwarp();
        fence_proxy_async();
        if (n > 2) issue_kb(t0, 2);
        if (n > 1) issue_vb(t0, 1, n);  // its (scale, min) of tile 2 reuses meta row 0: after softmax(0)

        for (int64_t i = 0; i < n && ok; i++) {
            const int cur = (int)(i & 1), nxt = cur ^ 1;
            const bool more = i + 1 < n;
            if (more) ok &= wait_slot(nxt);  // K(i+1)
            ok &= wait_slot(2 + cur);        // V(i): codes of i, (scale, min) of i+1
            if (!ok) break;
            if (kPrep && more) prep_slabs<T::P>(kslot(nxt) + T::OFF_KM);
            const uint16_t *pb = pb0 + cur * 4 * T::PROW;
            if (RP && more) {  // PV of tile i, then the CUDA-core QK of tile i+1 (a rolled loop)
#pragma unroll
                for (int s = 0; s < T::PV_STEPS; s++) pv_step(s, vslot(cur), pb, O);
                qk_rope(kslot(nxt), rpos(i + 1), reinterpret_cast<float (&)[CK::FPI][4]>(accr), z);
            } else if (more) {  // the PV steps spread evenly over the 8 key slabs
#pragma unroll
                for (int sl = 0; sl < 8; sl++) {
                    if (T::PV_STEPS >= 8) {
#pragma unroll
                        for (int r = 0; r < T::PV_STEPS / 8; r++) pv_step(sl * (T::PV_STEPS / 8) + r, vslot(cur), pb, O);
                    } else if (sl % (8 / T::PV_STEPS) == 0) {
                        pv_step(sl / (8 / T::PV_STEPS), vslot(cur), pb, O);
                    }
                    qk_slab(sl, kslot(nxt), acc, cm);
                }
                if (KITTY && p.n_boost > 0) qk_boost(kslot(nxt), acc);
            } else {
#pragma unroll
                for (int s = 0; s < T::PV_STEPS; s++) pv_step(s, vslot(cur), pb, O);
            }
            if (more) {
                float a0, a1;
                bool grow;
                if (RP) softmax_begin_z(z, m, l, mn, a0, a1, grow);
                else softmax_begin(acc, cm, z, m, l, mn, a0, a1, grow);
                if (grow) {  // O holds tiles <= i relative to the previous maximum
#pragma unroll
                    for (int o = 0; o < 8; o++) {
                        O[o][0] *= a0;
                        O[o][2] *= a0;
                        O[o][1] *= a1;
                        O[o][3] *= a1;
                    }
                }
                uint16_t *pbn = pb0 + nxt * 4 * T::PROW;
                uint32_t vm[CK::FPI];
                load_vm(vmslot(nxt), vm);
#pragma unroll
                for (int j = 0; j < CK::NJ; j++) softmax_chunk(j, z, vm, pbn, m, l, mn);
            }
            __syncwarp();
            fence_proxy_async();
            if (i + 3 < n) issue_kb(t0, (int)i + 3);     // key half (i+1)&1 is free
            if (i + 2 < n) issue_vb(t0, (int)i + 2, n);  // value half i&1, meta row (i+1)&1
        }
        if (!ok) {
            // let copies still in flight land before the shared memory is reused
            for (int s = 0; s < kSlots; s++)
                if (pending & (1u << s)) wait_slot(s);
        }
        finish(part, m, l, mn, O);
    }

    // O row set o = set*NJ + j: rows g <-> channel FPI*(g+8 set) + j, g+8 <-> + FPI/2.
    // Writes head rows 0..3 (columns 2t, 2t+1 of lanes t < 2) and m, l.
    __device__ void finish(float *part, float m, float l, float mn, const float (&O)[8][4]) const {
        const int gq = lane >> 2, t = lane & 3;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            mn += __shfl_xor_sync(0xffffffffu, mn, o);
        }
        const float mn0 = __shfl_sync(0xffffffffu, mn, (lane & ~3) | ((2 * t) & 3));
        const float mn1 = __shfl_sync(0xffffffffu, mn, (lane & ~3) | ((2 * t + 1) & 3));
        __syncwarp();
#define KVQ_SO(J)                                                                  \
    if (J < CV::NJ && t < 2) {                                                     \
        const float f = unscale<CV, J>();                                          \
        for (int set = 0; set < T::NSET; set++) {                                  \
            const int o = set * CV::NJ + (J % CV::NJ);                             \
            const int ch = CV::FPI * (gq + 8 * set) + (J % CV::NJ);                \
            const int ch2 = ch + CV::FPI / 2;                                      \
            part[(2 * t) * (T::D + 4) + ch] = fmaf(O[o][0], f, mn0);               \
            part[(2 * t + 1) * (T::D + 4) + ch] = fmaf(O[o][1], f, mn1);           \
            part[(2 * t) * (T::D + 4) + ch2] = fmaf(O[o][2], f, mn0);              \
            part[(2 * t + 1) * (T::D + 4) + ch2] = fmaf(O[o][3], f, mn1);          \
        }                                                                          \
    }
        KVQ_SO(0) KVQ_SO(1) KVQ_SO(2) KVQ_SO(3) KVQ_SO(4) KVQ_SO(5) KVQ_SO(6) KVQ_SO(7)
#undef KVQ_SO
        if (gq == 0) {
            part[t * (T::D + 4) + T::D] = m;
            part[t * (T::D + 4) + T::D + 1] = l;
        }
    }
};

// ---------------------------------------------------------------------------
// Packed tiles on a warp pair.  The query warp streams the key halves and the value
// (scale, min) rows, computes QK and the softmax, and hands each tile's p' and the
// per-head rescale factor to the value warp through shared memory; the value warp
// streams the value codes, rescales O and runs PV.  Handoff per p' buffer b:
// "full" (query -> value) and "empty" (value -> query) mbarriers, waits bounded.
// ---------------------------------------------------------------------------
template <int KB, int VB, bool KITTY, bool PG = false, bool RP = false>
struct PairWarp : FastWarp<KB, VB, KITTY, PG, RP> {
    using Base = FastWarp<KB, VB, KITTY, PG, RP>;
    using T = typename Base::T;
    using CK = typename T::K;
    using CV = typename T::V;
    static constexpr int B_FULL = 4, B_EMPTY = 6, B_QDONE = 8;

    __device__ PairWarp(const DecodeParams &pp, unsigned char *ub) : Base(pp, ub) {}

    __device__ void arrive(int s) {
        __syncwarp();
        if (this->lane == 0) mbar_arrive(&this->bars[s]);
        __syncwarp();
    }
    __device__ float *stats() const { return reinterpret_cast<float *>(this->wbase + this->L.stats); }
    __device__ float *alpha() const { return reinterpret_cast<float *>(this->wbase + this->L.alpha); }
    __device__ uint16_t *pbuf(int b) const {
        return reinterpret_cast<uint16_t *>(this->wbase + this->L.pbuf) + b * 4 * T::PROW;
    }

    // Batch K(j): key codes, key (scale, min), value (scale, min) of tile t0 + j ->
    // key half j&1 and meta row j&1; barrier j&1.
    __device__ void issue_kq(int64_t t0, int j) {
        const DecodeParams &p = this->p;
        const int s = j & 1, lane = this->lane;
        const int64_t ti = t0 + j;
        this->pending |= 1u << s;
        unsigned char *st = this->kslot(s);
        const int nb = KITTY ? p.n_boost : 0;
        const uint32_t bytes = 8 * T::D * 4 + T::D * 4 + (KITTY ? 8 * nb * 4 + T::D : 0) + T::TOK * 4;
        const int64_t pg = this->pid(p, ti >> p.tpp_shift), tin = ti & ((1 << p.tpp_shift) - 1);
        if (lane == 0) {
            mbar_arrive_expect_tx(&this->bars[s], bytes);
            issue_copy(st + T::OFF_K, p.k_codes + ((size_t)pg * (p.G / CK::FPI) + tin * 8) * T::D, 8 * T::D * 4,
                       &this->bars[s]);
            issue_copy(st + T::OFF_KM, p.k_meta + (size_t)pg * T::D * 2, T::D * 4, &this->bars[s]);
            issue_copy(this->vmslot(s), p.v_meta + ((size_t)pg * p.G + tin * T::TOK) * 2, T::TOK * 4,
                       &this->bars[s]);
        }
        if (KITTY) __syncwarp();  // the high-plane rows after lane 0's expect-tx
        if (KITTY && nb > 0 && lane >= 10 && lane < 18) {
            const int r = lane - 10;
            issue_copy(st + T::OFF_HI + r * hi_stride(nb), p.k_hi + ((size_t)pg * (p.G / 16) + tin * 8 + r) * nb,
                       nb * 4, &this->bars[s]);
        } else if (KITTY && lane == 18) {
            issue_copy(st + T::OFF_HI + 8 * hi_stride(nb), p.k_bidx + (size_t)pg * T::D, T::D, &this->bars[s]);
        }
    }

    // Batch V(j): value codes of tile t0 + j -> value half j&1; barrier 2 + j&1.
    __device__ void issue_vp(int64_t t0, int j) {
        const DecodeParams &p = this->p;
        const int s = 2 + (j & 1), lane = this->lane;
        const int64_t ti = t0 + j;
        this->pending |= 1u << s;
        unsigned char *st = this->vslot(j & 1);
        const int64_t pg = this->pid(p, ti >> p.tpp_shift), tin = ti & ((1 << p.tpp_shift) - 1);
        if (lane == 0) {  // the tile's value rows: one block of the tile-major page
            mbar_arrive_expect_tx(&this->bars[s], T::V_ROWS * T::TOK * 4);
            issue_copy(st, p.v_codes + ((size_t)pg * p.G + tin * T::TOK) * T::V_ROWS, T::V_ROWS * T::TOK * 4,
                       &this->bars[s]);
        }
    }

    __device__ void drain(uint32_t mask) {  // copies still in flight land before smem reuse
        for (int s = 0; s < kSlots; s++)
            if ((this->pending & mask) & (1u << s)) this->wait_slot(s);
    }

    // Query warp over tiles [t0, t1) of sequence uu.
    __device__ void run_q(int uu, int64_t t0, int64_t t1) {
        this->u = uu;
        this->pid.set(this->p, uu);
        const int lane = this->lane;
        const int64_t n = t1 - t0;
        const QRegs qr = load_q_regs(this->p, uu);
        issue_kq(t0, 0);
        if (n > 1) issue_kq(t0, 1);
        store_q_warp<T::P>(qr, reinterpret_cast<uint16_t *>(this->wbase + this->L.qraw),
                            reinterpret_cast<uint2 *>(this->wbase + this->L.qpair));
        float m = -INFINITY, l = 0.f, mn = 0.f;
        float acc[CK::NJ][4], cm[4], z[CK::NJ][2];
        bool ok = true;
        for (int64_t j = 0; j < n && ok; j++) {
            const int s = (int)(j & 1);
            ok &= this->wait_slot(s);  // K(j)
            if (!ok) break;
            if (Base::kPrep) prep_slabs<T::P>(this->kslot(s) + T::OFF_KM);
#pragma unroll
            for (int sl = 0; sl < 8; sl++) this->qk_slab(sl, this->kslot(s), acc, cm);
            if (KITTY && this->p.n_boost > 0) this->qk_boost(this->kslot(s), acc);
            float a;
            bool grow;
            this->softmax_begin_a(acc, cm, z, m, l, mn, a, grow);
            if (j >= 2) ok &= this->wait_slot(B_EMPTY + s);  // PV(j-2) is done with buffer s
            if (!ok) break;
            uint16_t *pb = pbuf(s);
            uint32_t vm[CK::FPI];
            this->load_vm(this->vmslot(s), vm);
#pragma unroll
            for (int jj = 0; jj < CK::NJ; jj++) this->softmax_chunk(jj, z, vm, pb, m, l, mn);
            if (lane < 4) alpha()[8 * s + lane] = a;
            arrive(B_FULL + s);
            fence_proxy_async();
            if (j + 2 < n) issue_kq(t0, (int)j + 2);  // key half and meta row s are free
        }
        // the value warp's last two "empty" arrivals (PV(n-2), PV(n-1))
        for (int64_t j = n >= 2 ? n - 2 : 0; j < n; j++) ok &= this->wait_slot(B_EMPTY + (int)(j & 1));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            mn += __shfl_xor_sync(0xffffffffu, mn, o);
        }
        if (lane < 4) {
            stats()[lane] = m;
            stats()[4 + lane] = l;
            stats()[8 + lane] = mn;
        }
        arrive(B_QDONE);
        if (!ok) drain(3u);
    }

    // Value warp over the same tiles; writes the pair's partial [4][D+4] to `part`.
    __device__ void run_p(int uu, int64_t t0, int64_t t1, float *part) {
        this->u = uu;
        this->pid.set(this->p, uu);
        const int lane = this->lane, gq = lane >> 2, t = lane & 3;
        const int64_t n = t1 - t0;
        issue_vp(t0, 0);
        if (n > 1) issue_vp(t0, 1);
        // entries 4..7 of each buffer (columns of no head) read as 1; the query warp
        // writes only entries 0..3
        if (lane < 8) alpha()[8 * (lane >> 2) + 4 + (lane & 3)] = 1.f;
        __syncwarp();
        float O[8][4];
#pragma unroll
        for (int o = 0; o < 8; o++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[o][e] = 0.f;
        bool ok = true;
        for (int64_t j = 0; j < n && ok; j++) {
            const int s = (int)(j & 1);
            ok &= this->wait_slot(2 + s);       // V(j)
            ok &= this->wait_slot(B_FULL + s);  // p'(j), alpha(j)
            if (!ok) break;
            const float a0 = alpha()[8 * s + 2 * t], a1 = alpha()[8 * s + 2 * t + 1];
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int o = 0; o < 8; o++) {
                    O[o][0] *= a0;
                    O[o][2] *= a0;
                    O[o][1] *= a1;
                    O[o][3] *= a1;
                }
            }
            const uint16_t *pb = pbuf(s);
#pragma unroll
            for (int sl = 0; sl < T::PV_STEPS; sl++) this->pv_step(sl, this->vslot(s), pb, O);
            arrive(B_EMPTY + s);
            fence_proxy_async();
            if (j + 2 < n) issue_vp(t0, (int)j + 2);  // value half s is free
        }
        ok &= this->wait_slot(B_QDONE);
        if (!ok) drain(12u);
        const float *st = stats();
        const float mn0 = st[8 + ((2 * t) & 3)], mn1 = st[8 + ((2 * t + 1) & 3)];
#define KVQ_SP(J)                                                                  \
    if (J < CV::NJ && t < 2) {                                                     \
        const float f = Base::template unscale<CV, J>();                           \
        for (int set = 0; set < T::NSET; set++) {                                  \
            const int o = set * CV::NJ + (J % CV::NJ);                             \
            const int ch = CV::FPI * (gq + 8 * set) + (J % CV::NJ);                \
            const int ch2 = ch + CV::FPI / 2;                                      \
            part[(2 * t) * (T::D + 4) + ch] = fmaf(O[o][0], f, mn0);               \
            part[(2 * t + 1) * (T::D + 4) + ch] = fmaf(O[o][1], f, mn1);           \
            part[(2 * t) * (T::D + 4) + ch2] = fmaf(O[o][2], f, mn0);              \
            part[(2 * t + 1) * (T::D + 4) + ch2] = fmaf(O[o][3], f, mn1);          \
        }                                                                          \
    }
        KVQ_SP(0) KVQ_SP(1) KVQ_SP(2) KVQ_SP(3) KVQ_SP(4) KVQ_SP(5) KVQ_SP(6) KVQ_SP(7)
#undef KVQ_SP
        if (gq == 0) {
            part[t * (T::D + 4) + T::D] = st[t];
            part[t * (T::D + 4) + T::D + 1] = st[4 + t];
        }
        __syncwarp();
    }
};

// ---------------------------------------------------------------------------
// NVFP4 tiles (BitDecoding notes, Sec. V-D: Blackwell's mxfp4 / nvfp4 formats): 64
// tokens of e2m1 codes with e4m3 scales per 16 elements along each product's
// contracted dimension and an fp32 scale per page.  The hardware conversion turns a
// code byte -- the two elements one mma register takes, by the page layouts -- into
// an exact f16x2; times its block scale it stays exact (a 2-bit by 4-bit significand).
// The fp16 query is the QK B operand as it is (even columns; odd columns zero) and the
// page scale S_K multiplies the logits; p' = p * S_V is the PV B operand, in natural
// token order.  Symmetric scales: no min terms.
//   QK: ldmatrix row = token, 16 bytes = 32 channels: lane (g, t) gets channels
//       32 grp + 8t .. 8t+7; k pairs (2t, 2t+1 | 2t+8, 2t+9) <- bytes (0 | 1) for the first
//       mma of a group, (2 | 3) for the second, and the query likewise.
//   PV: ldmatrix row = channel, 16 bytes = 32 tokens: lane (g, t) gets tokens
//       32 tg + 8t .. 8t+7, the same k pairing, and p' of those tokens (one 16-byte load).
// ---------------------------------------------------------------------------
template <bool PG = false>
struct F4Warp {
    static constexpr int D = 128, TOK = 64;
    static constexpr int K_CODES = 0, K_SCALES = 4096, K_HDR = 4608, V_HDR = 4624, K_STAGE = 4736;
    static constexpr int V_CODES = 0, V_SCALES = 4096, V_STAGE = 4608;
    static constexpr int PROW = TOK + 8;  // p' row (halves), padded
    static_assert(2 * K_STAGE + 2 * V_STAGE <= kF4Region, "the stages fit the 4-bit tile region");
    const DecodeParams &p;
    unsigned char *wbase;
    WarpSmem L;  // the 4-bit tile layout: its tile region holds the stages below (kF4Region)
    int u, lane;
    uint64_t *bars;
    uint32_t phase = 0, pending = 0;
    uint32_t qb[16];  // query B registers: group grp, mma m, register r at [4 grp + 2 m + r]

    __device__ F4Warp(const DecodeParams &pp, unsigned char *wb)
        : p(pp), wbase(wb), L(4, 4, false, 0), u(0), lane(threadIdx.x & 31) {
        bars = reinterpret_cast<uint64_t *>(wbase + L.bars);
    }
    __device__ unsigned char *kslot(int s) const { return wbase + L.k0 + s * K_STAGE; }
    __device__ unsigned char *vslot(int s) const { return wbase + 2 * K_STAGE + s * V_STAGE; }
    __device__ bool wait_slot(int s) {
        const bool ok = mbar_wait(&bars[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        pending &= ~(1u << s);
        return ok;
    }
    // page record and codes of the page holding tile ti
    __device__ const uint8_t *krec(int64_t pg) const {
        return reinterpret_cast<const uint8_t *>(p.k_meta) + ((size_t)u * (p.max_T / p.G) + pg) * p.nv_kms;
    }
    __device__ const uint8_t *vrec(int64_t pg) const {
        return reinterpret_cast<const uint8_t *>(p.v_meta) + ((size_t)u * (p.max_T / p.G) + pg) * p.nv_vms;
    }
    __device__ const uint8_t *kcodes(int64_t pg) const {
        return reinterpret_cast<const uint8_t *>(p.k_codes) + ((size_t)u * (p.max_T / p.G) + pg) * ((size_t)p.G * D / 2);
    }
    __device__ const uint8_t *vcodes(int64_t pg) const {
        return reinterpret_cast<const uint8_t *>(p.v_codes) + ((size_t)u * (p.max_T / p.G) + pg) * ((size_t)p.G * D / 2);
    }

    // Batch K(j): key codes (4 groups x 1 KB), key scales, both page headers -> key stage
    // j & 1, barrier j & 1.  Batch V(j): value codes (4 KB), value scales -> value stage,
    // barrier 2 + (j & 1).
    __device__ void issue_k(int64_t t0, int j) {
        const int s = j & 1;
        const int64_t ti = t0 + j, pg = ti >> p.tpp_shift;
        const int tok0 = (int)(ti & ((1 << p.tpp_shift) - 1)) * TOK;
        pending |= 1u << s;
        unsigned char *st = kslot(s);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], 4096 + 512 + 16 + 16);
        __syncwarp();
        if (lane < 4) {
            issue_copy(st + K_CODES + 1024 * lane, kcodes(pg) + ((size_t)lane * p.G + tok0) * 16, 1024, &bars[s]);
        } else if (lane == 4) {
            issue_copy(st + K_SCALES, krec(pg) + 16 + (size_t)tok0 * (D / 16), 512, &bars[s]);
        } else if (lane == 5) {
            issue_copy(st + K_HDR, krec(pg), 16, &bars[s]);
        } else if (lane == 6) {
            issue_copy(st + V_HDR, vrec(pg), 16, &bars[s]);
        }
    }
    __device__ void issue_v(int64_t t0, int j) {
        const int s = 2 + (j & 1);
        const int64_t ti = t0 + j, pg = ti >> p.tpp_shift;
        const int tok0 = (int)(ti & ((1 << p.tpp_shift) - 1)) * TOK;
        pending |= 1u << s;
        unsigned char *st = vslot(j & 1);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], 4096 + 512);
        __syncwarp();
        if (lane == 0) {
            issue_copy(st + V_CODES, vcodes(pg) + (size_t)(tok0 / 32) * D * 16, 4096, &bars[s]);
        } else if (lane == 1) {
            issue_copy(st + V_SCALES, vrec(pg) + 16 + (size_t)(tok0 / 16) * D, 512, &bars[s]);
        }
    }

    // f16x2 (s, s) of the e4m3 scale byte `sc`
    __device__ __forceinline__ static uint32_t scale2(uint32_t sc) {
        const uint32_t h = e4m3x2_to_f16x2(sc & 0xFFu);
        return prmt(h, h, 0x1010);
    }
    __device__ __forceinline__ static uint32_t deq(uint32_t w, int byte, uint32_t s2) {
        return hmul2(e2m1x2_to_f16x2((w >> (8 * byte)) & 0xFFu), s2);
    }

    // Query B registers (once per run): the fp16 query of head g >> 1 in even columns.
    __device__ void load_qb() {
        const int gq = lane >> 2, t = lane & 3;
        const uint16_t *qraw = reinterpret_cast<const uint16_t *>(wbase + L.qraw);
#pragma unroll
        for (int grp = 0; grp < 4; grp++)
#pragma unroll
            for (int m = 0; m < 2; m++)
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const int ch = 32 * grp + 8 * t + 4 * m + 2 * r;
                    qb[4 * grp + 2 * m + r] =
                        (gq & 1) ? 0u : *reinterpret_cast<const uint32_t *>(qraw + (gq >> 1) * 128 + ch);
                }
    }

    // QK of the key stage st: acc[rs] for tokens 16 rs + g (c0, c1), 16 rs + 8 + g (c2, c3)
    __device__ __forceinline__ void qk(const unsigned char *st, float (&acc)[4][4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const uint32_t cb = smem_u32(st + K_CODES);
#pragma unroll
        for (int rs = 0; rs < 4; rs++) {
            const int tk0 = 16 * rs + gq, tk1 = tk0 + 8;
            const uint2 sw0 = *reinterpret_cast<const uint2 *>(st + K_SCALES + tk0 * 8);
            const uint2 sw1 = *reinterpret_cast<const uint2 *>(st + K_SCALES + tk1 * 8);
#pragma unroll
            for (int gp = 0; gp < 2; gp++) {  // groups 2 gp, 2 gp + 1
                uint32_t w[4];
                const int L8 = lane & 7, m8 = (lane >> 3) & 1, g2 = (lane >> 4) & 1;
                ldmatrix_x4(w, cb + (2 * gp + g2) * 1024 + (16 * rs + 8 * m8 + L8) * 16);
#pragma unroll
                for (int gg = 0; gg < 2; gg++) {
                    const int grp = 2 * gp + gg, blk = 2 * grp + (t >> 1);  // this lane's 16-channel block
                    const uint32_t s0 = scale2((blk < 4 ? sw0.x : sw0.y) >> (8 * (blk & 3)));
                    const uint32_t s1 = scale2((blk < 4 ? sw1.x : sw1.y) >> (8 * (blk & 3)));
                    const uint32_t wa = w[2 * gg], wb = w[2 * gg + 1];  // rows g, g+8
#pragma unroll
                    for (int m = 0; m < 2; m++)
                        mma_16816(acc[rs], deq(wa, 2 * m, s0), deq(wb, 2 * m, s1), deq(wa, 2 * m + 1, s0),
                                  deq(wb, 2 * m + 1, s1), qb[4 * grp + 2 * m], qb[4 * grp + 2 * m + 1]);
                }
            }
        }
    }

    // PV of the value stage st with p' buffer pb: O[cs] rows = channels 16 cs + g, + 8
    __device__ __forceinline__ void pv(const unsigned char *st, const uint16_t *pb, float (&O)[8][4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const uint32_t cb = smem_u32(st + V_CODES);
        uint4 bp[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (gq < 4) {
#pragma unroll
            for (int tg = 0; tg < 2; tg++)
                bp[tg] = *reinterpret_cast<const uint4 *>(pb + gq * PROW + 32 * tg + 8 * t);
        }
#pragma unroll
        for (int cs = 0; cs < 8; cs++) {
            uint32_t w[4];
            const int L8 = lane & 7, m8 = (lane >> 3) & 1, g2 = (lane >> 4) & 1;
            ldmatrix_x4(w, cb + g2 * 2048 + (16 * cs + 8 * m8 + L8) * 16);
            const int c0 = 16 * cs + gq, c1 = c0 + 8;
#pragma unroll
            for (int tg = 0; tg < 2; tg++) {
                const int tb = 2 * tg + (t >> 1);  // this lane's 16-token block
                const uint32_t s0 = scale2(st[V_SCALES + tb * D + c0]), s1 = scale2(st[V_SCALES + tb * D + c1]);
                const uint32_t wa = w[2 * tg], wb = w[2 * tg + 1];
                mma_16816(O[cs], deq(wa, 0, s0), deq(wb, 0, s1), deq(wa, 1, s0), deq(wb, 1, s1), bp[tg].x, bp[tg].y);
                mma_16816(O[cs], deq(wa, 2, s0), deq(wb, 2, s1), deq(wa, 3, s0), deq(wb, 3, s1), bp[tg].z, bp[tg].w);
            }
        }
    }

    // Softmax of a tile: logits from acc (times S_K), running maximum, then p' = p S_V
    // into pb (natural token order, heads 0..3 = rows).
    __device__ __forceinline__ void softmax(const float (&acc)[4][4], const unsigned char *ks, uint16_t *pb,
                                            float &m, float &l, float &a0, float &a1, bool &grow) const {
        const int gq = lane >> 2, t = lane & 3;
        const float SK = *reinterpret_cast<const float *>(ks + K_HDR), SV = *reinterpret_cast<const float *>(ks + V_HDR);
        const float C = kLog2e * rsqrtf((float)D) * SK;
        float z[4][2], tm = -INFINITY;
#pragma unroll
        for (int rs = 0; rs < 4; rs++) {
            z[rs][0] = (acc[rs][0] + acc[rs][1]) * C;
            z[rs][1] = (acc[rs][2] + acc[rs][3]) * C;
            tm = fmaxf(tm, fmaxf(z[rs][0], z[rs][1]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
        const float nm = fmaxf(m, tm);
        const float a = ex2(m - nm);
        grow = __any_sync(0xffffffffu, nm > m);
        m = nm;
        l *= a;
        a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
        a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
        uint16_t *row = pb + t * PROW;
#pragma unroll
        for (int rs = 0; rs < 4; rs++) {
            const float p0 = ex2(z[rs][0] - m), p1 = ex2(z[rs][1] - m);
            l += p0 + p1;
            row[16 * rs + gq] = __half_as_ushort(__float2half_rn(p0 * SV));
            row[16 * rs + 8 + gq] = __half_as_ushort(__float2half_rn(p1 * SV));
        }
    }

    // Tiles [t0, t1) of sequence uu; the warp's partial [4][D+4] to `part`.  Pipeline as
    // the packed-code tiles: PV of tile i with QK of tile i+1, copies two tiles ahead.
    __device__ void run(int uu, int64_t t0, int64_t t1, float *part) {
        u = uu;
        const int64_t n = t1 - t0;
        const QRegs qr = load_q_regs(p, u);
        issue_k(t0, 0);
        issue_v(t0, 0);
        if (n > 1) issue_k(t0, 1);
        store_q_warp<4>(qr, reinterpret_cast<uint16_t *>(wbase + L.qraw), reinterpret_cast<uint2 *>(wbase + L.qpair));
        load_qb();
        uint16_t *pb0 = reinterpret_cast<uint16_t *>(wbase + L.pbuf);
        for (int i = lane; i < 4 * PROW; i += 32) reinterpret_cast<uint32_t *>(pb0)[i] = 0u;
        __syncwarp();
        float m = -INFINITY, l = 0.f, O[8][4], acc[4][4];
#pragma unroll
        for (int o = 0; o < 8; o++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[o][e] = 0.f;
        bool ok = wait_slot(0);
        if (ok) {
#pragma unroll
            for (int rs = 0; rs < 4; rs++)
#pragma unroll
                for (int e = 0; e < 4; e++) acc[rs][e] = 0.f;
            qk(kslot(0), acc);
            float a0, a1;
            bool grow;
            softmax(acc, kslot(0), pb0, m, l, a0, a1, grow);
        }
        __syncwarp();
        fence_proxy_async();
        if (n > 2) issue_k(t0, 2);
        if (n > 1) issue_v(t0, 1);
        for (int64_t i = 0; i < n && ok; i++) {
            const int cur = (int)(i & 1), nxt = cur ^ 1;
            const bool more = i + 1 < n;
            if (more) ok &= wait_slot(nxt);  // K(i+1)
            ok &= wait_slot(2 + cur);        // V(i)
            if (!ok) break;
            const uint16_t *pb = pb0 + cur * 4 * PROW;
            pv(vslot(cur), pb, O);
            if (more) {
#pragma unroll
                for (int rs = 0; rs < 4; rs++)
#pragma unroll
                    for (int e = 0; e < 4; e++) acc[rs][e] = 0.f;
                qk(kslot(nxt), acc);
                float a0, a1;
                bool grow;
                softmax(acc, kslot(nxt), pb0 + nxt * 4 * PROW, m, l, a0, a1, grow);
                if (grow) {
#pragma unroll
                    for (int o = 0; o < 8; o++) {
                        O[o][0] *= a0;
                        O[o][2] *= a0;
                        O[o][1] *= a1;
                        O[o][3] *= a1;
                    }
                }
            }
            __syncwarp();
            fence_proxy_async();
            if (i + 3 < n) issue_k(t0, (int)i + 3);
            if (i + 2 < n) issue_v(t0, (int)i + 2);
        }
        if (!ok) {
            for (int s = 0; s < kSlots; s++)
                if (pending & (1u << s)) wait_slot(s);
        }
        // partial: heads 0..3 (lanes t < 2 hold heads 2t, 2t+1 of channels g, g+8 per set)
        const int gq = lane >> 2, t = lane & 3;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        __syncwarp();
        if (t < 2) {
#pragma unroll
            for (int cs = 0; cs < 8; cs++) {
                const int ch = 16 * cs + gq;
                part[(2 * t) * (D + 4) + ch] = O[cs][0];
                part[(2 * t + 1) * (D + 4) + ch] = O[cs][1];
                part[(2 * t) * (D + 4) + ch + 8] = O[cs][2];
                part[(2 * t + 1) * (D + 4) + ch + 8] = O[cs][3];
            }
        }
        if (gq == 0) {
            part[t * (D + 4) + D] = m;
            part[t * (D + 4) + D + 1] = l;
        }
    }
};

// ---------------------------------------------------------------------------
// Mini tiles: 16 tokens with fp16 values
// ---------------------------------------------------------------------------
// Mini tile mi of a sequence: [sink tiles][packed-key blocks][fp16-buffer tiles].
struct MiniTile {
    int64_t tok0;   // first logical token
    int n;          // valid tokens (1..16)
    bool kpacked;   // keys from a packed 16-token block (Kitty), else fp16 rows
};

__device__ __forceinline__ MiniTile mini_tile(const DecodeParams &p, const SeqLen &sq, int64_t mi) {
    MiniTile m;
    const int64_t ms = (sq.n_sink + 15) >> 4, tok_fast = sq.n_fast * (256 / p.bits);
    const int64_t mp = (sq.T_k - tok_fast) >> 4;
    if (mi < ms) {
        m.tok0 = 16 * mi;
        m.n = (int)kvq_min64(16, sq.n_sink - m.tok0);
        m.kpacked = false;
    } else if (mi < ms + mp) {
        m.tok0 = sq.n_sink + tok_fast + 16 * (mi - ms);
        m.n = 16;
        m.kpacked = true;
    } else {
        m.tok0 = sq.n_sink + sq.T_k + 16 * (mi - ms - mp);
        m.n = (int)kvq_min64(16, sq.L - m.tok0);
        m.kpacked = false;
    }
    return m;
}

// fp16 value row of logical token tl (tl outside the packed values).
__device__ __forceinline__ const uint16_t *vrow16(const DecodeParams &p, const SeqLen &sq, int u, int64_t tl) {
    if (tl < sq.n_sink) return p.v_sink + ((size_t)u * p.S_cap + tl) * 128;
    const int64_t r = tl - sq.n_sink - sq.T_v;
    if (r < sq.n_vres) return p.v_res + ((size_t)u * p.cap_v + r) * 128;
    int64_t slot = sq.local_head + (r - sq.n_vres);  // < 2 R: local_head < R, r - n_vres < n_local <= R
    if (slot >= p.R_local) slot -= p.R_local;
    return p.v_local + ((size_t)u * p.R_local + slot) * 128;
}
__device__ __forceinline__ const uint16_t *krow16(const DecodeParams &p, const SeqLen &sq, int u, int64_t tl) {
    if (tl < sq.n_sink) return p.k_sink + ((size_t)u * p.S_cap + tl) * 128;
    return p.k_res + ((size_t)u * p.cap_k + (tl - sq.n_sink - sq.T_k)) * 128;
}

template <int KB, int VB, bool KITTY, bool PG = false, bool RP = false>
struct MiniWarp {
    const DecodeParams &p;
    unsigned char *wbase;
    WarpSmem L;  // the CTA's per-warp layout (slots are large enough for a mini tile)
    int u, lane;
    uint64_t *bars;
    uint32_t phase = 0, pending = 0;
    SeqLen sq;  // lengths of sequence u
    const float *rt = nullptr;  // RP: the RoPE tables

    // packed-key block layout in the key half of a slot
    static constexpr int MB_W = 0, MB_M = 512, MB_HI = 1024;

    __device__ MiniWarp(const DecodeParams &pp, unsigned char *wb, int slot_bits)
        : p(pp), wbase(wb), L(KB, VB, KITTY, pp.n_boost), u(0), lane(threadIdx.x & 31) {
        (void)slot_bits;
        bars = reinterpret_cast<uint64_t *>(wbase + L.bars);
    }
    __device__ unsigned char *slot(int s) const { return wbase + s * L.mslot; }
    __device__ void init_bars() {
        if (lane == 0) {
            for (int s = 0; s < kSlots; s++) mbar_init(&bars[s], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }
    __device__ bool wait_slot(int s) {
        const bool ok = mbar_wait(&bars[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        pending &= ~(1u << s);
        return ok;
    }

    // K half -> slot sk, V half -> slot sk+1.  Rows past the valid count repeat row 0.
    __device__ void issue(const MiniTile &mt, int sk) {
        pending |= 3u << sk;
        const int nb = KITTY ? p.n_boost : 0;
        const uint32_t kbytes = mt.kpacked ? 512 + 512 + 4 * nb + 128 : 16 * 256;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[sk], kbytes);
            mbar_arrive_expect_tx(&bars[sk + 1], 16 * 256);
        }
        __syncwarp();
        unsigned char *sK = slot(sk), *sV = slot(sk + 1);
        const int i = lane & 15;
        const int64_t tl = mt.tok0 + (i < mt.n ? i : 0);
        // appended in this launch: the last token's rows come from k_new / v_new (plain
        // loads, so they may be host memory the device can map), and this warp -- the
        // only one holding the sequence's last tile -- stores them into the residuals, 16
        // bytes per lane; its bulk copies below then read them from there
        if (p.k_new && mt.tok0 + mt.n == sq.L) {
            const uint4 *src = reinterpret_cast<const uint4 *>((lane < 16 ? p.k_new : p.v_new) + (size_t)u * 128);
            uint16_t *dst = lane < 16 ? const_cast<uint16_t *>(krow16(p, sq, u, sq.L - 1))
                                      : const_cast<uint16_t *>(vrow16(p, sq, u, sq.L - 1));
            reinterpret_cast<uint4 *>(dst)[i] = __ldg(src + i);
            __syncwarp();
            fence_proxy_async_global();
        }
        if (lane < 16) {
            if (!mt.kpacked) {
                issue_copy(sK + i * kMiniRow, krow16(p, sq, u, tl), 256, &bars[sk]);
            } else {  // Kitty mixed blocks (dense caches only)
                const int64_t tk = mt.tok0 - sq.n_sink, page = tk >> p.g_shift, blk = tk >> 4;
                if (i == 0) {
                    issue_copy(sK + MB_W, p.k_codes + ((size_t)u * (p.max_T / 16) + blk) * 128, 512, &bars[sk]);
                } else if (i == 1) {
                    issue_copy(sK + MB_M, p.k_meta + ((size_t)u * (p.max_T / p.G) + page) * 256, 512, &bars[sk]);
                } else if (i == 2 && nb > 0) {
                    issue_copy(sK + MB_HI, p.k_hi + ((size_t)u * (p.max_T / 16) + blk) * nb, 4 * nb, &bars[sk]);
                } else if (i == 3 && KITTY) {
                    issue_copy(sK + MB_HI + ((4 * nb + 15) & ~15),
                               p.k_bidx + ((size_t)u * (p.max_T / p.G) + page) * 128, 128, &bars[sk]);
                }
            }
        } else {
            issue_copy(sV + i * kMiniRow, vrow16(p, sq, u, tl), 256, &bars[sk + 1]);
        }
    }

    __device__ void run(int uu, int64_t m0, int64_t m1, float *part) {
        u = uu;
        sq = seq_len<PG>(p, uu);
        const int gq = lane >> 2, t = lane & 3, hq = gq >> 1;
        const bool lo_col = (gq & 1) != 0;
        const int64_t n = m1 - m0;
        uint16_t *qraw = reinterpret_cast<uint16_t *>(wbase + L.qraw);
        const QRegs qr = load_q_regs(p, u);
        issue(mini_tile(p, sq, u_base(m0)), 0);
        if (n > 1) issue(mini_tile(p, sq, u_base(m0 + 1)), 2);
        store_q_warp<8>(qr, qraw, reinterpret_cast<uint2 *>(wbase + L.qpair));
        uint16_t *pb = reinterpret_cast<uint16_t *>(wbase + L.pbuf);  // [4][16] p
        for (int i = lane; i < 8 * 16; i += 32) pb[i] = 0;           // heads 4..7 stay zero
        __syncwarp();
        float m = -INFINITY, l = 0.f;
        float O[8][4];
#pragma unroll
        for (int o = 0; o < 8; o++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[o][e] = 0.f;
        const float C = kLog2e * rsqrtf(128.f) / kQScale;
        bool ok = true;
        for (int64_t i = 0; i < n && ok; i++) {
            const int sk = 2 * (int)(i & 1);
            const MiniTile mt = mini_tile(p, sq, u_base(m0 + i));
            ok &= wait_slot(sk);
            ok &= wait_slot(sk + 1);
            if (!ok) break;
            const unsigned char *sK = slot(sk), *sV = slot(sk + 1);
            float s[4] = {0.f, 0.f, 0.f, 0.f}, cm[4] = {0.f, 0.f, 0.f, 0.f};
            float unsc = 1.0f;
            if (!mt.kpacked) {
                const uint32_t kb = smem_u32(sK) + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kMiniRow + 16 * (lane >> 4);
#pragma unroll
                for (int sl = 0; sl < 8; sl++) {
                    uint32_t a[4];
                    ldmatrix_x4(a, kb + 32 * sl);
                    uint32_t b0 = 0u, b1 = 0u;
                    if (!lo_col) {
                        b0 = hmul2(*reinterpret_cast<const uint32_t *>(qraw + hq * 128 + 16 * sl + 2 * t), 0x2C002C00u);
                        b1 = hmul2(*reinterpret_cast<const uint32_t *>(qraw + hq * 128 + 16 * sl + 8 + 2 * t),
                                   0x2C002C00u);
                    }
                    if (RP) {
                        // register r: channel pair 8 sl + t (+4 for r >= 2) of token tok0 + g
                        // (+8 for odd r), turned by its position in fp32, then split into
                        // fp16 hi + lo (two mmas, 22 significant bits)
                        uint32_t ah[4], al[4];
#pragma unroll
                        for (int r = 0; r < 4; r++) {
                            const int pr = 8 * sl + t + 4 * (r >> 1);
                            const float pos = (float)(mt.tok0 + gq + 8 * (r & 1));
                            const float2 cs = rope_cs(pos, rt[kRopeHi + pr], rt[kRopeLo + pr]);
                            const float2 kv = unpack_half2(a[r]);
                            const float rx = fmaf(kv.x, cs.x, -kv.y * cs.y), ry = fmaf(kv.x, cs.y, kv.y * cs.x);
                            ah[r] = pack_half2(rx, ry);
                            const float2 hv = unpack_half2(ah[r]);
                            al[r] = pack_half2(rx - hv.x, ry - hv.y);
                        }
                        mma_16816(s, ah[0], ah[1], ah[2], ah[3], b0, b1);
                        mma_16816(s, al[0], al[1], al[2], al[3], b0, b1);
                    } else {
                        mma_16816(s, a[0], a[1], a[2], a[3], b0, b1);
                    }
                }
            } else {
                // Kitty mixed block: 16 tokens of packed keys, rows g / g+8 <-> tokens g / g+8
                const uint32_t *w = reinterpret_cast<const uint32_t *>(sK + MB_W);
                const uint32_t *km = reinterpret_cast<const uint32_t *>(sK + MB_M);
                // the block is word row (tok0 - n_sink) / 16 of the cache, row rb of its
                // 8-row group: logical chunk c of the row is stored at chunk c ^ rb
                const int rb = (int)(((mt.tok0 - sq.n_sink) >> 4) & 7);
                const uint2 *qpair = reinterpret_cast<const uint2 *>(wbase + L.qpair);
#pragma unroll
                for (int sl = 0; sl < 8; sl++) {
                    const SlabB b = slab_b(qpair[(hq * 8 + sl) * 4 + t], km[chan_of<8>(sl, t, 0)],
                                           km[chan_of<8>(sl, t, 1)], km[chan_of<8>(sl, t, 2)],
                                           km[chan_of<8>(sl, t, 3)], col_const(lo_col));
                    mma_16816(cm, b.am0, b.am0, b.am1, b.am1, b.c0, b.c1);
                    uint32_t wv[4], x[4], xs[4];
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) wv[kk] = w[4 * ((4 * sl + kk) ^ rb) + t];
                    FastWarp<2, 2, KITTY, false, false>::template split<Codes<2>>(wv, x, xs);
                    uint32_t a[4];
#pragma unroll
                    for (int r = 0; r < 4; r++) a[r] = (x[r] >> (2 * gq)) & 0x00030003u;
                    mma_16816(s, a[0], a[1], a[2], a[3], b.b0, b.b1);
                }
                if (KITTY && p.n_boost > 0) {
                    const int nb = p.n_boost;
                    const uint32_t *hw = reinterpret_cast<const uint32_t *>(sK + MB_HI);
                    const uint8_t *bi = sK + MB_HI + ((4 * nb + 15) & ~15);
                    uint8_t *invb = wbase + L.invb;
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const int ch = lane * 4 + r;
                        const int sl = bi[ch];
                        if (sl < nb) invb[sl] = (uint8_t)ch;
                    }
                    __syncwarp();
                    for (int s2 = 0; s2 < nb / 16; s2++) {
                        uint32_t km4[4];
                        uint16_t qv[4];
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) {
                            const int ch = invb[chan_of<8>(s2, t, kk)] & 127;
                            km4[kk] = km[ch];
                            qv[kk] = qraw[hq * 128 + ch];
                        }
                        uint32_t q0 = hmul2((uint32_t)qv[0] | ((uint32_t)qv[1] << 16), 0x2C002C00u);
                        uint32_t q1 = hmul2((uint32_t)qv[2] | ((uint32_t)qv[3] << 16), 0x2C002C00u);
                        q0 = hmul2(q0, 0x44004400u);
                        q1 = hmul2(q1, 0x44004400u);
                        const SlabB b = slab_b(make_uint2(q0, q1), km4[0], km4[1], km4[2], km4[3], col_const(lo_col));
                        uint32_t wv[4], x[4], xs[4];
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) wv[kk] = hw[16 * s2 + 4 * kk + t];
                        FastWarp<2, 2, KITTY, false, false>::template split<Codes<2>>(wv, x, xs);
                        uint32_t a[4];
#pragma unroll
                        for (int r = 0; r < 4; r++) a[r] = (x[r] >> (2 * gq)) & 0x00030003u;
                        mma_16816(s, a[0], a[1], a[2], a[3], b.b0, b.b1);
                    }
                    __syncwarp();
                }
                unsc = 16777216.0f;  // codes sit at bit offset 0: c * 2^-24
            }
            // softmax over the 16 tokens (lane: head t, tokens gq and gq+8)
            const float cst = cm[0] * C;
            float z0 = fmaf(s[0] - s[1], unsc * C, cst), z1 = fmaf(s[2] - s[3], unsc * C, cst);
            if (gq >= mt.n) z0 = -INFINITY;
            if (gq + 8 >= mt.n) z1 = -INFINITY;
            float tm = fmaxf(z0, z1);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
            const float nm = fmaxf(m, tm);
            const float a = ex2(m - nm);
            m = nm;
            l *= a;
            const float a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
            const float a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
#pragma unroll
            for (int o = 0; o < 8; o++) {
                O[o][0] *= a0;
                O[o][2] *= a0;
                O[o][1] *= a1;
                O[o][3] *= a1;
            }
            const float p0 = ex2(z0 - m), p1 = ex2(z1 - m);
            l += p0 + p1;
            pb[t * 16 + gq] = __half_as_ushort(__float2half_rn(p0));
            pb[t * 16 + gq + 8] = __half_as_ushort(__float2half_rn(p1));
            __syncwarp();
            // O[ch][head] += V^T . P   (ldmatrix.trans of the fp16 value rows)
            uint32_t b0 = 0u, b1 = 0u;
            if (gq < 4) {
                b0 = *reinterpret_cast<const uint32_t *>(pb + gq * 16 + 2 * t);
                b1 = *reinterpret_cast<const uint32_t *>(pb + gq * 16 + 8 + 2 * t);
            }
            const uint32_t vb = smem_u32(sV) + ((lane & 7) + 8 * (lane >> 4)) * kMiniRow + 16 * ((lane >> 3) & 1);
#pragma unroll
            for (int o = 0; o < 8; o++) {
                uint32_t av[4];
                ldmatrix_x4_trans(av, vb + 32 * o);
                mma_16816(O[o], av[0], av[1], av[2], av[3], b0, b1);
            }
            __syncwarp();
            fence_proxy_async();
            if (i + 2 < n) issue(mini_tile(p, sq, u_base(m0 + i + 2)), sk);
        }
        if (!ok) {
            for (int s = 0; s < kSlots; s++)
                if (pending & (1u << s)) wait_slot(s);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        __syncwarp();
        if (t < 2) {  // head rows 0..3
#pragma unroll
            for (int o = 0; o < 8; o++) {
                const int ch = 16 * o + gq;
                part[(2 * t) * 132 + ch] = O[o][0];
                part[(2 * t + 1) * 132 + ch] = O[o][1];
                part[(2 * t) * 132 + ch + 8] = O[o][2];
                part[(2 * t + 1) * 132 + ch + 8] = O[o][3];
            }
        }
        if (gq == 0) {
            part[t * 132 + 128] = m;
            part[t * 132 + 129] = l;
        }
    }

    // mini index within the sequence (the caller passes per-sequence indices)
    __device__ __forceinline__ static int64_t u_base(int64_t mi) { return mi; }
};

}  // namespace kvq
