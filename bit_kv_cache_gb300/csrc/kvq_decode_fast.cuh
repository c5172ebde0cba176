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
constexpr int kSlots = 4;           // per-warp ring: K(i), V(i), K(i+1), V(i+1)

__host__ __device__ inline int hi_stride(int nb) { return nb * 4 + 16; }
// A warp / CTA partial: 8 head rows of prow(D) floats: o[0..D), m at D, l at D+1
// (rows padded to 16 bytes for vector access).
__host__ __device__ inline int prow(int D) { return D + 4; }
__host__ __device__ inline int part_bytes(int D) { return 8 * prow(D) * 4; }

template <int BITS>
struct Tile {
    static constexpr int D = 128;
    static constexpr int FPI = 32 / BITS;
    static constexpr int TOK = BITS == 2 ? 128 : 64;   // tokens per packed tile (8 key word rows)
    static constexpr int K_STRIDE = D * 4 + 16;        // padded key row: conflict-free ldmatrix
    static constexpr int V_ROWS = D / FPI;             // value channel blocks: 8 or 16
    static constexpr int V_STRIDE = TOK * 4 + 16;
    static constexpr int NJ = FPI / 2;                 // mma row sets per word: 8 or 4
    static constexpr int NSET = V_ROWS / 8;            // 1 or 2
    static constexpr int TSLABS = TOK / 16;            // 16-token slabs for PV
    static constexpr int JDIRECT = BITS == 2 ? 5 : 2;  // row sets readable without a pre-shift
    static constexpr int SH = BITS == 2 ? 6 : 8;       // pre-shift for the others
    static constexpr uint32_t MASK0 = BITS == 2 ? 0x00030003u : 0x000F000Fu;
    static constexpr int PS = BITS == 2 ? 8 : 4;       // k = 2t+1 pairs token/channel t with t + PS
    // key half-stage
    static constexpr int OFF_K = 0;
    static constexpr int OFF_KM = 8 * K_STRIDE;        // (scale, min) per channel, 512 B
    static constexpr int OFF_HI = OFF_KM + D * 4;      // Kitty: 8 rows of hi_stride(nb), then D bytes of index
    // value half-stage
    static constexpr int OFF_V = 0;
    static constexpr int OFF_VM = V_ROWS * V_STRIDE;   // (scale, min) per token
    static constexpr int V_HALF = OFF_VM + TOK * 4;
    static constexpr int PROW = TOK + 8;               // p' row (halves), padded
    static constexpr int PBUF = 4 * PROW * 2;          // one p' buffer: heads 0..3
};

constexpr int kMiniRow = 128 * 2 + 16;                 // padded fp16 row of the mini tiles
constexpr int kMiniHalf = 16 * kMiniRow;               // 16 fp16 rows

template <int BITS>
__host__ __device__ inline int slot_bytes(bool kitty, int nb) {
    using T = Tile<BITS>;
    int k = T::OFF_HI + (kitty ? 8 * hi_stride(nb) + T::D : 0);
    int s = k > T::V_HALF ? k : T::V_HALF;
    s = s > kMiniHalf ? s : kMiniHalf;
    return (s + 127) & ~127;
}

// Per-warp shared memory (fast and mini warps):
//   [kSlots slots][p' buffer x2][q fp16 [4][128]][q' pairs [4 heads][8 slabs][4 lanes] x 8 B]
//   [slot index 64 B][mbarriers kSlots x 8 B][first-segment partial [4][D+4] fp32]
template <int BITS>
struct WarpSmem {
    int slot, pbuf, qraw, qpair, invb, bars, part0, total;
    __host__ __device__ WarpSmem(bool kitty, int nb) {
        slot = slot_bytes<BITS>(kitty, nb);
        pbuf = kSlots * slot;
        qraw = pbuf + 2 * Tile<BITS>::PBUF;
        qpair = qraw + 4 * 128 * 2;
        invb = qpair + 4 * 8 * 4 * 8;
        bars = invb + 64;
        part0 = (bars + 8 * kSlots + 15) & ~15;     // partial of a first segment: 4 head rows
        total = (part0 + 4 * prow(128) * 4 + 127) & ~127;
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

// B operands of one 16-channel slab from the page's (scale, min) words kmA..kmD of
// channels chan_of(sl, t, 0..3): the folded query (hi or lo part by column parity)
// and q * 2^-4 for the min mma (zero in lo columns); A operand of the min mma.
struct SlabB {
    uint32_t b0, b1, c0, c1, am0, am1;
};
__device__ __forceinline__ SlabB slab_b(uint2 qp, uint32_t kmA, uint32_t kmB, uint32_t kmC, uint32_t kmD,
                                        bool lo_col) {
    SlabB r;
    const uint32_t s01 = prmt(kmA, kmB, 0x5410), s23 = prmt(kmC, kmD, 0x5410);
    const uint32_t hi01 = hmul2(qp.x, s01), hi23 = hmul2(qp.y, s23);
    if (lo_col) {
        r.b0 = hfma2(qp.x, s01, hi01 ^ 0x80008000u);
        r.b1 = hfma2(qp.y, s23, hi23 ^ 0x80008000u);
        r.c0 = r.c1 = 0u;
    } else {
        r.b0 = hi01;
        r.b1 = hi23;
        r.c0 = qp.x;
        r.c1 = qp.y;
    }
    r.am0 = prmt(kmA, kmB, 0x7632);  // (min A, min B)
    r.am1 = prmt(kmC, kmD, 0x7632);  // (min C, min D)
    return r;
}

__device__ __forceinline__ void issue_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    bulk_g2s(dst, src, bytes, bar);
}

// ---------------------------------------------------------------------------
// Packed tiles
// ---------------------------------------------------------------------------
template <int BITS, bool KITTY>
struct FastWarp {
    using T = Tile<BITS>;
    const DecodeParams &p;
    unsigned char *wbase;
    WarpSmem<BITS> L;
    int u, lane;
    uint64_t *bars;
    uint32_t phase = 0;    // bit s: parity of the next completion of slot s
    uint32_t pending = 0;  // bit s: slot s has copies in flight

    __device__ FastWarp(const DecodeParams &pp, unsigned char *wb)
        : p(pp), wbase(wb), L(KITTY, pp.n_boost), u(0), lane(threadIdx.x & 31) {
        bars = reinterpret_cast<uint64_t *>(wbase + L.bars);
    }
    __device__ unsigned char *slot(int s) const { return wbase + s * L.slot; }

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

    // key half of tile ti -> slot s
    __device__ void issue_k(int64_t ti, int s) {
        pending |= 1u << s;
        unsigned char *st = slot(s);
        const int nb = KITTY ? p.n_boost : 0;
        const uint32_t bytes = 8 * T::D * 4 + T::D * 4 + (KITTY ? 8 * nb * 4 + T::D : 0);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], bytes);
        __syncwarp();
        const int64_t page = ti >> p.tpp_shift;  // tiles per page: a power of two
        const int i = lane;
        if (i < 8) {
            issue_copy(st + T::OFF_K + i * T::K_STRIDE,
                       p.k_codes + ((size_t)u * (p.max_T / T::FPI) + ti * 8 + i) * T::D, T::D * 4, &bars[s]);
        } else if (i == 8) {
            issue_copy(st + T::OFF_KM, p.k_meta + ((size_t)u * (p.max_T / p.G) + page) * T::D * 2, T::D * 4,
                       &bars[s]);
        } else if (KITTY && nb > 0 && i < 17) {
            const int r = i - 9;
            issue_copy(st + T::OFF_HI + r * hi_stride(nb),
                       p.k_hi + ((size_t)u * (p.max_T / 16) + ti * 8 + r) * nb, nb * 4, &bars[s]);
        } else if (KITTY && i == 17) {
            issue_copy(st + T::OFF_HI + 8 * hi_stride(nb), p.k_bidx + ((size_t)u * (p.max_T / p.G) + page) * T::D,
                       T::D, &bars[s]);
        }
    }

    // value half of tile ti -> slot s
    __device__ void issue_v(int64_t ti, int s) {
        pending |= 1u << s;
        unsigned char *st = slot(s);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], T::V_ROWS * T::TOK * 4 + T::TOK * 4);
        __syncwarp();
        const int64_t tok0 = ti * T::TOK, page = ti >> p.tpp_shift;
        const int64_t off = (ti & ((1 << p.tpp_shift) - 1)) * T::TOK;
        const int i = lane;
        if (i < T::V_ROWS) {
            issue_copy(st + T::OFF_V + i * T::V_STRIDE,
                       p.v_codes + (((size_t)u * (p.max_T / p.G) + page) * T::V_ROWS + i) * p.G + off, T::TOK * 4,
                       &bars[s]);
        } else if (i == T::V_ROWS) {
            issue_copy(st + T::OFF_VM, p.v_meta + ((size_t)u * p.max_T + tok0) * 2, T::TOK * 4, &bars[s]);
        }
    }

    // 4 A registers of row set J from the split words (rows g / g+8, k pairs).
    template <int J>
    __device__ __forceinline__ static void frag(const uint32_t (&x)[4], const uint32_t (&xs)[4], uint32_t (&a)[4]) {
        constexpr int JJ = J < T::JDIRECT ? J : J - (T::SH / BITS);
        constexpr uint32_t M = T::MASK0 << (BITS * JJ);
#pragma unroll
        for (int r = 0; r < 4; r++) a[r] = (J < T::JDIRECT ? x[r] : xs[r]) & M;
    }
    template <int J>
    __device__ __forceinline__ static constexpr float unscale() {
        return (float)(1u << (24 - BITS * (J < T::JDIRECT ? J : J - (T::SH / BITS))));
    }
    // ldmatrix words W0..W3 (segments c = 0..3) -> k-paired registers (k = 2t, 2t+1 |
    // 2t+8, 2t+9) for rows g (low halves) and g+8 (high halves).
    __device__ __forceinline__ static void split(const uint32_t (&w)[4], uint32_t (&x)[4], uint32_t (&xs)[4]) {
        if (BITS == 2) {  // pairs (t, t+8) and (t+4, t+12)
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
        for (int r = 0; r < 4; r++) xs[r] = x[r] >> T::SH;
    }
    __device__ __forceinline__ static void mma_sets(float (&acc)[T::NJ][4], const uint32_t (&x)[4],
                                                    const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                                        \
    if (J < T::NJ) {                                                     \
        frag<J>(x, xs, a);                                               \
        mma_16816(acc[J % T::NJ], a[0], a[1], a[2], a[3], b0, b1);      \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }
    __device__ __forceinline__ static void mma_sets_o(float (&O)[8][4], int set, const uint32_t (&x)[4],
                                                      const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                                                  \
    if (J < T::NJ) {                                                               \
        frag<J>(x, xs, a);                                                         \
        mma_16816(O[set * T::NJ + (J % T::NJ)], a[0], a[1], a[2], a[3], b0, b1);  \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }

    // One 16-channel slab of S = Kcodes . q' (+ the min mma) for the key half in st.
    __device__ __forceinline__ void qk_slab(int sl, const unsigned char *st, float (&acc)[T::NJ][4],
                                            float (&cm)[4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const uint32_t *km = reinterpret_cast<const uint32_t *>(st + T::OFF_KM);
        const uint2 qp = reinterpret_cast<const uint2 *>(wbase + L.qpair)[((gq >> 1) * 8 + sl) * 4 + t];
        const SlabB b = slab_b(qp, km[chan_of<T::PS>(sl, t, 0)], km[chan_of<T::PS>(sl, t, 1)],
                               km[chan_of<T::PS>(sl, t, 2)], km[chan_of<T::PS>(sl, t, 3)], (gq & 1) != 0);
        mma_16816(cm, b.am0, b.am0, b.am1, b.am1, b.c0, b.c1);
        uint32_t w[4], x[4], xs[4];
        ldmatrix_x4(w, smem_u32(st + T::OFF_K) + (lane & 7) * T::K_STRIDE + 16 * (lane >> 3) + 64 * sl);
        split(w, x, xs);
        mma_sets(acc, x, xs, b.b0, b.b1);
    }

    // Kitty: S += hi-plane codes . (4 q') over the boosted slots.
    __device__ void qk_boost(const unsigned char *st, float (&acc)[T::NJ][4]) const {
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
                const int ch = invb[chan_of<T::PS>(s2, t, kk)] & (T::D - 1);
                km4[kk] = km[ch];
                qv[kk] = qraw[hq * 128 + ch];
            }
            q2[0] = hmul2((uint32_t)qv[0] | ((uint32_t)qv[1] << 16), 0x2C002C00u);
            q2[1] = hmul2((uint32_t)qv[2] | ((uint32_t)qv[3] << 16), 0x2C002C00u);
            q2[0] = hmul2(q2[0], s4);
            q2[1] = hmul2(q2[1], s4);
            const SlabB b = slab_b(make_uint2(q2[0], q2[1]), km4[0], km4[1], km4[2], km4[3], (gq & 1) != 0);
            uint32_t w[4], x[4], xs[4];
            ldmatrix_x4(w, hb + 64 * s2);
            split(w, x, xs);
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
        ldmatrix_x4(w, smem_u32(st + T::OFF_V) + (set * 8 + (lane & 7)) * T::V_STRIDE + 16 * (lane >> 3) + 64 * sl);
        split(w, x, xs);
        mma_sets_o(O, set, x, xs, bp.x, bp.y);
    }

    // Softmax of a tile from its S accumulators; rescales O; writes p' to pb.
    __device__ __forceinline__ void softmax(const float (&acc)[T::NJ][4], const float (&cm)[4],
                                            const unsigned char *stv, uint16_t *pb, float &m, float &l,
                                            float &mn, float (&O)[8][4]) const {
        const int gq = lane >> 2, t = lane & 3;
        const float C = kLog2e * rsqrtf((float)T::D) / kQScale;
        const float cst = cm[0] * C;  // row g, column 2t: sum_d q_d min_d of head t
        float z[T::NJ][2];
        float tm = -INFINITY;
#define KVQ_Z(J)                                                                        \
    if (J < T::NJ) {                                                                    \
        const float f = unscale<J>() * C;                                               \
        z[J % T::NJ][0] = fmaf(acc[J % T::NJ][0] + acc[J % T::NJ][1], f, cst);          \
        z[J % T::NJ][1] = fmaf(acc[J % T::NJ][2] + acc[J % T::NJ][3], f, cst);          \
        tm = fmaxf(tm, fmaxf(z[J % T::NJ][0], z[J % T::NJ][1]));                        \
    }
        KVQ_Z(0) KVQ_Z(1) KVQ_Z(2) KVQ_Z(3) KVQ_Z(4) KVQ_Z(5) KVQ_Z(6) KVQ_Z(7)
#undef KVQ_Z
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
        const float nm = fmaxf(m, tm);
        const float a = exp2f(m - nm);
        m = nm;
        l *= a;
        mn *= a;
        const float a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
        const float a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
#pragma unroll
        for (int o = 0; o < 8; o++) {
            O[o][0] *= a0;
            O[o][2] *= a0;
            O[o][1] *= a1;
            O[o][3] *= a1;
        }
        // value (scale, min) of the lane's tokens: 2 bits 16g..16g+15, 4 bits 8g..8g+7
        const uint32_t *vm = reinterpret_cast<const uint32_t *>(stv + T::OFF_VM);
        uint32_t vmr[16];
        if (BITS == 2) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(vm + 16 * gq);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const uint4 x = v4[i];
                vmr[4 * i] = x.x;
                vmr[4 * i + 1] = x.y;
                vmr[4 * i + 2] = x.z;
                vmr[4 * i + 3] = x.w;
            }
        } else {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(vm + 8 * gq);
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const uint4 x = v4[i];
                vmr[4 * i] = x.x;
                vmr[4 * i + 1] = x.y;
                vmr[4 * i + 2] = x.z;
                vmr[4 * i + 3] = x.w;
            }
        }
        uint16_t *row = pb + t * T::PROW;
#pragma unroll
        for (int j = 0; j < T::NJ; j++) {
            // rows g and g+8 of row set j: tokens (16g+j, 16g+j+8) or (8g+j, 8g+j+4)
            const int i0 = BITS == 2 ? j : j, i1 = BITS == 2 ? j + 8 : j + 4;
            const float2 sm0 = unpack_half2(vmr[i0]), sm1 = unpack_half2(vmr[i1]);
            const float p0 = exp2f(z[j][0] - m), p1 = exp2f(z[j][1] - m);
            l += p0 + p1;
            mn = fmaf(p0, sm0.y, fmaf(p1, sm1.y, mn));
            const int pos = BITS == 2 ? 16 * gq + 4 * (j & 3) + 2 * (j >> 2) : 16 * (gq >> 1) + 4 * j + 2 * (gq & 1);
            *reinterpret_cast<uint32_t *>(row + pos) = pack_half2(p0 * sm0.x, p1 * sm1.x);
        }
    }

    __device__ __forceinline__ void zero(float (&a)[T::NJ][4], float (&cm)[4]) const {
#pragma unroll
        for (int j = 0; j < T::NJ; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) a[j][e] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; e++) cm[e] = 0.f;
    }

    // Tiles [t0, t1) of sequence uu; writes the warp's partial [8][D+2] to `part`.
    // Software pipeline: PV of tile i runs interleaved with QK of tile i+1.
    __device__ void run(int uu, int64_t t0, int64_t t1, float *part) {
        u = uu;
        const int64_t n = t1 - t0;
        // slots: K(i) -> 2(i&1), V(i) -> 2(i&1)+1; the query's loads go out first, then
        // the first copies, whose latency overlaps staging the query
        const QRegs qr = load_q_regs(p, u);
        issue_k(t0, 0);
        issue_v(t0, 1);
        if (n > 1) {
            issue_k(t0 + 1, 2);
            issue_v(t0 + 1, 3);
        }
        store_q_warp<T::PS>(qr, reinterpret_cast<uint16_t *>(wbase + L.qraw),
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
        float acc[T::NJ][4], cm[4];
        bool ok = true;

        // prologue: QK(0), softmax(0)
        ok &= wait_slot(0);
        zero(acc, cm);
#pragma unroll
        for (int sl = 0; sl < 8; sl++) qk_slab(sl, slot(0), acc, cm);
        if (KITTY && p.n_boost > 0) qk_boost(slot(0), acc);
        __syncwarp();
        fence_proxy_async();
        if (n > 2) issue_k(t0 + 2, 0);
        ok &= wait_slot(1);
        softmax(acc, cm, slot(1), pb0, m, l, mn, O);
        __syncwarp();

        for (int64_t i = 0; i < n && ok; i++) {
            const int kv = 2 * (int)(i & 1), kn = 2 * (int)((i + 1) & 1);
            const uint16_t *pb = pb0 + (i & 1) * 4 * T::PROW;
            if (i + 1 < n) {
                ok &= wait_slot(kn);
                zero(acc, cm);
#pragma unroll
                for (int sl = 0; sl < 8; sl++) {
                    pv_step(sl, slot(kv + 1), pb, O);
                    qk_slab(sl, slot(kn), acc, cm);
                }
                if (KITTY && p.n_boost > 0) qk_boost(slot(kn), acc);
            } else {
#pragma unroll
                for (int sl = 0; sl < 8; sl++) pv_step(sl, slot(kv + 1), pb, O);
            }
            __syncwarp();
            fence_proxy_async();
            if (i + 2 < n) issue_v(t0 + i + 2, kv + 1);
            if (i + 1 < n) {
                if (i + 3 < n) issue_k(t0 + i + 3, kn);
                ok &= wait_slot(kn + 1);
                softmax(acc, cm, slot(kn + 1), pb0 + ((i + 1) & 1) * 4 * T::PROW, m, l, mn, O);
                __syncwarp();
            }
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
    if (J < T::NJ && t < 2) {                                                      \
        const float f = unscale<J>();                                              \
        for (int set = 0; set < T::NSET; set++) {                                  \
            const int o = set * T::NJ + (J % T::NJ);                               \
            const int ch = T::FPI * (gq + 8 * set) + (J % T::NJ);                  \
            const int ch2 = ch + T::FPI / 2;                                       \
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
// Mini tiles: 16 tokens with fp16 values
// ---------------------------------------------------------------------------
// Mini tile mi of a sequence: [sink tiles][packed-key blocks][fp16-buffer tiles].
struct MiniTile {
    int64_t tok0;   // first logical token
    int n;          // valid tokens (1..16)
    bool kpacked;   // keys from a packed 16-token block (Kitty), else fp16 rows
};

__device__ __forceinline__ MiniTile mini_tile(const DecodeParams &p, int64_t mi) {
    MiniTile m;
    const int64_t ms = (p.n_sink + 15) >> 4, tok_fast = p.n_fast * (p.bits == 2 ? 128 : 64);
    const int64_t mp = (p.T_k - tok_fast) >> 4;
    if (mi < ms) {
        m.tok0 = 16 * mi;
        m.n = (int)kvq_min64(16, p.n_sink - m.tok0);
        m.kpacked = false;
    } else if (mi < ms + mp) {
        m.tok0 = p.n_sink + tok_fast + 16 * (mi - ms);
        m.n = 16;
        m.kpacked = true;
    } else {
        m.tok0 = p.n_sink + p.T_k + 16 * (mi - ms - mp);
        m.n = (int)kvq_min64(16, p.L - m.tok0);
        m.kpacked = false;
    }
    return m;
}

// fp16 value row of logical token tl (tl outside the packed values).
__device__ __forceinline__ const uint16_t *vrow16(const DecodeParams &p, int u, int64_t tl) {
    if (tl < p.n_sink) return p.v_sink + ((size_t)u * p.S_cap + tl) * 128;
    const int64_t r = tl - p.n_sink - p.T_v;
    if (r < p.n_vres) return p.v_res + ((size_t)u * p.cap_v + r) * 128;
    int64_t slot = p.local_head + (r - p.n_vres);  // < 2 R: local_head < R, r - n_vres < n_local <= R
    if (slot >= p.R_local) slot -= p.R_local;
    return p.v_local + ((size_t)u * p.R_local + slot) * 128;
}
__device__ __forceinline__ const uint16_t *krow16(const DecodeParams &p, int u, int64_t tl) {
    if (tl < p.n_sink) return p.k_sink + ((size_t)u * p.S_cap + tl) * 128;
    return p.k_res + ((size_t)u * p.cap_k + (tl - p.n_sink - p.T_k)) * 128;
}

template <int BITS, bool KITTY>
struct MiniWarp {
    const DecodeParams &p;
    unsigned char *wbase;
    WarpSmem<BITS> L;  // the CTA's per-warp layout (slots are large enough for a mini tile)
    int u, lane;
    uint64_t *bars;
    uint32_t phase = 0, pending = 0;

    // packed-key block layout in the key half of a slot
    static constexpr int MB_W = 0, MB_M = 512, MB_HI = 1024;

    __device__ MiniWarp(const DecodeParams &pp, unsigned char *wb, int slot_bits)
        : p(pp), wbase(wb), L(KITTY, pp.n_boost), u(0), lane(threadIdx.x & 31) {
        (void)slot_bits;
        bars = reinterpret_cast<uint64_t *>(wbase + L.bars);
    }
    __device__ unsigned char *slot(int s) const { return wbase + s * L.slot; }
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
        if (lane < 16) {
            if (!mt.kpacked) {
                issue_copy(sK + i * kMiniRow, krow16(p, u, tl), 256, &bars[sk]);
            } else {
                const int64_t tk = mt.tok0 - p.n_sink, page = tk >> p.g_shift, blk = tk >> 4;
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
            issue_copy(sV + i * kMiniRow, vrow16(p, u, tl), 256, &bars[sk + 1]);
        }
    }

    __device__ void run(int uu, int64_t m0, int64_t m1, float *part) {
        u = uu;
        const int gq = lane >> 2, t = lane & 3, hq = gq >> 1;
        const bool lo_col = (gq & 1) != 0;
        const int64_t n = m1 - m0;
        uint16_t *qraw = reinterpret_cast<uint16_t *>(wbase + L.qraw);
        const QRegs qr = load_q_regs(p, u);
        issue(mini_tile(p, u_base(m0)), 0);
        if (n > 1) issue(mini_tile(p, u_base(m0 + 1)), 2);
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
            const MiniTile mt = mini_tile(p, u_base(m0 + i));
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
                    mma_16816(s, a[0], a[1], a[2], a[3], b0, b1);
                }
            } else {
                // Kitty mixed block: 16 tokens of packed keys, rows g / g+8 <-> tokens g / g+8
                const uint32_t *w = reinterpret_cast<const uint32_t *>(sK + MB_W);
                const uint32_t *km = reinterpret_cast<const uint32_t *>(sK + MB_M);
                const uint2 *qpair = reinterpret_cast<const uint2 *>(wbase + L.qpair);
#pragma unroll
                for (int sl = 0; sl < 8; sl++) {
                    const SlabB b = slab_b(qpair[(hq * 8 + sl) * 4 + t], km[chan_of<8>(sl, t, 0)],
                                           km[chan_of<8>(sl, t, 1)], km[chan_of<8>(sl, t, 2)],
                                           km[chan_of<8>(sl, t, 3)], lo_col);
                    mma_16816(cm, b.am0, b.am0, b.am1, b.am1, b.c0, b.c1);
                    uint32_t wv[4], x[4], xs[4];
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) wv[kk] = w[16 * sl + 4 * kk + t];
                    FastWarp<2, KITTY>::split(wv, x, xs);
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
                        const SlabB b = slab_b(make_uint2(q0, q1), km4[0], km4[1], km4[2], km4[3], lo_col);
                        uint32_t wv[4], x[4], xs[4];
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) wv[kk] = hw[16 * s2 + 4 * kk + t];
                        FastWarp<2, KITTY>::split(wv, x, xs);
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
            float z0 = fmaf(s[0] + s[1], unsc * C, cst), z1 = fmaf(s[2] + s[3], unsc * C, cst);
            if (gq >= mt.n) z0 = -INFINITY;
            if (gq + 8 >= mt.n) z1 = -INFINITY;
            float tm = fmaxf(z0, z1);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
            const float nm = fmaxf(m, tm);
            const float a = exp2f(m - nm);
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
            const float p0 = exp2f(z0 - m), p1 = exp2f(z1 - m);
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
            if (i + 2 < n) issue(mini_tile(p, u_base(m0 + i + 2)), sk);
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
