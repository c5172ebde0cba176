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

constexpr float kLog2e = 1.4426950408889634f;
constexpr int KVQ_DEV_BAD_STATE_BIT = 2;

__host__ __device__ __forceinline__ int64_t kvq_min64(int64_t a, int64_t b) { return a < b ? a : b; }

template <int BITS>
struct Tile {
    static constexpr int D = 128;
    static constexpr int FPI = 32 / BITS;
    static constexpr int TOK = BITS == 2 ? 128 : 64;     // tokens per tile (8 words of keys)
    static constexpr int K_STRIDE = D * 4 + 16;          // padded key row (conflict-free ldmatrix)
    static constexpr int V_ROWS = D / FPI;               // channel blocks: 8 or 16
    static constexpr int V_STRIDE = TOK * 4 + 16;
    static constexpr int NJ = FPI / 2;                   // row sets per word: 8 or 4
    static constexpr int NSET = V_ROWS / 8;              // 1 or 2
    static constexpr int TSLABS = TOK / 16;              // 16-token slabs for PV
    static constexpr int JDIRECT = BITS == 2 ? 5 : 2;    // row sets readable without a shift
    static constexpr int SH = BITS == 2 ? 6 : 8;         // pre-shift for the others
    static constexpr uint32_t MASK0 = BITS == 2 ? 0x00030003u : 0x000F000Fu;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + 8 * K_STRIDE;
    static constexpr int OFF_KM = OFF_V + V_ROWS * V_STRIDE;
    static constexpr int OFF_VM = OFF_KM + D * 4;
    static constexpr int OFF_HI = OFF_VM + TOK * 4;
    static constexpr int PBUF = 8 * TOK * 2;
};

__host__ __device__ inline int hi_stride(int nb) { return nb * 4 + 16; }

template <int BITS>
__host__ __device__ inline int stage_bytes(bool kitty, int nb) {
    int s = Tile<BITS>::OFF_HI + (kitty ? 8 * hi_stride(nb) + 128 : 0);
    return (s + 127) & ~127;
}

__host__ __device__ inline int part_bytes(int D) { return 8 * (D + 2) * 4; }
__host__ __device__ inline int qbuf_bytes(int D) { return 8 * D * 2; }

// Per-warp shared memory, fast kernel:
//   [stage 0 .. kStages-1][p' buffer][q buffer fp16 [8][D]][slot index 64 B][mbarriers]
// The warp's final partial is written over its stage 0 after its last tile.
template <int BITS>
__host__ __device__ inline int fast_warp_bytes(bool kitty, int nb) {
    int s = kStages * stage_bytes<BITS>(kitty, nb) + Tile<BITS>::PBUF + qbuf_bytes(Tile<BITS>::D) + 64 +
            8 * kStages;
    return (s + 127) & ~127;
}
template <int BITS>
__host__ __device__ inline int fast_qbuf_off(bool kitty, int nb) {
    return kStages * stage_bytes<BITS>(kitty, nb) + Tile<BITS>::PBUF;
}

// Per-warp shared memory, generic-only kernel: [partial][q buffer].
__host__ __device__ inline int gen_warp_bytes(int D) {
    return (part_bytes(D) + qbuf_bytes(D) + 127) & ~127;
}

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
        for (int i = 0; i < DPL; i++) part[h * (D + 2) + lane * DPL + i] = st.o[h][i];
        if (lane == 0) {
            part[h * (D + 2) + D] = st.m[h];
            part[h * (D + 2) + D + 1] = l;
        }
    }
}

// ---------------------------------------------------------------------------------
// Fast path: packed tiles on the tensor cores.
// ---------------------------------------------------------------------------------
template <int BITS, bool KITTY>
struct FastWarp {
    using T = Tile<BITS>;
    const DecodeParams &p;
    unsigned char *wbase;
    int u, lane;
    int sbytes;
    uint64_t *bars;
    uint32_t phase = 0;    // bit s: parity of the next completion of stage s
    uint32_t pending = 0;  // bit s: stage s has copies in flight

    __device__ void init_bars() {
        if (lane == 0) {
            for (int s = 0; s < kStages; s++) mbar_init(&bars[s], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }

    __device__ FastWarp(const DecodeParams &pp, unsigned char *wb)
        : p(pp), wbase(wb), u(0), lane(threadIdx.x & 31) {
        sbytes = stage_bytes<BITS>(KITTY, p.n_boost);
        bars = reinterpret_cast<uint64_t *>(wbase + fast_qbuf_off<BITS>(KITTY, p.n_boost) + qbuf_bytes(T::D) + 64);
    }

    __device__ unsigned char *stage(int s) const { return wbase + s * sbytes; }

    __device__ uint32_t tile_bytes() const {
        uint32_t b = 8 * T::D * 4 + T::V_ROWS * T::TOK * 4 + T::D * 4 + T::TOK * 4;
        if (KITTY) b += 8 * p.n_boost * 4 + T::D;
        return b;
    }

    // Enqueue the bulk copies of tile ti into stage s (whole warp).
    __device__ void issue(int64_t ti, int s) {
        pending |= 1u << s;
        unsigned char *st = stage(s);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], tile_bytes());
        __syncwarp();
        const int64_t tok0 = ti * T::TOK;                  // packed-token index
        const int64_t page = tok0 / p.G, off = tok0 % p.G;
        const int nk = 8, nv = T::V_ROWS;
        const int i = lane;
        if (i < nk) {
            const int32_t *src = p.k_codes + ((size_t)u * (p.max_T / T::FPI) + ti * 8 + i) * T::D;
            bulk_g2s(st + T::OFF_K + i * T::K_STRIDE, src, T::D * 4, &bars[s]);
        } else if (i < nk + nv) {
            const int m = i - nk;
            const int32_t *src = p.v_codes + (((size_t)u * (p.max_T / p.G) + page) * T::V_ROWS + m) * p.G + off;
            bulk_g2s(st + T::OFF_V + m * T::V_STRIDE, src, T::TOK * 4, &bars[s]);
        } else if (i == nk + nv) {
            const uint16_t *src = p.k_meta + ((size_t)u * (p.max_T / p.G) + page) * T::D * 2;
            bulk_g2s(st + T::OFF_KM, src, T::D * 4, &bars[s]);
        } else if (i == nk + nv + 1) {
            const uint16_t *src = p.v_meta + ((size_t)u * p.max_T + tok0) * 2;
            bulk_g2s(st + T::OFF_VM, src, T::TOK * 4, &bars[s]);
        } else if (KITTY && i < nk + nv + 2 + 8) {
            const int r = i - (nk + nv + 2);
            const int32_t *src = p.k_hi + ((size_t)u * (p.max_T / 16) + ti * 8 + r) * p.n_boost;
            bulk_g2s(st + T::OFF_HI + r * hi_stride(p.n_boost), src, p.n_boost * 4, &bars[s]);
        } else if (KITTY && i == nk + nv + 2 + 8) {
            const uint8_t *src = p.k_bidx + ((size_t)u * (p.max_T / p.G) + page) * T::D;
            bulk_g2s(st + T::OFF_HI + 8 * hi_stride(p.n_boost), src, T::D, &bars[s]);
        }
    }

    // The 4 A-operand registers of row set j from the 4 ldmatrix words (see header).
    template <int J>
    __device__ __forceinline__ static void frag(const uint32_t (&x)[4], const uint32_t (&xs)[4],
                                                uint32_t (&a)[4]) {
        constexpr int JJ = J < T::JDIRECT ? J : J - (T::SH / BITS);
        constexpr uint32_t M = T::MASK0 << (BITS * JJ);
#pragma unroll
        for (int r = 0; r < 4; r++) a[r] = (J < T::JDIRECT ? x[r] : xs[r]) & M;
    }
    template <int J>
    __device__ __forceinline__ static float unscale() {
        constexpr int JJ = J < T::JDIRECT ? J : J - (T::SH / BITS);
        return (float)(1u << (24 - BITS * JJ));
    }

    __device__ __forceinline__ static void split(const uint32_t (&w)[4], uint32_t (&x)[4], uint32_t (&xs)[4]) {
        x[0] = prmt(w[0], w[1], 0x5410);  // rows g   (low halves),  k = 2t, 2t+1
        x[1] = prmt(w[0], w[1], 0x7632);  // rows g+8 (high halves)
        x[2] = prmt(w[2], w[3], 0x5410);  // rows g,   k = 2t+8, 2t+9
        x[3] = prmt(w[2], w[3], 0x7632);
#pragma unroll
        for (int r = 0; r < 4; r++) xs[r] = x[r] >> T::SH;
    }

    // Token (within tile) of accumulator element e of row set j for this lane.
    __device__ __forceinline__ int tok_of(int j, int e) const {
        const int gq = lane >> 2;
        if (BITS == 2) return 16 * gq + j + ((e >> 1) ? 8 : 0);
        return 8 * gq + j + ((e >> 1) ? 4 : 0);
    }

    // Tiles [t0, t1) of sequence uu; writes the warp's partial [8][D+2] to `part`.
    // The mbarriers must be initialized (init_bars) and idle (all phases consumed).
    //
    // Query heads (g <= 4) and precision: q' = q * scale_k * log2e/sqrt(D) is split
    // into fp16 hi + lo parts (22 significant bits); mma column 2h carries hi(q'_h),
    // column 2h+1 carries lo(q'_h), so the lane that owns columns 2t, 2t+1 of the
    // S tile adds them and owns head t of the softmax.  For PV the p' tile has one
    // column per head (heads 4..7 zero), so the output lanes own heads 2t, 2t+1.
    __device__ void run(int uu, int64_t t0, int64_t t1, const uint16_t *q_w, float *part) {
        u = uu;
        const int gq = lane >> 2, t = lane & 3;
        const int hq = gq >> 1;            // head whose q' part feeds mma column gq
        const bool lo_col = (gq & 1) != 0;
        const float C = kLog2e * rsqrtf((float)T::D);
        const int64_t n = t1 - t0;
        for (int s = 0; s < kStages && s < n; s++) issue(t0 + s, s);

        float m = -INFINITY, l = 0.f, mn = 0.f;  // softmax state of head t
        float O[8][4];
#pragma unroll
        for (int o = 0; o < 8; o++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[o][e] = 0.f;
        bool failed = false;
        unsigned char *pbuf = wbase + kStages * sbytes;
        uint16_t *pb = reinterpret_cast<uint16_t *>(pbuf);
        uint8_t *invb = wbase + fast_qbuf_off<BITS>(KITTY, p.n_boost) + qbuf_bytes(T::D);  // [64]
        for (int i = lane; i < 4 * T::TOK / 2; i += 32)  // p' rows of heads 4..7 stay zero
            reinterpret_cast<uint32_t *>(pb + 4 * T::TOK)[i] = 0u;
        __syncwarp();

        for (int64_t i = 0; i < n && !failed; i++) {
            const int s = (int)(i % kStages);
            if (!mbar_wait(&bars[s], (phase >> s) & 1u, p.status)) {
                failed = true;
                break;
            }
            phase ^= 1u << s;
            pending &= ~(1u << s);
            unsigned char *st = stage(s);
            const uint32_t *km = reinterpret_cast<const uint32_t *>(st + T::OFF_KM);

            // ---- S = Kcodes . q'  (hi/lo columns), plus the per-head min constant ----
            float acc[T::NJ][4];
#pragma unroll
            for (int j = 0; j < T::NJ; j++)
#pragma unroll
                for (int e = 0; e < 4; e++) acc[j][e] = 0.f;
            float cst = 0.f;
            const uint32_t kb = smem_u32(st + T::OFF_K) + (lane & 7) * T::K_STRIDE + 16 * (lane >> 3);
#pragma unroll
            for (int sl = 0; sl < 8; sl++) {
                float qp[4];
#pragma unroll
                for (int cc = 0; cc < 4; cc++) {
                    const int ch = 16 * sl + 4 * cc + t;
                    const float2 sm = unpack_half2(km[ch]);
                    const float qv = h2f(q_w[hq * T::D + ch]);
                    qp[cc] = split_part(qv * sm.x * C, lo_col);
                    cst = fmaf(qv, sm.y, cst);
                }
                uint32_t w[4], x[4], xs[4];
                ldmatrix_x4(w, kb + 64 * sl);
                split(w, x, xs);
                mma_rowsets(acc, x, xs, pack_half2(qp[0], qp[1]), pack_half2(qp[2], qp[3]));
            }
            if (KITTY && p.n_boost > 0) {
                // Boosted channels: S += hi . (4 q'), slots gathered through the index.
                const uint8_t *bi = st + T::OFF_HI + 8 * hi_stride(p.n_boost);
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const int ch = lane * 4 + r;
                    const int sl = bi[ch];
                    if (sl < p.n_boost) invb[sl] = (uint8_t)ch;
                }
                __syncwarp();
                const int nsl = p.n_boost / 16;
                const uint32_t hb = smem_u32(st + T::OFF_HI) + (lane & 7) * hi_stride(p.n_boost) + 16 * (lane >> 3);
                for (int s2 = 0; s2 < nsl; s2++) {
                    float qp[4];
#pragma unroll
                    for (int cc = 0; cc < 4; cc++) {
                        const int ch = invb[16 * s2 + 4 * cc + t] & (T::D - 1);
                        const float2 sm = unpack_half2(km[ch]);
                        qp[cc] = split_part(4.0f * h2f(q_w[hq * T::D + ch]) * sm.x * C, lo_col);
                    }
                    uint32_t w[4], x[4], xs[4];
                    ldmatrix_x4(w, hb + 64 * s2);
                    split(w, x, xs);
                    mma_rowsets(acc, x, xs, pack_half2(qp[0], qp[1]), pack_half2(qp[2], qp[3]));
                }
                __syncwarp();
            }
            cst += __shfl_xor_sync(0xffffffffu, cst, 1);
            cst += __shfl_xor_sync(0xffffffffu, cst, 2);
            const float ct = __shfl_sync(0xffffffffu, cst, (2 * t) * 4) * C;  // head t

            // ---- online softmax over the tile (head t; rows g and g+8 of each row set) ----
            float z[T::NJ][2];
            unscale_logits(acc, z, ct);
            float tm = -INFINITY;
#pragma unroll
            for (int j = 0; j < T::NJ; j++) tm = fmaxf(tm, fmaxf(z[j][0], z[j][1]));
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
            const float nm = fmaxf(m, tm);
            const float a = exp2f(m - nm);
            m = nm;
            l *= a;
            mn *= a;
            // the output lanes own heads 2t, 2t+1: fetch their rescale factors
            const float a0 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t) & 3));
            const float a1 = __shfl_sync(0xffffffffu, a, (lane & ~3) | ((2 * t + 1) & 3));
#pragma unroll
            for (int o = 0; o < 8; o++) {
                O[o][0] *= a0;
                O[o][2] *= a0;
                O[o][1] *= a1;
                O[o][3] *= a1;
            }
            const uint32_t *vm = reinterpret_cast<const uint32_t *>(st + T::OFF_VM);
#pragma unroll
            for (int j = 0; j < T::NJ; j++) {
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const int tok = tok_of(j, 2 * e);
                    const float pe = exp2f(z[j][e] - m);
                    const float2 sm = unpack_half2(vm[tok]);
                    l += pe;
                    mn = fmaf(pe, sm.y, mn);
                    const int r = tok & 15;
                    pb[t * T::TOK + (tok & ~15) + 4 * (r & 3) + (r >> 2)] =
                        __half_as_ushort(__float2half_rn(pe * sm.x));
                }
            }
            __syncwarp();

            // ---- O += Vcodes . p' ----
            const uint32_t vb = smem_u32(st + T::OFF_V) + (lane & 7) * T::V_STRIDE + 16 * (lane >> 3);
#pragma unroll
            for (int sl = 0; sl < T::TSLABS; sl++) {
                const uint2 bp = *reinterpret_cast<const uint2 *>(pb + gq * T::TOK + 16 * sl + 4 * t);
#pragma unroll
                for (int set = 0; set < T::NSET; set++) {
                    uint32_t w[4], x[4], xs[4];
                    ldmatrix_x4(w, vb + set * 8 * T::V_STRIDE + 64 * sl);
                    split(w, x, xs);
                    mma_rowsets_o(O, set, x, xs, bp.x, bp.y);
                }
            }
            __syncwarp();
            fence_proxy_async();
            if (i + kStages < n) issue(t0 + i + kStages, s);
        }
        if (failed) {
            // let copies already in flight land before the shared memory is reused
            for (int s = 0; s < kStages; s++)
                if (pending & (1u << s)) mbar_wait(&bars[s], (phase >> s) & 1u, p.status);
            pending = 0;
        }
        // ---- warp partial ----
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            mn += __shfl_xor_sync(0xffffffffu, mn, o);
        }
        const float mn0 = __shfl_sync(0xffffffffu, mn, (lane & ~3) | ((2 * t) & 3));
        const float mn1 = __shfl_sync(0xffffffffu, mn, (lane & ~3) | ((2 * t + 1) & 3));
        __syncwarp();
        store_o(O, part, mn0, mn1);
        if (gq == 0) {
            part[t * (T::D + 2) + T::D] = m;
            part[t * (T::D + 2) + T::D + 1] = l;
        }
    }

    // hi part (fp16-rounded) or lo part (remainder, rounded later to fp16) of x.
    __device__ __forceinline__ static float split_part(float x, bool lo) {
        const float hi = __half2float(__float2half_rn(x));
        return lo ? x - hi : hi;
    }

    __device__ __forceinline__ static void mma_rowsets(float (&acc)[T::NJ][4], const uint32_t (&x)[4],
                                                       const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                           \
    if (J < T::NJ) {                                        \
        frag<J>(x, xs, a);                                  \
        mma_16816(acc[J % T::NJ], a[0], a[1], a[2], a[3], b0, b1); \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }

    __device__ __forceinline__ static void mma_rowsets_o(float (&O)[8][4], int set, const uint32_t (&x)[4],
                                                         const uint32_t (&xs)[4], uint32_t b0, uint32_t b1) {
        uint32_t a[4];
#define KVQ_RS(J)                                                              \
    if (J < T::NJ) {                                                           \
        frag<J>(x, xs, a);                                                     \
        mma_16816(O[set * T::NJ + (J % T::NJ)], a[0], a[1], a[2], a[3], b0, b1); \
    }
        KVQ_RS(0) KVQ_RS(1) KVQ_RS(2) KVQ_RS(3) KVQ_RS(4) KVQ_RS(5) KVQ_RS(6) KVQ_RS(7)
#undef KVQ_RS
    }

    // z[j][0] (row g) and z[j][1] (row g+8) of head t: hi + lo columns, unscaled, + constant.
    __device__ __forceinline__ static void unscale_logits(const float (&acc)[T::NJ][4], float (&z)[T::NJ][2],
                                                          float c) {
#define KVQ_US(J)                                                                   \
    if (J < T::NJ) {                                                                \
        const float f = unscale<J>();                                               \
        z[J % T::NJ][0] = fmaf(acc[J % T::NJ][0] + acc[J % T::NJ][1], f, c);        \
        z[J % T::NJ][1] = fmaf(acc[J % T::NJ][2] + acc[J % T::NJ][3], f, c);        \
    }
        KVQ_US(0) KVQ_US(1) KVQ_US(2) KVQ_US(3) KVQ_US(4) KVQ_US(5) KVQ_US(6) KVQ_US(7)
#undef KVQ_US
    }

    // O row set o = set*NJ + j: rows g <-> channel FPI*(gq+8*set) + j, g+8 <-> + FPI/2.
    __device__ __forceinline__ void store_o(const float (&O)[8][4], float *part, float mn0, float mn1) const {
        const int gq = lane >> 2, t = lane & 3;
#define KVQ_SO(J)                                                                        \
    if (J < T::NJ) {                                                                     \
        const float f = unscale<J>();                                                    \
        for (int set = 0; set < T::NSET; set++) {                                        \
            const int o = set * T::NJ + (J % T::NJ);                                     \
            const int ch = T::FPI * (gq + 8 * set) + (J % T::NJ);                        \
            const int ch2 = ch + T::FPI / 2;                                             \
            part[(2 * t) * (T::D + 2) + ch] = fmaf(O[o][0], f, mn0);                     \
            part[(2 * t + 1) * (T::D + 2) + ch] = fmaf(O[o][1], f, mn1);                 \
            part[(2 * t) * (T::D + 2) + ch2] = fmaf(O[o][2], f, mn0);                    \
            part[(2 * t + 1) * (T::D + 2) + ch2] = fmaf(O[o][3], f, mn1);                \
        }                                                                                \
    }
        KVQ_SO(0) KVQ_SO(1) KVQ_SO(2) KVQ_SO(3) KVQ_SO(4) KVQ_SO(5) KVQ_SO(6) KVQ_SO(7)
#undef KVQ_SO
    }
};

// ---------------------------------------------------------------------------------
// Schedule arithmetic shared by every CTA (closed forms, no tables).
// ---------------------------------------------------------------------------------
// Fast warp k (of W = 8*C_f) owns flattened tiles [a_k, a_{k+1}), a_k = floor(k*N/W).
__device__ __forceinline__ int64_t fast_a(const DecodeParams &p, int64_t k) {
    return k * p.N_f / (8 * (int64_t)p.C_f);
}
// The warp whose range holds flattened tile x: the largest k with a_k <= x.
__device__ __forceinline__ int64_t fast_warp_of(const DecodeParams &p, int64_t x) {
    const int64_t W = 8 * (int64_t)p.C_f;
    const int64_t k = ((x + 1) * W - 1) / p.N_f;
    return k < W - 1 ? k : W - 1;
}
__device__ __forceinline__ int n_fast_ctas(const DecodeParams &p, int u, int *first) {
    if (p.n_fast == 0) { *first = 0; return 0; }
    const int c0 = (int)(fast_warp_of(p, (int64_t)u * p.n_fast) / 8);
    const int c1 = (int)(fast_warp_of(p, (int64_t)(u + 1) * p.n_fast - 1) / 8);
    *first = c0;
    return c1 - c0 + 1;
}
__device__ __forceinline__ int n_gen_ctas(const DecodeParams &p, int u, int *first) {
    if (p.n_gc == 0) { *first = 0; return 0; }
    const int c0 = (int)(((int64_t)u * p.n_gc) / 8);
    const int c1 = (int)(((int64_t)(u + 1) * p.n_gc - 1) / 8);
    *first = c0;
    return c1 - c0 + 1;
}

__device__ __forceinline__ void load_q(const DecodeParams &p, int u, uint16_t *q_w) {
    const int lane = threadIdx.x & 31, D = p.D;
    for (int i = lane; i < 8 * D / 8; i += 32) {
        const int h = (i * 8) / D, d = (i * 8) % D;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < p.g) v = *reinterpret_cast<const uint4 *>(p.q + ((size_t)u * p.g + h) * D + d);
        *reinterpret_cast<uint4 *>(q_w + h * D + d) = v;
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------------
template <int BITS, bool KITTY, bool FAST, int DPL>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_seg[kWarps][2];   // sequence of each warp segment (-1: none)
    __shared__ int s_last[16];         // sequences this CTA must combine
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, D = p.D, g = p.g;
    const int wbytes = FAST ? fast_warp_bytes<BITS>(KITTY, p.n_boost) : gen_warp_bytes(D);
    unsigned char *wbase = smem + warp * wbytes;
    float *part = reinterpret_cast<float *>(wbase);  // final partial of this warp, [8][D+2]
    const bool fast_cta = FAST && c < p.C_f;
    int seg0 = -1, seg1 = -1;

    if (fast_cta) {
        // ---- fast warp: flattened tile range, at most two sequences ----
        const int64_t k = (int64_t)c * kWarps + warp;
        const int64_t x0 = fast_a(p, k), x1 = fast_a(p, k + 1);
        uint16_t *q_w = reinterpret_cast<uint16_t *>(wbase + fast_qbuf_off<BITS>(KITTY, p.n_boost));
        FastWarp<BITS, KITTY> fw(p, wbase);
        fw.init_bars();
        int64_t x = x0;
        if (x < x1) {
            const int u0 = (int)(x / p.n_fast);
            const int64_t e0 = kvq_min64(x1, (int64_t)(u0 + 1) * p.n_fast);
            // a first segment followed by another one is parked in global scratch;
            // the warp's last segment stays in its shared-memory slot
            const bool two = e0 < x1;
            float *dst = two ? p.scratch + (size_t)k * part_bytes(D) / 4 : part;
            load_q(p, u0, q_w);
            fw.run(u0, x - (int64_t)u0 * p.n_fast, e0 - (int64_t)u0 * p.n_fast, q_w, dst);
            if (two) seg0 = u0;
            else seg1 = u0;
            x = e0;
        }
        if (x < x1) {
            const int u1 = (int)(x / p.n_fast);
            load_q(p, u1, q_w);
            fw.run(u1, x - (int64_t)u1 * p.n_fast, x1 - (int64_t)u1 * p.n_fast, q_w, part);
            seg1 = u1;
        }
    } else {
        // ---- generic warp: one chunk of one sequence ----
        const int64_t j = (int64_t)(c - (FAST ? p.C_f : 0)) * kWarps + warp;
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
            uint16_t *q_w = reinterpret_cast<uint16_t *>(
                wbase + (FAST ? fast_qbuf_off<BITS>(KITTY, p.n_boost) : part_bytes(D)));
            load_q(p, u, q_w);
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
    int ulo = 0x7fffffff, uhi = -1;
    for (int w = 0; w < kWarps; w++)
        for (int e = 0; e < 2; e++)
            if (s_seg[w][e] >= 0) {
                ulo = min(ulo, s_seg[w][e]);
                uhi = max(uhi, s_seg[w][e]);
            }
    if (uhi - ulo >= 16) {  // cannot happen with the host schedule; never index past s_last
        report(p.status, KVQ_DEV_BAD_STATE_BIT);
        return;
    }
    const int wb = wbytes / 4;  // floats between warp partials in shared memory
    const float *wpart = reinterpret_cast<const float *>(smem);
    for (int u = ulo; u <= uhi; u++) {
        int f0, g0;
        const int nf = n_fast_ctas(p, u, &f0);
        const int ng = n_gen_ctas(p, u, &g0);
        const int slot = fast_cta ? c - f0 : nf + (c - (FAST ? p.C_f : 0) - g0);
        float *gpart = p.partials + ((size_t)u * p.max_slots + slot) * g * (D + 2);
        for (int i = tid; i < g * (D + 2); i += blockDim.x) {
            const int h = i / (D + 2), d = i % (D + 2);
            const float *src[2 * kWarps];
            int n = 0;
            for (int w = 0; w < kWarps; w++) {
                if (s_seg[w][0] == u)
                    src[n++] = p.scratch + ((size_t)c * kWarps + w) * part_bytes(D) / 4;
                if (s_seg[w][1] == u) src[n++] = wpart + w * wb;
            }
            float M = -INFINITY;
            for (int k2 = 0; k2 < n; k2++) M = fmaxf(M, src[k2][h * (D + 2) + D]);
            float acc = 0.f;
            for (int k2 = 0; k2 < n; k2++) {
                const float mw = src[k2][h * (D + 2) + D];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - M);
                if (d < D) acc = fmaf(src[k2][h * (D + 2) + d], f, acc);
                else if (d == D + 1) acc = fmaf(src[k2][h * (D + 2) + D + 1], f, acc);
            }
            gpart[h * (D + 2) + d] = (d == D) ? M : acc;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last[u - ulo] = (atomicAdd(&p.tickets[u], 1) == nf + ng - 1);
        __syncthreads();
    }
    if (uhi < 0) return;

    // ---- the last CTA of a sequence: log-sum-exp combine of its slots ----
    for (int u = ulo; u <= uhi; u++) {
        if (!s_last[u - ulo]) continue;
        __threadfence();
        int f0, g0;
        const int ns = n_fast_ctas(p, u, &f0) + n_gen_ctas(p, u, &g0);
        const float *up = p.partials + (size_t)u * p.max_slots * g * (D + 2);
        for (int i = tid; i < g * D; i += blockDim.x) {
            const int h = i / D, d = i % D;
            float M = -INFINITY;
            for (int cc = 0; cc < ns; cc++) M = fmaxf(M, __ldcg(up + ((size_t)cc * g + h) * (D + 2) + D));
            float L = 0.f, O = 0.f;
            for (int cc = 0; cc < ns; cc++) {
                const float *pc = up + ((size_t)cc * g + h) * (D + 2);
                const float mc = __ldcg(pc + D);
                if (mc == -INFINITY) continue;
                const float f = exp2f(mc - M);
                L = fmaf(__ldcg(pc + D + 1), f, L);
                O = fmaf(__ldcg(pc + d), f, O);
            }
            p.out[((size_t)u * g + h) * D + d] = __half_as_ushort(__float2half_rn(O / L));
        }
        if (tid == 0) p.tickets[u] = 0;
    }
}

// ---------------------------------------------------------------------------------
size_t decode_smem_bytes_impl(int bits, bool kitty, int n_boost, int D, bool fast) {
    size_t w;
    if (fast) w = bits == 2 ? fast_warp_bytes<2>(kitty, n_boost) : fast_warp_bytes<4>(kitty, n_boost);
    else w = gen_warp_bytes(D);
    return (size_t)kWarps * w;
}

size_t decode_smem_bytes(int bits, bool kitty, int n_boost, int D) {
    return decode_smem_bytes_impl(bits, kitty, n_boost, D, true);
}

template <int BITS, bool KITTY, bool FAST, int DPL>
static cudaError_t launch_one(const DecodeParams &p, cudaStream_t st) {
    const size_t smem = decode_smem_bytes_impl(BITS, KITTY, p.n_boost, p.D, FAST);
    auto k = decode_kernel<BITS, KITTY, FAST, DPL>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)(p.C_f + p.C_g), kWarps * 32, smem, st>>>(p);
    return cudaGetLastError();
}

int decode_max_ctas_per_sm(int bits, bool kitty, int n_boost, int D, bool fast) {
    (void)bits;
    (void)kitty;
    (void)n_boost;
    (void)D;
    (void)fast;
    return 1;  // __launch_bounds__(256, 1) and ~170 KB of shared memory per CTA
}

cudaError_t launch_decode(const DecodeParams &p, bool fast, cudaStream_t st) {
    if (fast) {
        if (p.kitty) return launch_one<2, true, true, 4>(p, st);
        if (p.bits == 2) return launch_one<2, false, true, 4>(p, st);
        return launch_one<4, false, true, 4>(p, st);
    }
    switch (p.D) {
        case 64: return launch_one<2, false, false, 2>(p, st);
        case 128: return launch_one<2, false, false, 4>(p, st);
        case 256: return launch_one<2, false, false, 8>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvq
