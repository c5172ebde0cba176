// kvq_internal.h -- kernel parameter blocks and launchers shared by the libkvq
// translation units (not part of the public ABI; see include/kvq.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// In-page arrangement of the packed words (KIVI codes and Kitty's low plane; NVFP4
// pages have their own layout).  The words themselves are pack_tensor's; only their
// order inside a page is chosen so that a decode tile arrives with one contiguous bulk
// copy and its ldmatrix reads are free of shared-memory bank conflicts:
//   keys:   a page is G/fpi word rows of D words; the word of channel d in row r
//           (0-based within the page) sits at kword_pos(d, r) -- the 16-byte chunks of
//           each row are permuted by XOR with r mod 8.
//   values: a page is G/TV tiles of TV tokens, each [D/fpi rows][TV words]; the word of
//           token j in row b sits at vword_pos(j, b, TV).  TV is the token count of a
//           decode tile, 256 / key bits (eight key word rows), when it divides G, else G.
__host__ __device__ __forceinline__ int kword_pos(int d, int r) { return d ^ ((r & 7) << 2); }
__host__ __device__ __forceinline__ int vword_pos(int j, int b, int TV) {
    return (TV & 31) ? j : j ^ ((b & 7) << 2);
}
__host__ __device__ __forceinline__ int v_tile_tokens(int kbits, int G) {
    const int t = 256 / kbits;
    return G % t == 0 ? t : G;
}

// Destination of the quant kernels' pages.  Dense (ptab null): grid unit u writes
// page u * max_T/G + pg0 + j.  Paged: grid unit i is head h = i % H_kv of listed
// sequence b = seq[i / H_kv]; its page j goes to physical page
// ptab[b * ptab_stride + lp0[i / H_kv] + j], page index (that page) * H_kv + h.  Its
// source unit is b * H_kv + h (src_by_seq) or h (a one-sequence source).
constexpr int kMaxListSeq = 256;
// A table entry outside [0, n_pages) is replaced by page 0 and sets the bad-state bit.
struct PageMap {
    const int32_t *ptab;
    int ptab_stride, H_kv, n_seq, src_by_seq;
    int64_t n_pages;
    int32_t *status;
    int32_t *lens;         // keys of a paged flush: lens[b] gets T = (lp0 + pages) * G, n_res = 0
    int16_t seq[kMaxListSeq];
    int32_t lp0[kMaxListSeq];
};

// fp16 rows copied by extra CTAs of a quant launch (the parts of a prefill that stay
// fp16: sink, residual, local window), so that a prefill side is one launch.  Dense
// caches only: row i of unit u goes from src[u * src_rows + src_r0 + i] to
// dst[u * dst_rows + dst_r0 + i] (rows of D halves, 16-byte aligned).
struct RowCopy {
    const uint16_t *src;
    uint16_t *dst;
    int64_t src_rows, src_r0, dst_rows, dst_r0, n_rows;
};
constexpr int kMaxRowCopies = 3;
struct RowCopies {
    RowCopy c[kMaxRowCopies];
    int n;                 // copies in c (0: none)
    int cols;              // CTAs per unit that copy (set by the launcher)
    int64_t x0;            // grid column of the first of them (set by the launcher)
};

struct QuantKParams {
    const uint16_t *src;   // fp16 [U][*][D]
    int64_t src_ustride;   // elements between sequences
    int64_t src_t0;        // first source row
    int64_t n_pages;       // pages of G tokens to quantize
    int64_t pg0;           // destination page index of the first one
    int64_t max_T;
    int U, D, G, n_boost, slices;
    int32_t *k_codes, *k_hi;
    uint8_t *k_bidx;
    uint16_t *k_meta;
    int32_t *status;       // device status word (may be null)
    RowCopies rc;
    PageMap pm;
};

struct QuantVParams {
    const uint16_t *src;
    int64_t src_ustride, src_t0;
    int64_t n_tok;         // tokens to quantize (multiple of G)
    int64_t tok0;          // destination packed-token index of the first one (multiple of G)
    int64_t max_T;
    int U, D, G, Gv;
    int TV;                // tokens per value tile of a page (v_tile_tokens)
    int32_t *v_codes;
    uint16_t *v_meta;
    int32_t *status;       // device status word (may be null)
    RowCopies rc;
    PageMap pm;
};

// NVFP4 pages: one CTA per page of G tokens (fp16 [G][D] at src rows src_t0 + j G of
// unit u) -> codes uint8 [U][max_T][D/2] (token-major) and a page record of `ms`
// bytes at meta + (u * max_T/G + pg0 + j) * ms: fp32 scale S, 12 bytes of padding,
// then e4m3 block scales ([G][D/16] for keys, [G/16][D] for values).
struct QuantNvParams {
    const uint16_t *src;
    int64_t src_ustride, src_t0;
    int64_t n_pages, pg0, max_T;
    int U, D, G, ms;
    uint8_t *codes, *meta;
};

struct CopyRowsParams {
    const uint16_t *src;
    uint16_t *dst;
    int64_t src_rows, src_r0, dst_rows, dst_r0, n_rows;
    int U, D;
};

struct AppendParams {
    const uint16_t *k_new, *v_new;
    uint16_t *k_dst, *v_dst, *v_evict;
    int64_t k_rows, k_row, v_rows, v_row, evict_rows, evict_row;  // evict_row < 0: none
    int U, D;
};

// Paged append: one CTA per batch slot; the rows follow the slot's device lengths,
// which the CTA then advances.
struct PagedAppendParams {
    const uint16_t *k_new, *v_new;
    uint16_t *k_sink, *v_sink, *k_res, *v_res;
    int32_t *lens;         // [B][4] n_sink, T, n_res, active
    int32_t *status;       // a full residual sets the bad-state bit (the host checks first)
    int B, H_kv, D, S, R;
};

// Writes lens[b] = {v0, v1, v2, v3} (prefill and release of a batch slot).
struct SetLensParams {
    int32_t *lens;
    int b, v0, v1, v2, v3;
};

// Decode attention schedule.  Work items of one sequence:
//   fast tiles: TOK tokens whose keys and values are both packed (tensor cores);
//   mini tiles: 16 tokens whose values are fp16 -- sink, residual / Q-buffer, local
//               window -- with fp16 keys or a packed key block (tensor cores);
//   generic chunks: any token, CUDA cores (only for shapes the tile paths do not
//               cover; then there are no fast or mini items).
// Each kind has a pool of CTAs whose warps cut the sequence-major list of all
// sequences' items into equal ranges; a range touches at most two sequences.
// A CTA merges its warps' partial softmax states per sequence into one slot; the
// CTA that completes a sequence's item count combines the slots.
struct DecodeParams {
    // shape
    int B, H_kv, g, D, G, bits, vbits, Gv, n_boost, kitty;  // bits: keys, vbits: values
    int v_tile;            // tokens per value tile of a page (v_tile_tokens)
    int S_cap, cap_k, cap_v, R_local;
    int64_t max_T;
    int rope;              // keys stored before RoPE: rotate key t by t * theta_j
    float rope_base;
    int nvfp4, nv_kms, nv_vms;  // NVFP4 pages (CUDA-core path): page record bytes of keys, values
    // lengths
    int64_t n_sink, T_k, n_kres, T_v, n_vres, n_local, local_head, L;
    // buffers
    const int32_t *k_codes, *k_hi;
    const uint8_t *k_bidx;
    const uint16_t *k_meta;
    const int32_t *v_codes;
    const uint16_t *v_meta;
    const uint16_t *k_sink, *v_sink, *k_res, *v_res, *v_local;
    const uint16_t *q;
    uint16_t *out;
    // appended in the same launch (dense KIVI caches, mini tiles): the new token's key
    // and value rows [U][D]; it is the last logical token, and the warp whose mini
    // tile holds it stores it into k_res / v_res.  Null: no append.
    const uint16_t *k_new, *v_new;
    float *partials;       // [U][max_slots][g][D + 4]
    int32_t *slot_ctr;     // [U] slots taken (paged caches; zero between calls)
    unsigned long long *item_ctr;  // [U] items merged << 32 | CTAs arrived (zero between calls)
    int32_t *status;       // workspace status word
    // blocking host step (null: none): done is a host word that receives U, at system
    // scope, once every sequence's output is visible there; done_ctr counts the
    // combined sequences (workspace, zero between calls)
    unsigned int *done, *done_ctr;
    // schedule
    int U, wpc;            // sequences, warps per CTA
    int C_f, C_m, C_g;     // CTAs of the fast, mini and generic pools (grid: mini, fast; or generic)
    int n_gc, max_slots;
    int n_items;           // items per sequence over all pools
    int W_f, qN_f, rN_f;   // fast pool: warps, N_f / W_f, N_f % W_f
    int W_m, qN_m, rN_m;   // mini pool: the same
    int tpp_shift, g_shift;  // log2(packed tiles per page), log2(G) (tile paths only)
    int64_t n_fast, N_f;   // fast tiles per sequence, in all
    int64_t n_mini, N_m;   // mini tiles per sequence, in all
    int64_t n_gen;         // generic tokens per sequence
    int64_t gen_chunk;     // tokens per generic chunk (multiple of 32)
    // paged cache (tile paths, KIVI): page table and per-sequence lengths.  Items of
    // sequence b in a pool are laid out b-major like the dense ones, each sequence with
    // its own count; a unit range may then cross several sequences.  Segments that are
    // neither the first nor the last of a range hold a whole sequence's items of that
    // pool and are published by their unit alone.
    const int32_t *ptab;   // [B][ptab_stride] physical page of logical page j (null: dense)
    int ptab_stride;
    int64_t n_pages;       // pool size; an entry outside [0, n_pages) reads page 0 and sets a status bit
    const int32_t *lens;   // [B][4] n_sink, T, n_res, active (null: the lengths above)
    int32_t *seq_slots;    // [U][smax] partial slot ids of each sequence (paged)
    int smax;              // slot ids per sequence
    int mid_base;          // first slot id of the middle segments: pool * U + u above it
    // Packed tiles [0, early_tiles) of every sequence lie in pages that no prefill or
    // flush has written since the cache's previous decode: their copies may start
    // before the preceding kernel in the stream has completed (dense caches).
    int early_tiles;
};

constexpr int kMaxWarps = 8;

cudaError_t launch_quant_k(const QuantKParams &p, int bits, bool kitty, cudaStream_t st);
cudaError_t launch_quant_v(const QuantVParams &p, int bits, cudaStream_t st);
cudaError_t launch_nvfp4(const QuantNvParams &p, bool values, cudaStream_t st);
cudaError_t launch_copy_rows(const CopyRowsParams &p, cudaStream_t st);
cudaError_t launch_append(const AppendParams &p, cudaStream_t st);
cudaError_t launch_paged_append(const PagedAppendParams &p, cudaStream_t st);
cudaError_t launch_set_lens(const SetLensParams &p, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams &p, bool fast, cudaStream_t st);
cudaError_t launch_decode_paged(const DecodeParams &p, cudaStream_t st);  // p.lens set
cudaError_t launch_decode_rope(const DecodeParams &p, bool fast, cudaStream_t st);  // p.rope set
cudaError_t launch_decode_nvfp4(const DecodeParams &p, cudaStream_t st);            // NVFP4 tiles
size_t decode_smem_bytes(int bits, int vbits, bool kitty, int n_boost, int D, bool fast);
int decode_warps_per_cta(int bits, int vbits, bool kitty, int n_boost, bool fast);

}  // namespace kvq
