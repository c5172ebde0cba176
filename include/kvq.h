/*
 * kvq.h -- C ABI of the GB300 low-bit KV-cache library (libkvq.so).
 *
 * The library quantizes the key/value cache of one attention layer into 2-, 4- or
 * 8-bit codes and runs single-query (and grouped-query) decode attention
 * directly on the packed codes.  It follows:
 *   - KIVI ("KV Cache 量化算子：KIVI"): min-max asymmetric quantization,
 *     scale = (max-min)/(2^b-1), keys per channel over groups of G tokens,
 *     values per token, 32/b codes packed per int32 (pack_tensor), an fp16
 *     residual of recent tokens, decode attention that unpacks in-kernel;
 *   - Kitty ("Kitty: Accurate and Efficient 2-Bit KV Cache Quantization with
 *     Dynamic Channel-wise Precision Boost"): fp16 sink tokens, key/value
 *     Q-buffers of G tokens, a value local window of R tokens, and per page the
 *     top n_boost key channels kept at INT4 as a low 2-bit plane plus a compact
 *     high 2-bit plane and a boost index (Sec. 3.2, Sec. 4.1, Algorithm 1);
 *   - BitDecoding (arXiv 2503.18773): attention softmax(q D(K')^T) D(V') on the
 *     packed cache, with the query heads of a GQA group processed together as
 *     one tensor-core tile (Sec. V-A, query transformation).
 *
 * Conventions for every entry point:
 *   - All buffers are caller-owned.  Pointers marked "device" are CUDA device
 *     memory of the current device, 16-byte aligned.  The library never
 *     allocates memory.
 *   - fp16 data is passed as uint16_t (IEEE binary16 bit patterns).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; the host-side lengths in kvq_cache are updated at
 *     enqueue time.  No entry point synchronizes the stream except
 *     kvq_read_status.
 *   - Return value: KVQ_OK or a negative kvq_status.  No entry point aborts or
 *     throws.  On an argument error nothing is enqueued and the cache is not
 *     modified.  KVQ_ERR_CUDA means a launch failed (cudaGetLastError).
 *   - Every sequence (b, h_kv) of a kvq_cache has the same length.  The paged
 *     cache (kvq_paged, below) holds sequences of different lengths.
 *   - Decode attention kernels (kvq_decode_attn, kvq_append_decode,
 *     kvq_decode_step_host, kvq_decode_attn_noalloc, kvq_paged_decode_attn) are
 *     launched as programmatic dependent launches: a kernel may start while the
 *     preceding kernel in the stream is still running, and reads nothing that kernel
 *     may write (q, new tokens, residuals, lengths, workspace) before that kernel has
 *     completed.  The one exception is the packed pages of a dense cache: the first
 *     copies of pages that no kvq_quant_pack_k / _v or kvq_flush_group call has
 *     written since the cache's previous decode attention may start early.  The
 *     library tracks those calls per cache (by its k_codes pointer), so a cache's
 *     packed buffers (k_codes, k_hi, k_bidx, k_meta, v_codes, v_meta) must be written
 *     only through the library's calls.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = -1,  /* bad shape, pointer, alignment or length       */
    KVQ_ERR_UNSUPPORTED = -2,  /* valid but not implemented (bits, D, g, ...)    */
    KVQ_ERR_CAPACITY = -3,     /* packed region or a buffer would overflow       */
    KVQ_ERR_WORKSPACE = -4,    /* workspace missing or too small                 */
    KVQ_ERR_CUDA = -5,         /* a CUDA launch or copy failed                    */
    KVQ_ERR_DEVICE = -6        /* a kernel reported an error in the status word   */
} kvq_status;

enum { KVQ_MODE_KIVI = 0, KVQ_MODE_KITTY = 1, KVQ_MODE_NVFP4 = 2 };

/* Device status bits (see kvq_read_status). */
enum { KVQ_DEV_TIMEOUT = 1, KVQ_DEV_BAD_STATE = 2 };

/* Shape of one layer's cache.
 *   B, H_q, H_kv, D : batch, query heads, key/value heads (H_q % H_kv == 0), head dim
 *   G               : group / page size in tokens (keys are quantized per channel over
 *                     G tokens; values per token over Gv = min(G, D) channels)
 *   bits            : key code width, 2, 4 or 8 (Kitty: 2; its boosted key channels
 *                     reach 4 bits)
 *   v_bits          : value code width, 2, 4 or 8; 0 means the same as bits (the
 *                     K4V2 / K2V4 variants of the Kitty notes, Sec. 3.1).  Every
 *                     pair of widths decodes on tensor-core tiles when D = 128,
 *                     H_q/H_kv <= 4 and G is a multiple of the tile (256/bits
 *                     tokens); other shapes on the CUDA-core path.
 *   S               : fp16 attention-sink tokens kept at the start (0 = none)
 *   R               : KIVI: fp16 residual capacity, a multiple of G, flushed as R/G
 *                     groups once full.  Kitty: the value local window.
 *   n_boost         : Kitty: key channels per page kept at INT4 (0..min(D,254)).
 *                     Must be 0 in KIVI mode.
 *   mode            : KVQ_MODE_KIVI, KVQ_MODE_KITTY or KVQ_MODE_NVFP4 (below)
 *   max_T           : packed-token capacity per sequence, a multiple of G
 *   rope            : 0: keys are attended as stored.  1: keys are stored before
 *                     the rotary position embedding and decode attention rotates
 *                     each one by its position (KVQuant notes, mechanism two:
 *                     pre-RoPE quantization); the query is passed already rotated.
 *                     Channel pair (2j, 2j+1) of the key at position t (its 0-based
 *                     index in [sink | packed | residual]) turns by
 *                     t * rope_base^(-2j/D).  KIVI mode, dense cache only.
 *   rope_base       : the RoPE base (10000 if 0)                                */
typedef struct {
    int32_t B, H_q, H_kv, D, G, bits;
    int32_t S, R, n_boost, mode;
    int32_t v_bits;
    int64_t max_T;
    int32_t rope;
    float rope_base;
} kvq_config;

/* Caller-owned device buffers and host-side lengths of one layer's cache.
 * Layouts (U = B*H_kv sequences, fpi = 32/bits codes per int32 for keys and
 * 32/v_bits for values, element j of a word at bit bits*j, least significant first):
 *   k_codes  int32 [U][max_T/fpi][D]     keys packed along tokens: row w holds the
 *                                        words of tokens fpi*w .. fpi*w+fpi-1, one per
 *                                        channel; the word of channel d sits at
 *                                        position d ^ (4 * (r mod 8)), r = w mod (G/fpi)
 *                                        its row within the page (16-byte chunks of a
 *                                        row permuted, so that a decode tile of eight
 *                                        rows is one contiguous copy whose tensor-core
 *                                        reads avoid shared-memory bank conflicts).
 *                                        Kitty: the low 2-bit plane (fpi = 16).
 *   k_hi     int32 [U][max_T/16][n_boost] Kitty: high 2 bits of the boosted channels,
 *                                        slot order; NULL if n_boost == 0.
 *   k_bidx   uint8 [U][max_T/G][D]       Kitty: channel -> slot, n_boost+1 if not
 *                                        boosted; NULL in KIVI mode.
 *   k_meta   fp16  [U][max_T/G][D][2]    (scale, min) per channel per group.
 *   v_codes  int32 [U][max_T/G][G/TV][D/fpi][TV]  values packed along channels: a
 *                                        page of G tokens is G/TV tiles of TV tokens
 *                                        (TV = 256/key bits -- 2 for Kitty -- when
 *                                        that divides G, else G); in a tile, row m holds
 *                                        the words of channels fpi*m .. fpi*m+fpi-1, and
 *                                        token j's word sits at position j ^ (4*(m mod 8))
 *                                        when TV is a multiple of 32, else at j.
 *   v_meta   fp16  [U][max_T][D/Gv][2]   (scale, min) per token per channel group.
 *   k_sink, v_sink  fp16 [U][S][D]       (NULL if S == 0)
 *   k_res    fp16  [U][cap_k][D]         cap_k = R (KIVI residual) or G (Kitty Q-buffer)
 *   v_res    fp16  [U][cap_v][D]         cap_v = R (KIVI residual) or G (Kitty Q-buffer)
 *   v_local  fp16  [U][R][D]             Kitty local window (ring, oldest at
 *                                        local_head); NULL in KIVI mode.
 *   status   int32 device word that kernels OR error bits into (may be NULL).
 * KVQ_MODE_NVFP4 (BitDecoding notes, Sec. V-D: Blackwell's native mxfp4 / nvfp4
 * formats; bits = 4, v_bits 0 or 4, G and D multiples of 16, G <= 256, R as KIVI):
 * pages hold e2m1 codes with an e4m3 scale per block of 16 elements along the
 * dimension each product contracts and an fp32 scale per page,
 *   S = amax(page) / 2688,  s = e4m3((amax(block) / 6) / S),  code = e2m1(x / (s S)),
 * rounded to nearest even with saturation, in fp32 IEEE arithmetic (S = 0 for an
 * all-zero page; a zero s S gives code 0).  Buffers in this mode:
 *   k_codes  uint8 [U][max_T/G][D/32][G][16]  per page, per 32-channel group, per token:
 *                                            byte i = channels 2i, 2i+1 (low nibble first)
 *   v_codes  uint8 [U][max_T/G][G/32][D][16]  per page, per 32-token group, per channel:
 *                                            byte m = tokens 2m, 2m+1 (low nibble first)
 *   k_meta  bytes [U][max_T/G][16 + G*D/16]  per page: fp32 S, 12 bytes padding, e4m3
 *                                            key scales [G][D/16] (16 channels of a token)
 *   v_meta  bytes [U][max_T/G][16 + G*D/16]  the same with value scales [G/16][D]
 *                                            (16 tokens of a channel)
 *   k_hi, k_bidx, v_local unused.  Decode attention runs on tensor-core tiles of 64
 *   tokens (each code byte converted to an exact f16x2 operand, fp32 accumulation) when
 *   D = 128, H_q/H_kv <= 4, rope = 0 and G is a power-of-two multiple of 64; other
 *   shapes run on the CUDA-core path.
 * Lengths: n_sink sink tokens, T_k / T_v packed key / value tokens, n_kres keys in
 * k_res, n_vres values in v_res, n_local values in v_local.  A fresh cache has all
 * lengths 0.  Logical token order: keys [sink | packed | k_res], values
 * [sink | packed | v_res | v_local (oldest first)]. */
typedef struct {
    int32_t *k_codes;
    int32_t *k_hi;
    uint8_t *k_bidx;
    uint16_t *k_meta;
    int32_t *v_codes;
    uint16_t *v_meta;
    uint16_t *k_sink, *v_sink;
    uint16_t *k_res, *v_res, *v_local;
    int32_t *status;
    int64_t n_sink, T_k, n_kres, T_v, n_vres, n_local, local_head;
} kvq_cache;

/* Text for a kvq_status value (static string). */
const char *kvq_status_str(int status);

/* Validates a configuration.  KVQ_OK, KVQ_ERR_INVALID_ARG (H_q % H_kv, G % fpi,
 * D % fpi, Gv | D, R % G (KIVI), n_boost range, max_T % G, non-positive sizes) or
 * KVQ_ERR_UNSUPPORTED (bits or v_bits not 2/4/8, Kitty with bits != 2, D not 64,
 * 128 or 256, more than 8 query heads per KV head, rope with Kitty; rope not 0/1 or
 * a negative or non-finite rope_base is KVQ_ERR_INVALID_ARG). */
int kvq_config_check(const kvq_config *cfg);

/* Byte size of each cache buffer for cfg: which = 0 k_codes, 1 k_hi, 2 k_bidx,
 * 3 k_meta, 4 v_codes, 5 v_meta, 6 k_sink (= v_sink), 7 k_res, 8 v_res, 9 v_local.
 * Returns 0 for a buffer the mode does not use or for an invalid cfg. */
size_t kvq_buffer_bytes(const kvq_config *cfg, int which);

/* Prefill of the keys (KIVI page, Step 3: after prefill the cache is split into
 * a low-bit part and an fp16 residual).  k: device fp16 [B][H_kv][L0][D].
 * The first min(S, L0) tokens go to k_sink; the next floor((L0-n_sink)/G)*G are
 * quantized per channel in groups of G tokens into k_codes/k_meta (Kitty: the
 * top n_boost channels of each page by sum |k| at 4 bits, the rest at 2); the
 * remainder (< G) is copied to k_res.  Requires an empty key cache (T_k == 0,
 * n_kres == 0) and 1 <= L0.  KVQ_ERR_CAPACITY if the packed part exceeds max_T. */
int kvq_quant_pack_k(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k,
                     int64_t L0, void *stream);

/* Prefill of the values.  v: device fp16 [B][H_kv][L0][D].  Sink as for keys.
 * KIVI: floor((L0-n_sink)/G)*G tokens quantized per token in groups of Gv
 * channels, the rest copied to v_res.  Kitty: the last min(R, L0-n_sink) tokens go
 * to the local window; of the older ones floor(./G)*G are quantized and the rest
 * copied to the value Q-buffer (v_res).  Requires an empty value cache. */
int kvq_quant_pack_v(const kvq_config *cfg, kvq_cache *cache, const uint16_t *v,
                     int64_t L0, void *stream);

/* Stage (1) of the Kitty decode pipeline (Sec. 4.3): insert one new token.
 * k_new, v_new: device fp16 [B][H_kv][D].  While the sink is not full the token
 * goes to the sink.  Otherwise the key goes to k_res; the value goes to v_res
 * (KIVI) or to the local window, whose oldest value moves to the value Q-buffer
 * once the window is full (Kitty).  KVQ_ERR_CAPACITY if a destination buffer is
 * full (call kvq_flush_group first). */
int kvq_append_token(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k_new,
                     const uint16_t *v_new, void *stream);

/* Stage (3): quantize every full buffer.  A key buffer holding cap_k tokens is
 * packed as cap_k/G new groups at the end of the packed keys and emptied; the same
 * for the value buffer.  *flushed_k / *flushed_v (may be NULL) receive 1 if that
 * buffer was flushed, else 0.  KVQ_ERR_CAPACITY if max_T would be exceeded. */
int kvq_flush_group(const kvq_config *cfg, kvq_cache *cache, int *flushed_k,
                    int *flushed_v, void *stream);

/* Workspace bytes kvq_decode_attn needs for cfg (split-T partials, one counter per
 * sequence and the status word).  The workspace must be zero-filled before its
 * first use (kvq_workspace_init); every call leaves its counters at zero again. */
size_t kvq_decode_attn_workspace_bytes(const kvq_config *cfg);

/* Zero-fills a workspace (cudaMemsetAsync on stream). */
int kvq_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Stage (2): decode attention for one query token per sequence,
 *   out[b][h] = softmax_t( q[b][h] . K_t / sqrt(D) ) . V_t
 * over every cached token (sink, packed, buffers), with packed keys and values
 * dequantized (code*scale+min) on the fly in registers; query head h reads key /
 * value head h / (H_q/H_kv).  q: device fp16 [B][H_q][D]; out: device fp16
 * [B][H_q][D]; ws: device workspace of ws_bytes >= kvq_decode_attn_workspace_bytes.
 * Accumulation is fp32 (fp16 tensor-core operands for the packed tiles).
 * KVQ_ERR_INVALID_ARG if the cache is empty or its key and value lengths differ. */
int kvq_decode_attn(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                    uint16_t *out, void *ws, size_t ws_bytes, void *stream);

/* Bytes of the device staging buffer of kvq_decode_step_host for cfg (0 if cfg is
 * invalid): q, k_new, v_new and out of one step, each 256-byte aligned. */
size_t kvq_step_io_bytes(const kvq_config *cfg);

/* One whole decode step from host memory: the three stages of the decode pipeline in
 * order (Kitty Sec. 4.3), with the transfers in and out.
 *   1. k_new, v_new (host fp16 [B][H_kv][D]) and q (host fp16 [B][H_q][D]) reach the
 *      device;
 *   2. kvq_append_decode, then kvq_flush_group;
 *   3. the attention output reaches out (host fp16 [B][H_q][D]).
 * When all four host buffers are page-locked memory mapped into the device's address
 * space (cudaHostAlloc / cudaHostRegister; with unified addressing every page-locked
 * allocation is), the kernels read the inputs and write the output in place over the
 * host link (plain loads and stores) and io is not touched.  Otherwise there is one
 * cudaMemcpyAsync per buffer through io, in and out (asynchronous only for page-locked
 * memory).
 * Everything is enqueued on `stream` and nothing is synchronized: out holds the result
 * once the stream has passed this point (cudaStreamSynchronize or an event), and the
 * host inputs must stay unchanged until then.
 * io: device buffer of io_bytes >= kvq_step_io_bytes(cfg), 256-byte aligned, owned by
 * the caller (KVQ_ERR_WORKSPACE if too small); ws, ws_bytes as for kvq_decode_attn;
 * flushed_k, flushed_v as for kvq_flush_group.
 * Returns KVQ_OK or the status of the first stage that fails; the stages before it
 * have taken effect, as if called one by one (a refused append leaves the cache as it
 * was; only the copies into io, if the buffers are not mapped, were enqueued). */
int kvq_decode_step_host(const kvq_config *cfg, kvq_cache *cache, const uint16_t *q,
                         const uint16_t *k_new, const uint16_t *v_new, uint16_t *out, void *io,
                         size_t io_bytes, void *ws, size_t ws_bytes, int *flushed_k,
                         int *flushed_v, void *stream);

/* kvq_decode_step_host for page-locked, mapped host buffers, returning once the
 * output is in out: a blocking decode step (Kitty Sec. 4.3 stages 1-3 with the host
 * transfers).
 * done: a 4-byte-aligned unsigned int in page-locked host memory mapped into the
 * device's address space, owned by the caller, used as a completion word: the call
 * sets it to 0 before it launches; the decode kernel counts the sequences whose
 * output stores it has made visible at system scope (in the workspace) and, when the
 * count reaches B * H_kv, stores B * H_kv to *done (release, system scope); the call
 * spins until it reads that value (after 200 ms it synchronizes the stream instead).
 * When it returns KVQ_OK, out holds the result; a flush enqueued by the step may still
 * be running on `stream`.
 * KVQ_ERR_INVALID_ARG if any of q, k_new, v_new, out, done is missing or not mapped
 * page-locked memory, or a buffer is not 16-byte aligned (done: 4); KVQ_ERR_DEVICE if
 * the stream completed without *done reaching B * H_kv.  Other errors as for
 * kvq_decode_step_host (no io buffer is needed). */
int kvq_decode_step_host_wait(const kvq_config *cfg, kvq_cache *cache, const uint16_t *q,
                              const uint16_t *k_new, const uint16_t *v_new, uint16_t *out,
                              unsigned int *done, void *ws, size_t ws_bytes, int *flushed_k,
                              int *flushed_v, void *stream);

/* Self-test of the kernels' bounded waits (no counterpart on the pages): one warp
 * waits, through the same bounded mbarrier wait the decode kernels use, on a barrier
 * that nothing completes.  At the kernels' bound (4e9 SM clock cycles, about 2 s at
 * 2 GHz) the wait gives up, ORs KVQ_DEV_TIMEOUT into *status (device int32, 4-byte
 * aligned) and the kernel returns; the context stays usable.  Enqueued on `stream`.
 * KVQ_ERR_INVALID_ARG for a missing or misaligned status word. */
int kvq_selftest_wait_timeout(int32_t *status, void *stream);

/* Stages (1) and (2) together: kvq_append_token(k_new, v_new), then kvq_decode_attn(q,
 * out), with the same arguments, layouts, results and errors.  Where the token goes to
 * the key and value residuals of a KIVI cache (sink full) and the packed-tile path
 * serves the attention, both run in one launch: the warp that owns the 16-token tile
 * holding the new token reads its key and value rows from k_new and v_new (plain loads)
 * and stores them into the residuals, from where that tile's copies read them.  No other
 * copy of the launch reads those rows.  Otherwise the two calls run one
 * after the other (then, if the attention stage fails, the append has taken effect).
 * *fused (may be NULL) receives 1 if one launch did both, else 0. */
int kvq_append_decode(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k_new,
                      const uint16_t *v_new, const uint16_t *q, uint16_t *out, void *ws,
                      size_t ws_bytes, int *fused, void *stream);

/* Size of the library's own decode scratch region (16 MiB per device). */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Decode attention exactly as kvq_decode_attn, but without a caller workspace: it
 * uses a fixed KVQ_NOALLOC_SCRATCH_BYTES region that the library module itself
 * reserves on each device when its code is loaded.  The pages have no counterpart;
 * this exists for callers that cannot hand out device memory in their decode step,
 * for example an inference engine whose memory pool is already fully reserved for
 * weights and KV pages, or a plugin called from a host runtime that forbids
 * allocations inside its step callback.  Nothing here allocates.
 *   - The first call on a device (with that device current) looks the region up;
 *     that may load the library's module onto the device, so the first call is
 *     refused with KVQ_ERR_INVALID_ARG while `stream` is capturing.  Make it before
 *     any stream capture.
 *   - Every call enqueues on `stream` a zero fill of the region's first bytes (its
 *     per-sequence counters, whose extent depends on cfg), then the decode kernel.
 *     Calls with different configurations may therefore follow one another.
 *   - Configurations whose workspace (kvq_decode_attn_workspace_bytes) exceeds the
 *     region are refused with KVQ_ERR_WORKSPACE; nothing is enqueued.  Argument errors
 *     enqueue nothing; a later refusal (KVQ_ERR_UNSUPPORTED from the scheduler) may
 *     leave the zero fill enqueued, which touches only the library's own region.
 *   - The region is shared by all calls on a device: two calls whose kernels may
 *     overlap (different streams, or different host threads without ordering)
 *     race on it and give wrong results.  Serialize them, e.g. on one stream.
 *   - cache->status must be set (else KVQ_ERR_INVALID_ARG): the kernels' device error
 *     bits go there, and kvq_read_status(cache, NULL, ...) returns and clears them.
 * Other arguments, layouts, results and errors as for kvq_decode_attn. */
int kvq_decode_attn_noalloc(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                            uint16_t *out, void *stream);

/* ---------------------------------------------------------------------------------
 * Paged cache with per-sequence lengths (Kitty Sec. 4.1 "page-centric memory layout":
 * every quantization group of G tokens is a page, stored apart from the fp16 sink and
 * residual buffers, after PagedAttention; the KIVI notes name PagedAttention as the
 * way to cut a cache into fixed blocks reached through a mapping table).
 *
 * Physical page p (0 <= p < n_pages) holds one group of G tokens of all H_kv heads of
 * one sequence.  The page pools use the page-major layouts of kvq_cache with the page
 * index (u * max_T/G + logical page) replaced by (p * H_kv + h):
 *   k_codes  int32 [n_pages][H_kv][G/fpi_k][D]        (rows arranged as in kvq_cache)
 *   k_meta   fp16  [n_pages][H_kv][D][2]
 *   v_codes  int32 [n_pages][H_kv][G/TV][D/fpi_v][TV]  (tiles arranged as in kvq_cache)
 *   v_meta   fp16  [n_pages][H_kv][G][D/Gv][2]
 * page_table int32 [B][max_T/G] (device) maps logical page j of sequence b to its
 * physical page.  The caller owns the pool and the table and chooses the pages: before
 * kvq_paged_prefill(b, L0) row b must map the packed pages of the prefill, and before
 * kvq_paged_flush every sequence that kvq_paged_flush_plan lists must map its next R/G
 * logical pages.  Entries must be valid page ids; a page must not be mapped twice.
 * Per-sequence fp16 buffers keep the kvq_cache layouts ([U][S][D] sink, [U][R][D]
 * residual; U = B*H_kv, unit b*H_kv + h).
 * lens (device) and lens_host (host) are int32 [B][4] = {n_sink, T, n_res, active}:
 * sink tokens, packed tokens (keys and values alike), residual tokens, and 1 if the
 * batch slot holds a sequence.  The library keeps both; the caller only allocates
 * them and calls kvq_paged_init once.  Sequence b's logical tokens are
 * [sink | packed pages | residual].
 * Supported: KIVI mode, any widths, D = 128, H_q/H_kv <= 4, G a multiple of the tile
 * (256/bits tokens) and a power of two, B <= KVQ_PAGED_MAX_B, rope = 0.
 * --------------------------------------------------------------------------------- */
#define KVQ_PAGED_MAX_B 512

typedef struct {
    int32_t *k_codes;
    uint16_t *k_meta;
    int32_t *v_codes;
    uint16_t *v_meta;
    int64_t n_pages;
    const int32_t *page_table;
    uint16_t *k_sink, *v_sink;
    uint16_t *k_res, *v_res;
    int32_t *lens;
    int32_t *lens_host;
    int32_t *status;
} kvq_paged;

/* Byte size of a paged buffer: which = 0 k_codes, 3 k_meta, 4 v_codes, 5 v_meta
 * (pools of n_pages pages), 6 k_sink (= v_sink), 7 k_res, 8 v_res, 10 lens (= lens_host),
 * 11 page_table.  0 for an unused buffer or an unsupported cfg. */
size_t kvq_paged_bytes(const kvq_config *cfg, int64_t n_pages, int which);

/* Marks every batch slot empty (host and device lengths; cudaMemsetAsync on stream). */
int kvq_paged_init(const kvq_config *cfg, kvq_paged *pc, void *stream);

/* Prefill of batch slot b, which must be empty: k, v device fp16 [H_kv][L0][D].  The
 * first min(S, L0) tokens go to the sink, the next floor((L0-n_sink)/G)*G are
 * quantized (keys per channel, values per token) into the physical pages that
 * page_table row b maps for logical pages 0.., and the rest (< G) go to the residual
 * (KIVI Step 3).  KVQ_ERR_CAPACITY if the packed part exceeds max_T. */
int kvq_paged_prefill(const kvq_config *cfg, kvq_paged *pc, int b, const uint16_t *k,
                      const uint16_t *v, int64_t L0, void *stream);

/* One new token for every active sequence: k_new, v_new device fp16 [B][H_kv][D]
 * (rows of empty slots are ignored).  Into the sink while it is not full, else into
 * the residual.  KVQ_ERR_CAPACITY if an active sequence's residual is full (flush
 * first). */
int kvq_paged_append(const kvq_config *cfg, kvq_paged *pc, const uint16_t *k_new,
                     const uint16_t *v_new, void *stream);

/* Host only: the sequences whose residual is full, ascending, into seqs (room for B);
 * *n their count.  Sequence b needs logical pages [T_b/G, T_b/G + R/G) mapped before
 * kvq_paged_flush. */
int kvq_paged_flush_plan(const kvq_config *cfg, const kvq_paged *pc, int32_t *seqs, int *n);

/* Packs the full residual of every sequence kvq_paged_flush_plan lists into its next
 * R/G pages and empties it.  *n_flushed (may be NULL): the number of sequences.
 * KVQ_ERR_CAPACITY if a sequence would exceed max_T. */
int kvq_paged_flush(const kvq_config *cfg, kvq_paged *pc, int *n_flushed, void *stream);

/* Empties batch slot b (its pages may then be reused by the caller). */
int kvq_paged_release(const kvq_config *cfg, kvq_paged *pc, int b, void *stream);

/* Workspace bytes kvq_paged_decode_attn needs (zero-filled once, kvq_workspace_init). */
size_t kvq_paged_workspace_bytes(const kvq_config *cfg);

/* Decode attention, as kvq_decode_attn, for every active sequence over its own
 * length: q, out device fp16 [B][H_q][D]; rows of empty slots are not written. */
int kvq_paged_decode_attn(const kvq_config *cfg, const kvq_paged *pc, const uint16_t *q,
                          uint16_t *out, void *ws, size_t ws_bytes, void *stream);

/* As kvq_read_status, for the workspace status word and pc->status. */
int kvq_paged_read_status(const kvq_paged *pc, void *ws, int32_t *dev_status, void *stream);

/* Synchronizes `stream`, then returns in *dev_status the OR of the error bits the
 * kernels wrote into the workspace status word and into cache->status (if cache is
 * not NULL and its status pointer is set), and clears both.  KVQ_ERR_DEVICE if any
 * bit was set, else KVQ_OK. */
int kvq_read_status(const kvq_cache *cache, void *ws, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
