/*
 * csa.h - C ABI of the GB300 (sm_103a) compressed sparse attention library.
 *
 * Compressed sparse attention (CSA) as in DeepSeek-V4 / V4.1: a gated
 * compressor pools every `ratio` raw KV rows into one compressed entry, an
 * INT8 "lightning" indexer scores the compressed entries of every query row
 * and keeps the top-k, and shared-KV sparse attention runs over the selected
 * entries plus a 128-token causal raw window with a per-head sink logit.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensors are caller-owned DEVICE pointers, dense and row-major in the
 *   shapes given below, except the paged pools, which take explicit strides
 *   (see "Pool strides").  The library keeps no
 *   pointer after a call returns and allocates no device memory: scratch is
 *   the caller's `workspace`.  Calling with workspace == NULL only stores the
 *   number of bytes the call needs in `workspace_bytes` and returns CSA_OK.
 * - Paged pools hold 128-row pages ([pages, 128, width]).  A block table row
 *   b maps request b's logical page j to a physical page; entries of pages a
 *   call never reads may be -1 ("DeepSeek V4-Flash, MTP point", "Deployment
 *   configuration": 128-token pages; "DeepSeek V4.1 Flash", compressed KV and
 *   index keys share one block table).
 * - BF16 tensors are passed as `const void*` (IEEE bfloat16 bit patterns).
 * - RoPE tables are FP32 half-width [rope_cap, 32] cos/sin tables; the last 64
 *   channels of a vector are rotated by adjacent pairs (x[2i], x[2i+1]) ->
 *   (x[2i]c - x[2i+1]s, x[2i]s + x[2i+1]c) at a position's table row; a
 *   negative position means the identity ("DeepSeek V4.1 Flash",
 *   "Serving-owned full RoPE tables").  A position >= rope_cap also gives the
 *   identity and raises CSA_DEV_POS_GE_CAP.
 * - Every call is asynchronous on `stream` (a cudaStream_t) and never
 *   synchronises.  The return value reports host-side argument checks and
 *   launch errors only.  Data errors found on the device (bad page, bad
 *   position, bad index) are OR-ed into the optional caller word
 *   `*status_dev` (CSA_DEV_* bits) and the offending element is skipped; the
 *   device never traps.
 * - A row with row_req[t] < 0 is padding: it is neither read nor written
 *   ("DeepSeek-V4.1 native paged runtime": a padding token's batch id is -1).
 * - Every args struct starts with `struct_size`; set it to sizeof(struct).
 * - Pool strides.  A paged pool [pages, 128, width] may be a view into a
 *   larger allocation (a cache holding several layers, or several fields
 *   per row): `*_page_stride` is the byte distance between consecutive
 *   pages and `*_row_stride` between consecutive rows of a page; a row's
 *   own bytes are contiguous.  0 means dense (row stride = the row's bytes,
 *   page stride = 128 row strides); a struct_size that ends before the
 *   fields means dense.  Strides must be multiples of 16 bytes, a row
 *   stride at least the row's bytes and a page stride at least 128 row
 *   strides; otherwise CSA_ERR_INVALID_ARG.  The low-bit cache formats take
 *   dense pools only (non-zero strides: CSA_ERR_UNSUPPORTED).
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_API __attribute__((visibility("default")))

typedef void *csa_stream_t; /* a cudaStream_t */

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size or a misaligned pointer */
  CSA_ERR_UNSUPPORTED = 2, /* a shape this library does not implement */
  CSA_ERR_CUDA = 3,        /* a CUDA launch or runtime error */
  CSA_ERR_TIMEOUT = 4      /* a bounded wait gave up (device waits report CSA_DEV_TIMEOUT) */
} csa_status_t;

/* bits OR-ed into *status_dev by the kernels */
#define CSA_DEV_BAD_BLOCK 0x1u  /* block-table entry < 0 or >= pool pages on a page that is read */
#define CSA_DEV_BAD_POS 0x2u    /* a window position >= kv_len, or a bad request id */
#define CSA_DEV_BAD_INDEX 0x4u  /* a top-k entry outside [0, visible count) */
#define CSA_DEV_POS_GE_CAP 0x8u /* a position >= rope_cap (rotation skipped) */
#define CSA_DEV_TIMEOUT 0x10u   /* a bounded device wait gave up; the call's outputs are invalid */

#define CSA_BLOCK 128    /* rows per page */
#define CSA_ROPE_DIM 64  /* rotated channels (the last 64) */
#define CSA_WINDOW 128   /* raw window, self included */
#define CSA_MAX_TOPK 2048

/* Publication formats of csa_compress (csa_out_mode_t) and cache formats
 * read by csa_index_topk and the attention calls (csa_cache_fmt_t).  The
 * low-bit formats are the production cache ABI of "DeepSeek V4.1 Flash":
 *  - FP4_E4M3: packed E2M1 (two channels per byte, channel 2i in the low
 *    nibble), one E4M3 scale byte per 16 channels (compressed KV).  A row of
 *    512 channels is 256 code bytes plus 32 scale bytes.
 *  - FP4_E8M0: packed E2M1, one E8M0 scale byte (2^(byte-127)) per 32
 *    channels (index keys: 64 code bytes plus 4 scale bytes per 128-dim key).
 *  - MXFP8: one E4M3 byte per channel, one E8M0 scale byte per 32 channels
 *    (window KV: 512 code bytes plus 16 scale bytes per row; the FP8 index
 *    plane, read as the same layout: 128 code bytes plus 4 scale bytes per
 *    key).
 * A value is its code times its group's scale.  Publication (readings; the
 * pages give the formats only): FP4_E8M0 takes for each group the smallest
 * 2^e with 6 * 2^e >= amax (amax = 0: e = -127), FP4_E4M3 the E4M3 value
 * nearest to amax / 6 (saturating at 448); codes are the nearest E2M1 of
 * value / scale (ties to the even code, saturating at 6, the sign bit set for
 * negative values), quotients taken in FP32; a zero E4M3 scale gives zero
 * codes.  MXFP8 takes the smallest 2^e with 448 * 2^e >= amax and codes the
 * nearest E4M3 of value / 2^e (ties to the even code).  Code pools are uint8 [n_blocks, 128, code bytes per row] and scale
 * pools uint8 [n_blocks, 128, groups per row], both through the block table
 * of the pool they replace. */
typedef enum {
  CSA_OUT_BF16 = 0,
  CSA_OUT_INT8 = 1,
  CSA_OUT_FP4_E4M3 = 2, /* codes into cmp_pool, scales into scale_pool */
  CSA_OUT_FP4_E8M0 = 3, /* codes into cmp_pool, scales into scale_pool */
  CSA_OUT_MXFP8 = 4     /* codes (one byte a channel) into cmp_pool, scales into scale_pool */
} csa_out_mode_t;
typedef enum {
  CSA_FMT_BF16 = 0,     /* attention pools: bf16 rows */
  CSA_FMT_INT8 = 1,     /* index keys: int8 codes, f32 scale per row */
  CSA_FMT_FP4_E4M3 = 2, /* compressed KV */
  CSA_FMT_FP4_E8M0 = 3, /* index keys */
  CSA_FMT_MXFP8 = 4     /* window KV; index keys (the FP8 index plane) */
} csa_cache_fmt_t;
typedef enum { CSA_MODE_AUTO = 0, CSA_MODE_DECODE = 1, CSA_MODE_PREFILL = 2 } csa_mode_t;

/* ------------------------------------------------------------------------
 * csa_compress - gated compression of every complete group of `ratio` rows.
 *
 * Source: "DeepSeek V4.1 Flash", "Compressor state ownership" (each token
 * carries a KV projection and a gate score of the same width; the pooling
 * softmax; BF16 rounding before RMSNorm) and "Serving-owned full RoPE tables"
 * (compressed rows rotate at their compression-group start position);
 * "DeepSeek V4-Flash, MTP point", "Attention paths" (main compressor
 * rotate=False, index-key compressor rotate=True) and "What is quantized"
 * (INT8 idx_kv quantised on write: amax floored at 1e-4 scaled to 127, FP32
 * per-row scale).
 *
 * Group g of request b is positions g*r .. g*r+r-1.  Without a state ring it
 * is written iff rows t-r+1 .. t of this chunk are request b at exactly those
 * positions.  Per
 * channel d:  logit[j,d] = (x_j . w_gate[:,d]) + ape[j,d];  w = softmax_j;
 * y[d] = sum_j w[j,d] kv_j[d];  y = bf16(y);  optionally
 * y = bf16(gamma * y / sqrt(mean(y^2) + rms_eps));  optionally rotate at g*r;
 * then store BF16 into cmp_pool, or INT8 codes + FP32 scale into
 * idx_pool/idx_scale_pool, at logical entry g of request b.
 *
 * Shapes: x bf16 [n_rows, dx]; kv bf16 [n_rows, d]; w_gate bf16 [dx, d];
 * ape f32 [ratio, d]; gamma bf16 [d] or NULL; positions, row_req i32 [n_rows];
 * block_table i32 [n_req, max_blocks]; cmp_pool bf16 [n_blocks, 128, d];
 * idx_pool i8 [n_blocks, 128, d]; idx_scale_pool f32 [n_blocks, 128].
 * Supported: ratio in {1, 2, 4, 128} (128: HCA's non-overlapping groups,
 * "Hyper-Parallel ... DeepSeek V4 CP", "ratio=128"); d in {128, 512}; dx a
 * multiple of 64 <= 1024.
 * Workspace: n_rows * d * 4 bytes (gate logits), rounded up.
 *
 * Recurrent state ring ("DeepSeek V4.1 Flash", "Compressor state ownership"),
 * optional (state_cache == NULL: none).  state_cache f32
 * [n_state_blocks, state_capacity, 2 * d] is in/out: slot p % state_capacity
 * of block state_block_table[b] holds the kv row of position p (as FP32)
 * followed by its gate score x_p . w_gate + ape[p % ratio].  A row closing a
 * group takes each predecessor from this chunk when it is a preceding row of
 * the same request, else (a position before the chunk start) from the ring.
 * All ring reads complete before any ring write; then the last
 * min(chunk length, state_capacity) rows of each request's chunk (its rows
 * must be consecutive) write their slots.  state_block_table i32 [n_req]:
 * -1 disables the request (nothing published or written); a block >=
 * n_state_blocks sets CSA_DEV_BAD_BLOCK and skips the request.  Rows with a
 * negative position neither publish nor write.  Requires state_capacity >=
 * ratio (at most 256).  A caller built against a header without these four fields passes a
 * smaller struct_size and gets no ring.
 *
 * Low-bit publication (out_mode CSA_OUT_FP4_E4M3, CSA_OUT_FP4_E8M0 or
 * CSA_OUT_MXFP8, see csa_cache_fmt_t): the row as it would be published in
 * BF16 (rotated when `rotate`, in FP32) is quantised per group; codes go to
 * cmp_pool as uint8 [n_blocks, 128, d / 2] (FP4) or [n_blocks, 128, d]
 * (MXFP8) and scale bytes to scale_pool.  Needs a struct_size that covers
 * scale_pool.
 *
 * Overlapping compression (overlap = 1; "Hyper-Parallel ... DeepSeek V4
 * CP", "6.1 ratio4 CSA: compressor halo": the ratio-4 compressor overlaps,
 * a group needing the ratio tokens before it, so the first shard's first
 * slot is padding).
 * Entry g pools the window of the n = min(g*r + r, 2r) tokens ending at
 * g*r + r - 1 -- the tokens of groups g-1 and g, entry 0 only its own --
 * with the same per-channel softmax, token q's logit being
 * x_q . w_gate[:,d] + ape[q % ratio, d].  Without a ring the whole window
 * must be this chunk's rows of request b at those positions; with a ring,
 * state_capacity >= 2 * ratio.  Supported for ratio <= 64 (else
 * CSA_ERR_UNSUPPORTED).  A struct_size that ends before `overlap` means 0.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint32_t struct_size;
  int32_t n_rows;
  int32_t ratio;
  int32_t dx;
  int32_t d;
  int32_t out_mode; /* csa_out_mode_t */
  int32_t rotate;   /* 1: rotate at the group start (needs rope tables) */
  int32_t rope_cap;
  const void *x;
  const void *kv;
  const void *w_gate;
  const float *ape;
  const void *gamma;
  float rms_eps;
  const int32_t *positions;
  const int32_t *row_req;
  const float *rope_cos;
  const float *rope_sin;
  const int32_t *block_table;
  int32_t n_req;
  int32_t max_blocks;
  int32_t n_blocks;
  void *cmp_pool;
  int8_t *idx_pool;
  float *idx_scale_pool;
  uint32_t *status_dev;
  void *workspace;
  size_t workspace_bytes;
  float *state_cache;                /* see "Recurrent state ring" above, or NULL */
  const int32_t *state_block_table;  /* [n_req] */
  int32_t n_state_blocks;
  int32_t state_capacity;
  uint8_t *scale_pool; /* FP4 out modes: scale bytes [n_blocks, 128, d / group] */
  int32_t overlap;     /* 1: each entry pools the previous group too (see above) */
  int64_t pool_page_stride;  /* cmp_pool (BF16) or idx_pool (INT8), bytes; 0: dense */
  int64_t pool_row_stride;   /* ditto */
  int64_t scale_page_stride; /* idx_scale_pool, bytes between pages (rows contiguous); 0: dense */
} csa_compress_args;

CSA_API csa_status_t csa_compress(csa_compress_args *args, csa_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_compress_pair: the two compressors of one attention layer -- the main
 * KV compressor and the index-key compressor, which pool the same rows --
 * in one call.  The result is exactly that of csa_compress(first) followed by
 * csa_compress(second) on the same stream; when both calls take the
 * short-chunk path (at most 256 rows) they share one kernel launch, so the
 * next call on the stream waits for one grid instead of two.
 *
 * Each struct is checked, size-queried (workspace == NULL stores its
 * workspace_bytes; the call then returns CSA_OK without launching) and owns
 * its workspace exactly as in csa_compress.  The two calls must not write the
 * same pool rows.
 * ---------------------------------------------------------------------- */
CSA_API csa_status_t csa_compress_pair(csa_compress_args *first, csa_compress_args *second,
                                       csa_stream_t stream);

/* ------------------------------------------------------------------------
 * csa_index_topk - lightning-indexer scores and deterministic top-k.
 *
 * Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2), sections
 * "10. ratio=4 Global Top-k" (per-row index queries and head weights against
 * the compressed index keys; outputs are compressed slot ids), "10.3 Causal
 * mask" (slot c is visible to position p iff c < (p+1)//ratio); "DeepSeek
 * V4.1 Flash", "Compressor state ownership" (selections in logical-position
 * order with trailing -1 padding); "DeepSeek V4-Flash, MTP point" (INT8
 * idx_kv with FP32 per-row idx_kv_scale).
 *
 * For row t of request b = row_req[t] at p = row_pos[t], visible entries are
 * c < V = min(n_cmp[b], (p+1)/ratio) and
 *   score[c] = scale_c * sum_h w[t,h] * act(q_h . k_c),   act = ReLU if relu
 * where q_h is q_idx[t,h,:] rotated at p when rope tables are given (NULL:
 * q_idx is already rotated) and k_c the INT8 key.  The k best entries by
 * (score descending, index ascending) are written to topk_idx[t] as logical
 * positions in ascending order, padded with -1 when V < k; topk_score (if
 * non-NULL) gets their scores in the same order (padding: -inf).  `scores`
 * (if non-NULL, f32 [n_rows, score_cols], score_cols >= max_blocks*128)
 * receives every visible score; entries c >= V are left untouched.
 *
 * Shapes: q_idx bf16 [n_rows, n_heads, 128]; weights f32 [n_rows, n_heads];
 * row_req, row_pos i32 [n_rows]; n_cmp i32 [n_req]; idx_pool i8
 * [n_blocks, 128, 128]; idx_scale_pool f32 [n_blocks, 128]; cmp_block_table
 * i32 [n_req, max_blocks]; topk_idx i32 [n_rows, topk]; topk_score f32
 * [n_rows, topk] or NULL.  Supported: 1 <= n_heads <= 128 (index heads;
 * the hierarchical modes below: n_heads <= 64), head_dim == 128,
 * 1 <= topk <= 2048, ratio >= 1.
 *
 * Hierarchical indexer ("DeepSeek V4.1 Flash", model structure and the
 * hierarchical indexer: a level-one layer picks 2,048 blocks of eight
 * compressed positions; later reindex layers compute their own index query
 * and select their final positions only inside those blocks).  Candidate
 * block j of a row holds positions j*cand_block .. j*cand_block+cand_block-1.
 *  - Level one (cand_out != NULL): besides the top-k above, cand_out[t]
 *    receives the n_cand blocks with the largest block score, where a
 *    block's score is the largest score of its visible entries (ties: the
 *    lower block), ascending with trailing -1 padding.
 *  - Reindex (cand_in != NULL): row t scores only the visible positions of
 *    its candidate blocks, the longest prefix of cand_in[t] that is
 *    strictly ascending with every block in [0, ceil(V/cand_block)); a
 *    later entry other than -1 raises CSA_DEV_BAD_INDEX and is ignored
 *    (a level-one cand_out row of the same position is always valid).
 *    topk_idx[t] gets the k best of those positions, ascending, -1 padded.
 *    `scores` then holds the candidate scores in candidate order: entry
 *    i < the row's eligible count is the score of position
 *    cand_in[t][i / cand_block] * cand_block + i % cand_block; score_cols
 *    >= n_cand * cand_block.
 * cand_block is 8, 16 or 32; 1 <= n_cand <= 2048; at most one of cand_out
 * and cand_in is set.  A struct_size that ends before `cand_block` (the
 * struct without these fields) turns both off.  csa_index_topk_noalloc
 * returns CSA_ERR_UNSUPPORTED for either mode.
 *
 * Bounded waits: the top-k of rows longer than 16384 entries splits each
 * row over the CTAs of a cooperative launch, which meet at barriers in
 * global memory.  Each
 * wait there gives up after wait_limit_ns (0, or a struct_size that ends
 * before the field: 1 s; negative: at once, without waiting -- a hook for
 * testing the timeout path); a wait that gives up ORs CSA_DEV_TIMEOUT into
 * *status_dev and its CTA stops, so the call's outputs are invalid but the
 * device stays usable.  The call still returns CSA_OK: it does not wait for
 * the device.
 *
 * Key format: key_fmt CSA_FMT_FP4_E8M0 reads idx_pool as packed E2M1 codes
 * uint8 [n_blocks, 128, 64] with key_scale_pool, CSA_FMT_MXFP8 as E4M3
 * codes uint8 [n_blocks, 128, 128] with key_scale_pool (E8M0 bytes
 * [n_blocks, 128, 4] either way); k_c is the dequantised key and scale_c = 1
 * (idx_scale_pool unused).  CSA_FMT_INT8 (or 0, or a
 * struct_size that ends before key_fmt) is the INT8 + FP32 layout above.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint32_t struct_size;
  int32_t n_rows;
  int32_t n_heads;
  int32_t head_dim;
  int32_t ratio;
  int32_t topk;
  int32_t relu;
  int32_t mode; /* csa_mode_t: a tiling hint only; results do not depend on it.
                    AUTO and DECODE: rows in pairs; PREFILL: rows in fours */
  const void *q_idx;
  const float *weights;
  const int32_t *row_req;
  const int32_t *row_pos;
  const int32_t *n_cmp;
  const int8_t *idx_pool;
  const float *idx_scale_pool;
  const int32_t *cmp_block_table;
  int32_t n_req;
  int32_t max_blocks;
  int32_t n_blocks;
  const float *rope_cos;
  const float *rope_sin;
  int32_t rope_cap;
  int32_t *topk_idx;
  float *topk_score;
  float *scores;
  int32_t score_cols;
  uint32_t *status_dev;
  void *workspace;
  size_t workspace_bytes;
  int32_t cand_block;       /* positions per candidate block (8, 16 or 32) */
  int32_t n_cand;           /* candidate blocks per row */
  int32_t *cand_out;        /* i32 [n_rows, n_cand] or NULL: level-one selection */
  const int32_t *cand_in;   /* i32 [n_rows, n_cand] or NULL: reindex candidates */
  int32_t key_fmt;          /* csa_cache_fmt_t: CSA_FMT_INT8 (0 reads as INT8), FP4_E8M0 or MXFP8 */
  const uint8_t *key_scale_pool; /* FP4_E8M0, MXFP8: scale bytes [n_blocks, 128, 4] */
  int64_t wait_limit_ns;    /* bounded device waits: 0 = 1 s, < 0 = give up at once (see above) */
  int64_t key_page_stride;  /* idx_pool (INT8 or FP8 keys), bytes; 0: dense */
  int64_t key_row_stride;   /* ditto */
  int64_t scale_page_stride; /* idx_scale_pool, bytes between pages (rows contiguous); 0: dense */
} csa_index_args;

CSA_API csa_status_t csa_index_topk(csa_index_args *args, csa_stream_t stream);

/* ------------------------------------------------------------------------
 * csa_index_topk_noalloc - csa_index_topk that needs no caller workspace.
 *
 * No counterpart on the pages.  Some callers cannot hand this library device
 * memory: an engine plugin whose device memory is planned once when the
 * engine is built and may not call the CUDA allocator while it serves, or a
 * latency-critical decode loop that must not call cudaMalloc/cudaFree because
 * those can synchronise the whole device and stall every other stream.  This
 * variant computes exactly what csa_index_topk computes, with the same
 * arguments; `workspace`/`workspace_bytes` are ignored and it allocates
 * nothing.  Its score scratch is one array of CSA_NOALLOC_MAX_SCORES FP32
 * entries (4 MiB) inside the library, held on every GPU that loads the
 * library until the process exits.  Limits: a row may hold at most 8192
 * entries (max_blocks * 128 <= 8192) and, unless the caller passes its own
 * `scores` buffer, n_rows * max_blocks * 128 <= CSA_NOALLOC_MAX_SCORES; larger
 * calls return CSA_ERR_UNSUPPORTED and launch nothing.
 * Every call looks up the array's device address in the current device's
 * context (cudaGetSymbolAddress, a host-side lookup); the first call on a
 * device may also load the library's device code there, so make that first
 * call before any stream capture.  Every
 * call on a device shares the array, so calls that overlap on the GPU (two
 * streams, or two threads) race and must be serialised by the caller.  The
 * array keeps the previous call's scores; nothing in it has to start at zero,
 * because only entries a call writes are read back.
 * ---------------------------------------------------------------------- */
#define CSA_NOALLOC_MAX_SCORES (1u << 20)

CSA_API csa_status_t csa_index_topk_noalloc(csa_index_args *args, csa_stream_t stream);

/* ------------------------------------------------------------------------
 * csa_sparse_attn_decode / csa_sparse_attn_prefill - shared-KV sparse
 * attention with an attention sink.
 *
 * Source: "Hyper-Parallel ... DeepSeek V4 CP", "二阶段 CP 总体算法" (Stage-2:
 * sparse attention over the window KV and the selected compressed KV with
 * sinks, softmax_scale and ori_win_left = 127; outputs out and lse), "9.1"
 * (the candidate list is the window rows followed by the compressed rows),
 * "7. Window KV Halo" (the window includes the query's own position);
 * "DeepSeek V4-Flash, MTP point", "Deployment configuration" (decode: 2 rows
 * per request; prefill: up to 8192 tokens walked in 128-token tiles).
 *
 * For row t (request b, position p), candidates are cmp entry c for every
 * c = topk_idx[t, i] >= 0 and raw row p' for p' in [max(0, p-window+1), p].
 * topk_idx == NULL selects dense compressed visibility (HCA: "Hyper-Parallel
 * ... DeepSeek V4 CP", "ratio=128" and "10.3 Causal mask"): every visible
 * entry c < V = min(n_cmp[b], (p+1)/ratio) is a candidate; topk is then the
 * capacity, and V > topk raises CSA_DEV_BAD_INDEX and keeps entries
 * 0 .. topk-1.
 * Each candidate row k_i is both key and value.  Per head h, with q_h =
 * q[t,h,:] rotated at p:
 *   l_i = softmax_scale * q_h . k_i
 *   out[t,h,:] = sum_i e^{l_i} k_i / (sum_i e^{l_i} + e^{sink_h})
 *   lse[t,h]   = log(sum_i e^{l_i} + e^{sink_h})
 * sink == NULL means -inf (plain softmax).  inv_rope_out rotates the output
 * back by -p.  Top-k entries must be unique (the indexer guarantees it); an
 * entry outside [0, min(n_cmp[b], (p+1)/ratio)) raises CSA_DEV_BAD_INDEX and
 * is skipped; a window position >= kv_len[b] raises CSA_DEV_BAD_POS and is
 * skipped.
 *
 * Shapes: q bf16 [n_rows, n_heads, 512]; kv_pool, cmp_pool bf16
 * [*, 128, 512]; kv_block_table i32 [n_req, kv_max_blocks]; cmp_block_table
 * i32 [n_req, cmp_max_blocks]; kv_len, n_cmp i32 [n_req]; topk_idx i32
 * [n_rows, topk]; sink f32 [n_heads] or NULL; out bf16 [n_rows, n_heads,
 * 512]; lse f32 [n_rows, n_heads] or NULL.  Supported: 1 <= n_heads <= 128
 * (the kernels work in groups of 64 heads, a group of a row at a time),
 * head_dim == 512, window == 128, topk <= 2048.
 * The decode call splits each row's candidates over up to 17 CTAs (one per
 * 128-candidate tile while the whole grid fits one CTA per SM) and merges the
 * partial softmaxes through its workspace: per (row, group of 64 heads) and
 * split, 64 KB of BF16 partial output and 512 bytes of statistics, plus two
 * 32-bit counters per (row, head group) at the end.  The counters must read
 * zero before the workspace's first decode call; every call that completes
 * leaves them at zero (a call that raised CSA_DEV_TIMEOUT may not: zero them
 * again).  Counters that do not start at zero make the call raise
 * CSA_DEV_TIMEOUT (a wait for exactly the number of splits runs out); its
 * output is then undefined.  The workspace must be 256-byte aligned.  The prefill call is tiled for many rows; with BF16 pools
 * it needs no workspace (the size query returns 0; a workspace passed in is
 * unused, but a non-null pointer is what makes the call launch) and with a
 * low-bit pool it needs the arena below.  Both compute the same function.
 *
 * Low-bit caches (see csa_cache_fmt_t): kv_fmt CSA_FMT_MXFP8 reads kv_pool
 * as uint8 [*, 128, 512] with kv_scale_pool; cmp_fmt CSA_FMT_FP4_E4M3 reads
 * cmp_pool as uint8 [*, 128, 256] with cmp_scale_pool.  Each candidate row is
 * dequantised (exactly: every such value is a BF16 value).  The decode call
 * dequantises each candidate row as it gathers it.  The prefill call first
 * dequantises every mapped page of the requests' block tables into a BF16
 * arena in its workspace (per low-bit pool: n_req * max_blocks pages of
 * 128 KB plus an INT32 table, as the size query reports; a table entry
 * outside the pool is left unmapped in the arena), then reads the arena.
 * A struct_size that ends before kv_fmt reads both pools as BF16.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint32_t struct_size;
  int32_t n_rows;
  int32_t n_heads;
  int32_t head_dim;
  int32_t ratio;
  int32_t topk;
  int32_t window;
  int32_t inv_rope_out;
  float softmax_scale;
  const void *q;
  const int32_t *row_req;
  const int32_t *row_pos;
  const int32_t *topk_idx;
  const void *kv_pool;
  const int32_t *kv_block_table;
  int32_t kv_max_blocks;
  int32_t kv_n_blocks;
  const int32_t *kv_len;
  const void *cmp_pool;
  const int32_t *cmp_block_table;
  int32_t cmp_max_blocks;
  int32_t cmp_n_blocks;
  const int32_t *n_cmp;
  int32_t n_req;
  const float *sink;
  const float *rope_cos;
  const float *rope_sin;
  int32_t rope_cap;
  void *out;
  float *lse;
  uint32_t *status_dev;
  void *workspace;
  size_t workspace_bytes;
  int32_t kv_fmt;  /* csa_cache_fmt_t: CSA_FMT_BF16 (0) or CSA_FMT_MXFP8 */
  int32_t cmp_fmt; /* csa_cache_fmt_t: CSA_FMT_BF16 (0) or CSA_FMT_FP4_E4M3 */
  const uint8_t *kv_scale_pool;  /* MXFP8: scale bytes [kv_n_blocks, 128, 16] */
  const uint8_t *cmp_scale_pool; /* FP4_E4M3: scale bytes [cmp_n_blocks, 128, 32] */
  int64_t kv_page_stride;  /* kv_pool (BF16), bytes; 0: dense (see "Pool strides") */
  int64_t kv_row_stride;
  int64_t cmp_page_stride; /* cmp_pool (BF16), bytes; 0: dense */
  int64_t cmp_row_stride;
} csa_attn_args;

CSA_API csa_status_t csa_sparse_attn_decode(csa_attn_args *args, csa_stream_t stream);
CSA_API csa_status_t csa_sparse_attn_prefill(csa_attn_args *args, csa_stream_t stream);

/* ------------------------------------------------------------------------
 * Library information and measurement hooks (no counterpart on the pages).
 * ---------------------------------------------------------------------- */

/* "csa <version> sm_103a" */
CSA_API const char *csa_version(void);
/* human-readable name of a status code */
CSA_API const char *csa_status_string(csa_status_t s);
/* number of kernels this process has launched through the library */
CSA_API uint64_t csa_launch_count(void);

/* Kernel identifiers for the timing hooks. */
typedef enum {
  CSA_K_COMPRESS_GATE = 0,  /* long chunks: gate logits GEMM */
  CSA_K_COMPRESS_POOL = 1,  /* long chunks: softmax pooling and publication */
  CSA_K_COMPRESS_FUSED = 2, /* short chunks: the whole compressor in one kernel */
  CSA_K_INDEX_SCORE = 3,
  CSA_K_INDEX_TOPK = 4,
  CSA_K_ATTN_DECODE = 5,
  CSA_K_ATTN_PREFILL = 6,
  CSA_K_DEQUANT = 7,        /* low-bit pools into the prefill call's BF16 arena */
  CSA_K_COUNT = 8
} csa_kernel_id_t;

/* Time every launch of kernel `kernel_id` (up to `max_launches` launches)
 * with a CUDA event pair: the first event completes when the work issued on
 * the launching stream before the kernel is done, the second when the kernel
 * is done.  Both are recorded on a library-owned side stream forked from the
 * launching stream, so the launching stream gains no node between the kernel
 * and its neighbours (their programmatic launch overlap is kept).  Events and
 * the side stream are created by the library; no device memory is allocated.
 * Inside stream capture, csa_prof_join must bring the side stream back into
 * the captured stream before the capture ends. */
CSA_API csa_status_t csa_prof_enable(int32_t kernel_id, int32_t max_launches);
/* Make `stream` wait for every timing event recorded so far (a no-op when
 * timing is off). */
CSA_API csa_status_t csa_prof_join(csa_stream_t stream);
/* Synchronise the recorded events and return the summed device time (ms) and
 * the number of launches recorded since csa_prof_enable. */
CSA_API csa_status_t csa_prof_read(int32_t kernel_id, float *total_ms, int32_t *n_launches);
CSA_API csa_status_t csa_prof_disable(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
