// Internal declarations shared by the CSA kernels and the C-ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

constexpr int kBlock = CSA_BLOCK;       // rows per page
constexpr int kRopeDim = CSA_ROPE_DIM;  // rotated channels
constexpr int kRopeHalf = kRopeDim / 2;
constexpr int kHeadDim = 512;           // attention head / KV width
constexpr int kIdxDim = 128;            // index-key width
constexpr int kHeads = 64;              // heads per MMA tile (a group of heads)
constexpr int kMaxHeads = 128;          // query heads and index heads of a call, at most
constexpr int kWindow = CSA_WINDOW;

// ---------------------------------------------------------------- host side

// Bracket one kernel launch: counts launches and, when enabled, records a
// CUDA event pair on the launching stream for that kernel id.
void launch_begin(int kernel_id, cudaStream_t s);
void launch_end(int kernel_id, cudaStream_t s);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A paged pool's strides in bytes, 0 meaning dense (a row stride of
// `row_bytes`, a page stride of 128 row strides); false when they are not
// multiples of 16, the row stride is below the row's bytes or the page
// stride below 128 row strides.
inline bool normalize_strides(int64_t *page, int64_t *row, int64_t row_bytes) {
  if (*row == 0) *row = row_bytes;
  if (*page == 0) *page = 128 * *row;
  return *row % 16 == 0 && *page % 16 == 0 && *row >= row_bytes && *page >= 128 * *row;
}

// Launch a kernel with programmatic dependent launch: it may be scheduled
// while the previous kernel on the stream finishes, and waits for it in
// griddep_wait() before touching global memory.  `cluster_x` > 0 launches
// clusters of that many CTAs along x; `cooperative` makes the grid's CTAs
// co-resident (the launch fails if they cannot all be) and is launched
// without the early start.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, int cluster_x, bool cooperative, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[3];
  unsigned n = 0;
  if (!cooperative) {  // a cooperative grid is launched whole, after its predecessor
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = (unsigned)cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  if (cooperative) {
    attrs[n].id = cudaLaunchAttributeCooperative;
    attrs[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Launchers (one per kernel family); each returns cudaGetLastError().
cudaError_t launch_compress(const csa_compress_args &a, float *logits, cudaStream_t s);
// two compressors of one layer; one launch when both take the short-chunk path
cudaError_t launch_compress_pair(const csa_compress_args &a, float *logits_a,
                                 const csa_compress_args &b, float *logits_b, cudaStream_t s);
// Words per row of the long-row top-k control block (barrier counter and
// three digit histograms).
constexpr int kTopkCtlWords = 32 + 2048 + 2048 + 1024;
// Hierarchical-indexer options of the scoring kernel (all off by default).
struct ScoreSel {
  const int32_t *cand_in = nullptr;  // reindex: candidate blocks [n_rows, n_cand]
  int n_cand = 0;
  int cb_shift = 3;                  // log2(positions per candidate block)
  int32_t *v_row = nullptr;          // reindex: each row's eligible entry count (written)
  float *blk = nullptr;              // level one: block maxima [n_rows, blk_cols] (written)
  int blk_cols = 0;
  uint32_t *zero2 = nullptr;         // a second control block range to clear (n_rows rows)
};
// Options of one top-k launch (all off by default: the indexer's own selection).
struct TopkSel {
  int v_div = 1;                     // a row holds ceil(V / v_div) entries (block scores)
  const int32_t *v_row = nullptr;    // a row holds v_row[t] entries (reindex)
  const int32_t *cand = nullptr;     // emitted entry i is position cand[t][i >> cb_shift] ...
  int cand_stride = 0;               // ... << cb_shift | (i & (2^cb_shift - 1))
  int cb_shift = 3;
  int n_cap = 0;                     // longest row (0: max_blocks * 128)
};
// `zero_ctr` (n_rows x kTopkCtlWords words, may be null) is cleared by the
// scoring kernel for the top-k kernel that follows it on the stream.
cudaError_t launch_index_scores(const csa_index_args &a, float *scores, int score_cols,
                                uint32_t *zero_ctr, cudaStream_t s,
                                const ScoreSel &sel = ScoreSel());
cudaError_t launch_index_topk(const csa_index_args &a, const float *scores, int score_cols,
                              void *topk_ws, cudaStream_t s, const TopkSel &sel = TopkSel());
// The caller's csa_index_args as this library's struct (fields past the
// caller's struct_size zeroed); index_struct_ok checks that struct_size
// covers every field before the hierarchical-indexer ones.
csa_index_args full_index_args(const csa_index_args *a);
bool index_struct_ok(const csa_index_args *a);
// Pointer, count and alignment checks of a launching index call.
bool index_pointers_ok(const csa_index_args *a);
// The key pool's strides made explicit (0: dense); CSA_OK, or the status to
// return.
csa_status_t index_normalize_strides(csa_index_args *a);
bool topk_is_long(int n_cap);
size_t topk_ws_bytes(int n_rows, int n_cap);
uint32_t *topk_counters(void *ws, int n_rows, int n_cap);
// Low-bit pools of a prefill call dequantised into a BF16 arena in the
// workspace (k_dequant.cu): its size, and the launch that fills it and
// points `bf` (a copy of `a`) at it.
size_t attn_arena_bytes(const csa_attn_args &a);
cudaError_t launch_dequant_arena(const csa_attn_args &a, void *ws, csa_attn_args *bf,
                                 cudaStream_t s);
// The persistent prefill kernel (k_attn_prefill.cu).
bool attn_prefill_supported(const csa_attn_args &a);
cudaError_t launch_attn_prefill(const csa_attn_args &a, cudaStream_t s);
// Decode attention (k_attn.cu): a row's candidate tiles split over the CTAs
// of one cluster, merged in distributed shared memory.
void attn_decode_geometry(const csa_attn_args &a, int *n_splits, int *tiles_per_split);
size_t attn_decode_workspace(const csa_attn_args &a);
cudaError_t launch_attn_decode(const csa_attn_args &a, cudaStream_t s);

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void flag(uint32_t *status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Physical row of logical position `pos` of request b in a paged pool, or -1
// (and a flag) when the page is unmapped or outside the pool.
__device__ __forceinline__ long long page_row(const int32_t *table, int max_blocks, int n_blocks,
                                              int b, int pos, uint32_t *status) {
  int page = pos / kBlock;
  if (page >= max_blocks) {
    flag(status, CSA_DEV_BAD_BLOCK);
    return -1;
  }
  int phys = table[(long long)b * max_blocks + page];
  if (phys < 0 || phys >= n_blocks) {
    flag(status, CSA_DEV_BAD_BLOCK);
    return -1;
  }
  return (long long)phys * kBlock + (pos % kBlock);
}

// Byte offset of pool row `row` (physical page * 128 + row in the page).
__device__ __forceinline__ long long pool_offset(long long row, long long page_stride,
                                                 long long row_stride) {
  return (row >> 7) * page_stride + (row & 127) * row_stride;
}

// Number of compressed entries visible to a query at position p:
// min(n_cmp, (p + 1) / ratio), 0 for negative positions.
__device__ __forceinline__ int visible_count(int p, int ratio, int n_cmp) {
  if (p < 0) return 0;
  int v = (p + 1) / ratio;
  return v < n_cmp ? v : n_cmp;
}

}  // namespace csa
