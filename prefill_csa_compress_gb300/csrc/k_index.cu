// Deterministic top-k over the lightning-indexer scores.
//
// Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2), "10. ratio=4
// Global Top-k" and "10.3 Causal mask"; "DeepSeek V4.1 Flash", "Compressor
// state ownership" (logical positions in ascending order, trailing -1);
// "DeepSeek V4-Flash, MTP point", "What is quantized" (INT8 keys, FP32 scale).
#include "csa_internal.cuh"

namespace csa {
namespace {

// Order-preserving 32-bit key of a float score: larger score -> larger key.
// +0 and -0 share a key; NaN maps to the smallest key.
__device__ __forceinline__ uint32_t order_key(float s) {
  if (s != s) return 0u;
  if (s == 0.f) s = 0.f;
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const int base = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[31];
  return base + x - v;
}

// One CTA (1024 threads) per row: 4-pass radix select of the k-th largest
// key, then an ordered compaction so the output is ascending by position.
__global__ void __launch_bounds__(1024) index_topk_kernel(csa_index_args a,
                                                          const float *__restrict__ scores,
                                                          int score_cols) {
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int t = blockIdx.x;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;
  const int p = a.row_pos[t];
  const int V = min(visible_count(p, a.ratio, a.n_cmp[b]), a.max_blocks * kBlock);
  const int k = a.topk;
  int32_t *out = a.topk_idx + (long long)t * k;
  float *out_s = a.topk_score ? a.topk_score + (long long)t * k : nullptr;
  const float *sc = scores + (long long)t * score_cols;

  if (V <= k) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
      out[i] = i < V ? i : -1;
      if (out_s) out_s[i] = i < V ? sc[i] : -INFINITY;
    }
    return;
  }

  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < V; c += blockDim.x) {
      uint32_t key = order_key(sc[c]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, sel = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        if (cum + hist[dgt] >= remaining) {
          sel = dgt;
          break;
        }
        cum += hist[dgt];
      }
      s_prefix = prefix | ((uint32_t)sel << shift);
      s_remaining = remaining - cum;
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix is now the exact k-th largest key; `remaining` entries equal to it
  // are taken, smallest positions first.
  const uint32_t T = prefix;
  int eq_base = 0, sel_base = 0;
  for (int c0 = 0; c0 < V; c0 += blockDim.x) {
    const int c = c0 + threadIdx.x;
    uint32_t key = c < V ? order_key(sc[c]) : 0u;
    const int gt = (c < V && key > T) ? 1 : 0;
    const int eq = (c < V && key == T) ? 1 : 0;
    int eq_total;
    const int eq_rank = eq_base + block_exclusive_scan(eq, warp_sums, &eq_total);
    const int sel = gt | (eq && eq_rank < remaining);
    int sel_total;
    const int pos = sel_base + block_exclusive_scan(sel, warp_sums, &sel_total);
    if (sel && pos < k) {
      out[pos] = c;
      if (out_s) out_s[pos] = sc[c];
    }
    eq_base += eq_total;
    sel_base += sel_total;
  }
}

}  // namespace

cudaError_t launch_index_topk(const csa_index_args &a, const float *scores, int score_cols,
                              cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  launch_begin(CSA_K_INDEX_TOPK, s);
  index_topk_kernel<<<a.n_rows, 1024, 0, s>>>(a, scores, score_cols);
  launch_end(CSA_K_INDEX_TOPK, s);
  return cudaGetLastError();
}

}  // namespace csa
