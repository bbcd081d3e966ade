// Shared-KV sparse attention with an attention sink: candidates are the
// selected compressed entries plus the raw causal window; each candidate row
// is both key and value.
//
// Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2),
// "二阶段 CP 总体算法" (Stage-2 sparse attention with sinks, softmax_scale,
// ori_win_left = 127, outputs out and lse) and "7. Window KV Halo" (window
// includes self).
//
// Each CTA handles one query row and a contiguous slice of its candidate
// list (split-K); slices are merged by their softmax statistics.  With a
// single slice the CTA writes the final output directly.
#include "csa_internal.cuh"

namespace csa {
namespace {

constexpr int AT_TILE = 32;           // candidates per shared-memory tile
constexpr int AT_THREADS = 256;
constexpr int AT_QS = kHeadDim + 4;   // padded row stride (floats)

struct AttnSmem {
  float q[kHeads][AT_QS];
  float kv[AT_TILE][AT_QS];
  float p[kHeads][AT_TILE + 1];
  float corr[kHeads];
  float m[kHeads];
  float l[kHeads];
  int valid[AT_TILE];
};

// Row of candidate `gi` of query row t, or -1 when the slot is empty.
__device__ __forceinline__ const uint16_t *candidate_row(const csa_attn_args &a, int t, int b,
                                                        int p, int V, int gi) {
  if (gi < a.topk) {
    const int c = a.topk_idx[(long long)t * a.topk + gi];
    if (c < 0) return nullptr;
    if (c >= V) {
      flag(a.status_dev, CSA_DEV_BAD_INDEX);
      return nullptr;
    }
    long long row = page_row(a.cmp_block_table, a.cmp_max_blocks, a.cmp_n_blocks, b, c,
                             a.status_dev);
    return row < 0 ? nullptr : static_cast<const uint16_t *>(a.cmp_pool) + row * kHeadDim;
  }
  const int j = gi - a.topk;
  const int pp = p - a.window + 1 + j;
  if (pp < 0) return nullptr;
  if (pp >= a.kv_len[b]) {
    flag(a.status_dev, CSA_DEV_BAD_POS);
    return nullptr;
  }
  long long row = page_row(a.kv_block_table, a.kv_max_blocks, a.kv_n_blocks, b, pp,
                           a.status_dev);
  return row < 0 ? nullptr : static_cast<const uint16_t *>(a.kv_pool) + row * kHeadDim;
}

__device__ __forceinline__ void store_bf16x2(void *base, long long idx, float x0, float x1) {
  __nv_bfloat162 v = __floats2bfloat162_rn(x0, x1);
  reinterpret_cast<__nv_bfloat162 *>(base)[idx / 2] = v;
}

// Final normalisation of one row: out = o / L, lse = M + log L, where the
// sink joins the denominator.  Optional inverse rotation of the output.
__device__ void finalize_row(const csa_attn_args &a, int t, int p, const float *o_src,
                             int o_stride_h, const float *M, const float *L, float *obuf) {
  // o_src[h * o_stride_h + d] holds the unnormalised sum at max M[h]
  bool inv = a.inv_rope_out && a.rope_cos != nullptr && p >= 0 && p < a.rope_cap;
  for (int e = threadIdx.x; e < kHeads * (kHeadDim / 2); e += blockDim.x) {
    const int h = e / (kHeadDim / 2), d = 2 * (e % (kHeadDim / 2));
    const float invL = L[h] > 0.f ? 1.f / L[h] : 0.f;
    float x0 = o_src[h * o_stride_h + d] * invL;
    float x1 = o_src[h * o_stride_h + d + 1] * invL;
    if (inv && d >= kHeadDim - kRopeDim) {
      const int i = (d - (kHeadDim - kRopeDim)) >> 1;
      const float c = a.rope_cos[(long long)p * kRopeHalf + i];
      const float s = a.rope_sin[(long long)p * kRopeHalf + i];
      const float y0 = x0 * c + x1 * s, y1 = -x0 * s + x1 * c;
      x0 = y0;
      x1 = y1;
    }
    store_bf16x2(a.out, ((long long)t * kHeads + h) * kHeadDim + d, x0, x1);
  }
  if (a.lse && threadIdx.x < kHeads) {
    const int h = threadIdx.x;
    a.lse[(long long)t * kHeads + h] = L[h] > 0.f ? M[h] + logf(L[h]) : -INFINITY;
  }
  (void)obuf;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_partial_kernel(csa_attn_args a, int n_splits, int tiles_per_split,
                        float *__restrict__ partials) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem &S = *reinterpret_cast<AttnSmem *>(smem_raw);
  const int t = blockIdx.y;
  const int split = blockIdx.x;
  const int b = a.row_req[t];
  if (b < 0) return;
  if (b >= a.n_req) {
    if (threadIdx.x == 0 && split == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int p = a.row_pos[t];
  const int V = visible_count(p, a.ratio, a.n_cmp[b]);
  const int n_cand = a.topk + a.window;
  const int g_begin = split * tiles_per_split * AT_TILE;
  const int g_end = min(n_cand, g_begin + tiles_per_split * AT_TILE);

  // q rotated at p, FP32
  bool rot = a.rope_cos != nullptr && p >= 0;
  if (rot && p >= a.rope_cap) {
    rot = false;
    if (threadIdx.x == 0 && split == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
  }
  const uint16_t *qg = static_cast<const uint16_t *>(a.q) + (long long)t * kHeads * kHeadDim;
  for (int e = threadIdx.x; e < kHeads * kHeadDim / 2; e += blockDim.x) {
    const int h = e / (kHeadDim / 2), d = 2 * (e % (kHeadDim / 2));
    float x0 = bf16_bits_to_float(qg[h * kHeadDim + d]);
    float x1 = bf16_bits_to_float(qg[h * kHeadDim + d + 1]);
    if (rot && d >= kHeadDim - kRopeDim) {
      const int i = (d - (kHeadDim - kRopeDim)) >> 1;
      const float c = a.rope_cos[(long long)p * kRopeHalf + i];
      const float s = a.rope_sin[(long long)p * kRopeHalf + i];
      const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
      x0 = y0;
      x1 = y1;
    }
    S.q[h][d] = x0 * a.softmax_scale;
    S.q[h][d + 1] = x1 * a.softmax_scale;
  }
  if (threadIdx.x < kHeads) {
    S.m[threadIdx.x] = -INFINITY;
    S.l[threadIdx.x] = 0.f;
  }
  float o[kHeads][2];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) o[h][0] = o[h][1] = 0.f;
  const int dcol = threadIdx.x * 2;  // this thread's two output channels
  __syncthreads();

  for (int g0 = g_begin; g0 < g_end; g0 += AT_TILE) {
    // ---- gather the tile (bf16 -> fp32)
    for (int e = threadIdx.x; e < AT_TILE * (kHeadDim / 8); e += blockDim.x) {
      const int j = e / (kHeadDim / 8), v = e % (kHeadDim / 8);
      const int gi = g0 + j;
      const uint16_t *src = gi < g_end ? candidate_row(a, t, b, p, V, gi) : nullptr;
      // every thread of a row evaluates the same candidate; only v == 0 records validity
      float f[8];
      if (src) {
        int4 raw = reinterpret_cast<const int4 *>(src)[v];
        const uint16_t *h16 = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = bf16_bits_to_float(h16[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) S.kv[j][v * 8 + i] = f[i];
      if (v == 0) S.valid[j] = src != nullptr;
    }
    __syncthreads();

    // ---- logits: thread -> head h, candidates j = tid%4 + 4m
    {
      const int h = threadIdx.x / 4, j0 = threadIdx.x % 4;
      float acc[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) acc[m] = 0.f;
      for (int d = 0; d < kHeadDim; d += 4) {
        const float4 qv = *reinterpret_cast<const float4 *>(&S.q[h][d]);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float4 kv4 = *reinterpret_cast<const float4 *>(&S.kv[j0 + 4 * m][d]);
          acc[m] = fmaf(qv.x, kv4.x, acc[m]);
          acc[m] = fmaf(qv.y, kv4.y, acc[m]);
          acc[m] = fmaf(qv.z, kv4.z, acc[m]);
          acc[m] = fmaf(qv.w, kv4.w, acc[m]);
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j = j0 + 4 * m;
        S.p[h][j] = S.valid[j] ? acc[m] : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax statistics per head
    if (threadIdx.x < kHeads) {
      const int h = threadIdx.x;
      float mx = S.m[h];
      for (int j = 0; j < AT_TILE; ++j) mx = fmaxf(mx, S.p[h][j]);
      float corr = 1.f, sum = 0.f;
      if (mx == -INFINITY) {
        for (int j = 0; j < AT_TILE; ++j) S.p[h][j] = 0.f;
      } else {
        corr = expf(S.m[h] - mx);  // exp(-inf) = 0 on the first tile
        for (int j = 0; j < AT_TILE; ++j) {
          const float e = expf(S.p[h][j] - mx);
          S.p[h][j] = e;
          sum += e;
        }
        S.m[h] = mx;
      }
      S.l[h] = S.l[h] * corr + sum;
      S.corr[h] = corr;
    }
    __syncthreads();

    // ---- o[h][dcol..dcol+1] = o * corr + sum_j p[h][j] * kv[j][dcol..]
    // (fully unrolled over h so that o[][] stays in registers)
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      float o0 = o[h][0] * S.corr[h], o1 = o[h][1] * S.corr[h];
#pragma unroll 8
      for (int j = 0; j < AT_TILE; ++j) {
        const float pj = S.p[h][j];
        const float2 v = *reinterpret_cast<const float2 *>(&S.kv[j][dcol]);
        o0 = fmaf(pj, v.x, o0);
        o1 = fmaf(pj, v.y, o1);
      }
      o[h][0] = o0;
      o[h][1] = o1;
    }
    __syncthreads();
  }

  if (n_splits == 1) {
    // fold the sink into the denominator and write the output directly
    __syncthreads();
    if (threadIdx.x < kHeads) {
      const int h = threadIdx.x;
      const float sink = a.sink ? a.sink[h] : -INFINITY;
      float M = fmaxf(S.m[h], sink);
      float L = 0.f;
      if (M != -INFINITY) {
        const float cs = expf(S.m[h] - M);  // rescale of o and l
        L = S.l[h] * cs + expf(sink - M);
        S.corr[h] = cs;
      } else {
        S.corr[h] = 0.f;
      }
      S.m[h] = M;
      S.l[h] = L;
    }
    __syncthreads();
    // stage o * corr in shared memory, reusing S.q as [64][AT_QS] scratch
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      S.q[h][dcol] = o[h][0] * S.corr[h];
      S.q[h][dcol + 1] = o[h][1] * S.corr[h];
    }
    __syncthreads();
    finalize_row(a, t, p, &S.q[0][0], AT_QS, S.m, S.l, nullptr);
    return;
  }

  // partial record: [h][d] unnormalised o, then m[h], l[h]
  float *rec = partials + ((long long)t * n_splits + split) * (kHeads * (kHeadDim + 2));
#pragma unroll
  for (int h = 0; h < kHeads; ++h)
    *reinterpret_cast<float2 *>(&rec[h * kHeadDim + dcol]) = make_float2(o[h][0], o[h][1]);
  if (threadIdx.x < kHeads) {
    rec[kHeads * kHeadDim + threadIdx.x] = S.m[threadIdx.x];
    rec[kHeads * kHeadDim + kHeads + threadIdx.x] = S.l[threadIdx.x];
  }
}

// Merge the split partials of one row with the sink.
__global__ void __launch_bounds__(512) attn_combine_kernel(csa_attn_args a, int n_splits,
                                                           const float *__restrict__ partials) {
  __shared__ float M[kHeads], L[kHeads];
  __shared__ float obuf[kHeads * 8];  // unused placeholder for finalize_row signature
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float *osum = reinterpret_cast<float *>(smem_raw);  // [64][512]
  const int t = blockIdx.x;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;
  const int p = a.row_pos[t];
  const float *rec0 = partials + (long long)t * n_splits * (kHeads * (kHeadDim + 2));
  const int rec_sz = kHeads * (kHeadDim + 2);
  if (threadIdx.x < kHeads) {
    const int h = threadIdx.x;
    const float sink = a.sink ? a.sink[h] : -INFINITY;
    float mx = sink;
    for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, rec0[s * rec_sz + kHeads * kHeadDim + h]);
    float l = 0.f;
    if (mx != -INFINITY) {
      l = expf(sink - mx);
      for (int s = 0; s < n_splits; ++s) {
        const float ms = rec0[s * rec_sz + kHeads * kHeadDim + h];
        const float ls = rec0[s * rec_sz + kHeads * kHeadDim + kHeads + h];
        if (ms != -INFINITY) l += ls * expf(ms - mx);
      }
    }
    M[h] = mx;
    L[h] = l;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kHeads * kHeadDim; e += blockDim.x) {
    const int h = e / kHeadDim;
    float acc = 0.f;
    if (M[h] != -INFINITY) {
      for (int s = 0; s < n_splits; ++s) {
        const float ms = rec0[s * rec_sz + kHeads * kHeadDim + h];
        if (ms != -INFINITY) acc = fmaf(rec0[s * rec_sz + e], expf(ms - M[h]), acc);
      }
    }
    osum[e] = acc;
  }
  __syncthreads();
  finalize_row(a, t, p, osum, kHeadDim, M, L, obuf);
}

}  // namespace

cudaError_t launch_attn(const csa_attn_args &a, int n_splits, int tiles_per_split,
                        float *partials, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  const int smem = (int)sizeof(AttnSmem);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(attn_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kHeads * kHeadDim * 4);
    attr_set[dev] = true;
  }
  dim3 grid(n_splits, a.n_rows);
  const int kid = n_splits == 1 ? CSA_K_ATTN_PREFILL : CSA_K_ATTN_PARTIAL;
  launch_begin(kid, s);
  attn_partial_kernel<<<grid, AT_THREADS, smem, s>>>(a, n_splits, tiles_per_split, partials);
  launch_end(kid, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_splits == 1) return e;
  launch_begin(CSA_K_ATTN_COMBINE, s);
  attn_combine_kernel<<<a.n_rows, 512, kHeads * kHeadDim * 4, s>>>(a, n_splits, partials);
  launch_end(CSA_K_ATTN_COMBINE, s);
  return cudaGetLastError();
}

}  // namespace csa
