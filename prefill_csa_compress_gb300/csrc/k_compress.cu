// Gated compressor: gate logits GEMM, then per-group softmax pooling with the
// BF16 / RMSNorm / RoPE / INT8 epilogue.
//
// Source: "DeepSeek V4.1 Flash", "Compressor state ownership" (per-token KV and
// gate score of the same width, pooling softmax, BF16 rounding before RMSNorm)
// and "Serving-owned full RoPE tables" (group-start rotation); "DeepSeek
// V4-Flash, MTP point", "What is quantized" (INT8 on write, amax floored at
// 1e-4, scaled to 127).
#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

// ---------------------------------------------------------------------------
// logits[t, d] = sum_k x[t, k] * w_gate[k, d]   (FP32 accumulate)
// Tile: 32 rows x 64 columns per CTA, K staged through shared memory in 64s.
// ---------------------------------------------------------------------------
constexpr int GT_ROWS = 32, GT_COLS = 64, GT_K = 64;

__global__ void __launch_bounds__(256) gate_logits_kernel(const uint16_t *__restrict__ x,
                                                          const uint16_t *__restrict__ w,
                                                          float *__restrict__ logits, int n_rows,
                                                          int dx, int d) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  __shared__ float xs[GT_ROWS][GT_K + 1];
  __shared__ float ws[GT_K][GT_COLS];
  const int tx = threadIdx.x % GT_COLS;
  const int ty = threadIdx.x / GT_COLS;  // 0..3, 8 rows each
  const int col = blockIdx.x * GT_COLS + tx;
  const int row0 = blockIdx.y * GT_ROWS;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  for (int k0 = 0; k0 < dx; k0 += GT_K) {
    for (int e = threadIdx.x; e < GT_ROWS * GT_K; e += blockDim.x) {
      int r = e / GT_K, k = e % GT_K;
      int gr = row0 + r;
      xs[r][k] = gr < n_rows ? bf16_bits_to_float(x[(long long)gr * dx + k0 + k]) : 0.f;
    }
    for (int e = threadIdx.x; e < GT_K * GT_COLS; e += blockDim.x) {
      int k = e / GT_COLS, c = e % GT_COLS;
      int gc = blockIdx.x * GT_COLS + c;
      ws[k][c] = gc < d ? bf16_bits_to_float(w[(long long)(k0 + k) * d + gc]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < GT_K; ++k) {
      float wv = ws[k][tx];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(xs[ty * 8 + i][k], wv, acc[i]);
    }
    __syncthreads();
  }
  if (col < d) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int gr = row0 + ty * 8 + i;
      if (gr < n_rows) logits[(long long)gr * d + col] = acc[i];
    }
  }
}

// ---------------------------------------------------------------------------
// One CTA per candidate group-end row t; one thread per channel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float *red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < (int)blockDim.x / 32; ++i) s += red[i];
  return s;
}

__device__ __forceinline__ float block_max(float v, float *red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = red[0];
  for (int i = 1; i < (int)blockDim.x / 32; ++i) s = fmaxf(s, red[i]);
  return s;
}

__global__ void compress_pool_kernel(csa_compress_args a, const float *__restrict__ logits) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  __shared__ float ys[512];
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int r = a.ratio, D = a.d;
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || p < 0 || (p % r) != r - 1 || t < r - 1) return;
  for (int j = 1; j < r; ++j)
    if (a.row_req[t - j] != b || a.positions[t - j] != p - j) return;
  if (b >= a.n_req) {
    if (threadIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int g = p / r;
  const int page = g / kBlock;
  int phys = -1;
  if (page < a.max_blocks) phys = a.block_table[(long long)b * a.max_blocks + page];
  if (phys < 0 || phys >= a.n_blocks) {
    if (threadIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
    return;
  }
  const long long dst_row = (long long)phys * kBlock + (g % kBlock);
  const int d = threadIdx.x;
  const int t0 = t - r + 1;
  const uint16_t *kv = static_cast<const uint16_t *>(a.kv);

  // pooling softmax over the r tokens of the group, per channel
  float lg[4];
  float mx = -INFINITY;
  for (int j = 0; j < r; ++j) {
    lg[j] = logits[(long long)(t0 + j) * D + d] + a.ape[j * D + d];
    mx = fmaxf(mx, lg[j]);
  }
  float s = 0.f, y = 0.f;
  for (int j = 0; j < r; ++j) {
    float e = expf(lg[j] - mx);
    s += e;
    y = fmaf(e, bf16_bits_to_float(kv[(long long)(t0 + j) * D + d]), y);
  }
  y = round_bf16(y / s);

  if (a.gamma) {
    float ss = block_sum(y * y, red);
    float inv = rsqrtf(ss / (float)D + a.rms_eps);
    y = round_bf16(y * inv *
                   bf16_bits_to_float(static_cast<const uint16_t *>(a.gamma)[d]));
  }

  if (a.rotate) {
    const int pos = g * r;
    ys[d] = y;
    __syncthreads();
    if (pos >= a.rope_cap) {
      if (d == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
    } else if (d >= D - kRopeDim) {
      const int i = (d - (D - kRopeDim)) >> 1;
      const float c = a.rope_cos[(long long)pos * kRopeHalf + i];
      const float sn = a.rope_sin[(long long)pos * kRopeHalf + i];
      if ((d & 1) == 0)
        y = ys[d] * c - ys[d + 1] * sn;
      else
        y = ys[d - 1] * sn + ys[d] * c;
    }
  }

  if (a.out_mode == CSA_OUT_BF16) {
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.cmp_pool);
    dst[dst_row * D + d] = __float2bfloat16_rn(y);
  } else {
    float amax = block_max(fabsf(y), red);
    float scale = fmaxf(amax, 1e-4f) / 127.0f;
    float q = rintf(y / scale);
    q = fminf(fmaxf(q, -127.f), 127.f);
    a.idx_pool[dst_row * D + d] = static_cast<int8_t>(q);
    if (d == 0) a.idx_scale_pool[dst_row] = scale;
  }
}

// ---------------------------------------------------------------------------
// Short chunks: one CTA per (group-end row, column tile) does the whole group.
// COLS = 64 for a BF16 slice of a wide row (no row-wide statistic needed), or
// COLS = d = 128 for the whole row (RMSNorm / INT8 amax inside the CTA).
// ---------------------------------------------------------------------------
constexpr int FC_THREADS = 256;
constexpr int FC_MAX_W_BYTES = 128 * 1024;

template <int COLS>
__global__ void __launch_bounds__(FC_THREADS) compress_fused_kernel(csa_compress_args a) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t fc_smem[];
  constexpr int PARTS = FC_THREADS / COLS;
  const int dx = a.dx, D = a.d, r = a.ratio;
  uint16_t *Ws = reinterpret_cast<uint16_t *>(fc_smem);               // [dx][COLS]
  uint16_t *Xs = Ws + (size_t)dx * COLS;                               // [r][dx]
  float *part = reinterpret_cast<float *>(Xs + 4 * dx);               // [PARTS][4][COLS]
  float *ys = part + PARTS * 4 * COLS;                                 // [COLS]
  float *red = ys + COLS;                                              // [32]
  const int t = blockIdx.y, c0 = blockIdx.x * COLS, tid = threadIdx.x;
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || p < 0 || (p % r) != r - 1 || t < r - 1) return;
  for (int j = 1; j < r; ++j)
    if (a.row_req[t - j] != b || a.positions[t - j] != p - j) return;
  if (b >= a.n_req) {
    if (tid == 0 && blockIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int g = p / r, page = g / kBlock;
  const int phys = page < a.max_blocks ? a.block_table[(long long)b * a.max_blocks + page] : -1;
  if (phys < 0 || phys >= a.n_blocks) {
    if (tid == 0 && blockIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
    return;
  }
  const int t0 = t - r + 1;
  // stage the weight slice and the group's x rows (all copies in flight at once)
  const uint16_t *wg = static_cast<const uint16_t *>(a.w_gate);
  const uint16_t *xg = static_cast<const uint16_t *>(a.x);
  for (int e = tid; e < dx * (COLS / 8); e += FC_THREADS) {
    const int k = e / (COLS / 8), q = e % (COLS / 8);
    tc::cp_async16(Ws + k * COLS + q * 8, wg + (long long)k * D + c0 + q * 8);
  }
  for (int e = tid; e < r * (dx / 8); e += FC_THREADS) {
    const int j = e / (dx / 8), q = e % (dx / 8);
    tc::cp_async16(Xs + j * dx + q * 8, xg + (long long)(t0 + j) * dx + q * 8);
  }
  tc::cp_async_wait_all();
  __syncthreads();
  // logits: thread (column c, part) sums its K range for the r rows
  {
    const int c = tid % COLS, pr = tid / COLS;
    const int k_lo = pr * (dx / PARTS), k_hi = k_lo + dx / PARTS;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = k_lo; k < k_hi; ++k) {
      const float w = bf16_bits_to_float(Ws[k * COLS + c]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < r) acc[j] = fmaf(bf16_bits_to_float(Xs[j * dx + k]), w, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[(pr * 4 + j) * COLS + c] = acc[j];
  }
  __syncthreads();
  const uint16_t *kv = static_cast<const uint16_t *>(a.kv);
  float y = 0.f;
  const int c = tid, d = c0 + c;
  if (c < COLS) {
    float lg[4];
    float mx = -INFINITY;
    for (int j = 0; j < r; ++j) {
      float l = a.ape[j * D + d];
      for (int pr = 0; pr < PARTS; ++pr) l += part[(pr * 4 + j) * COLS + c];
      lg[j] = l;
      mx = fmaxf(mx, l);
    }
    float s = 0.f;
    for (int j = 0; j < r; ++j) {
      const float e = expf(lg[j] - mx);
      s += e;
      y = fmaf(e, bf16_bits_to_float(kv[(long long)(t0 + j) * D + d]), y);
    }
    y = round_bf16(y / s);
  }
  // row-wide statistics exist only in the whole-row variant (COLS == D)
  if (a.gamma && COLS == D) {
    float v = c < COLS ? y * y : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    __syncthreads();
    float ss = 0.f;
    for (int i = 0; i < FC_THREADS / 32; ++i) ss += red[i];
    __syncthreads();
    if (c < COLS)
      y = round_bf16(y * rsqrtf(ss / (float)D + a.rms_eps) *
                     bf16_bits_to_float(static_cast<const uint16_t *>(a.gamma)[d]));
  }
  if (a.rotate) {
    const int pos = g * r;
    if (c < COLS) ys[c] = y;
    __syncthreads();
    if (pos >= a.rope_cap) {
      if (tid == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
    } else if (c < COLS && d >= D - kRopeDim) {
      const int i = (d - (D - kRopeDim)) >> 1;
      const float cs = a.rope_cos[(long long)pos * kRopeHalf + i];
      const float sn = a.rope_sin[(long long)pos * kRopeHalf + i];
      y = (d & 1) == 0 ? ys[c] * cs - ys[c + 1] * sn : ys[c - 1] * sn + ys[c] * cs;
    }
  }
  const long long dst_row = (long long)phys * kBlock + (g % kBlock);
  if (a.out_mode == CSA_OUT_BF16) {
    if (c < COLS) static_cast<__nv_bfloat16 *>(a.cmp_pool)[dst_row * D + d] = __float2bfloat16_rn(y);
  } else {
    float v = c < COLS ? fabsf(y) : 0.f;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((tid & 31) == 0) red[tid >> 5] = v;
    __syncthreads();
    float amax = 0.f;
    for (int i = 0; i < FC_THREADS / 32; ++i) amax = fmaxf(amax, red[i]);
    const float scale = fmaxf(amax, 1e-4f) / 127.0f;
    if (c < COLS) {
      const float q = fminf(fmaxf(rintf(y / scale), -127.f), 127.f);
      a.idx_pool[dst_row * D + d] = static_cast<int8_t>(q);
    }
    if (tid == 0) a.idx_scale_pool[dst_row] = scale;
  }
}

template <int COLS>
size_t fused_smem(const csa_compress_args &a) {
  return (size_t)a.dx * COLS * 2 + 4 * (size_t)a.dx * 2 +
         (FC_THREADS / COLS) * 4 * COLS * 4 + COLS * 4 + 32 * 4;
}

template <int COLS>
cudaError_t launch_fused(const csa_compress_args &a, cudaStream_t s) {
  const size_t smem = fused_smem<COLS>(a);
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(compress_fused_kernel<COLS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FC_MAX_W_BYTES + 32 * 1024);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  launch_begin(CSA_K_COMPRESS_POOL, s);
  const cudaError_t e = launch_kernel(compress_fused_kernel<COLS>, dim3(a.d / COLS, a.n_rows),
                                      dim3(FC_THREADS), smem, s, 0, false, a);
  launch_end(CSA_K_COMPRESS_POOL, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const csa_compress_args &a, float *logits, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  // short chunks (decode): one fused kernel per call
  if (a.n_rows <= 256) {
    if (a.d == 128 && (size_t)a.dx * 128 * 2 <= FC_MAX_W_BYTES) return launch_fused<128>(a, s);
    if (a.d == 512 && a.out_mode == CSA_OUT_BF16 && !a.gamma &&
        (size_t)a.dx * 64 * 2 <= FC_MAX_W_BYTES)
      return launch_fused<64>(a, s);
  }
  dim3 g1((a.d + GT_COLS - 1) / GT_COLS, (a.n_rows + GT_ROWS - 1) / GT_ROWS);
  launch_begin(CSA_K_COMPRESS_GATE, s);
  cudaError_t e = launch_kernel(gate_logits_kernel, g1, dim3(256), 0, s, 0, false,
                                static_cast<const uint16_t *>(a.x),
                                static_cast<const uint16_t *>(a.w_gate), logits, a.n_rows, a.dx,
                                a.d);
  launch_end(CSA_K_COMPRESS_GATE, s);
  if (e != cudaSuccess) return e;
  launch_begin(CSA_K_COMPRESS_POOL, s);
  e = launch_kernel(compress_pool_kernel, dim3(a.n_rows), dim3(a.d), 0, s, 0, false, a,
                    static_cast<const float *>(logits));
  launch_end(CSA_K_COMPRESS_POOL, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
