// Gated compressor: gate logits GEMM, then per-group softmax pooling with the
// BF16 / RMSNorm / RoPE / INT8 epilogue.
//
// Source: "DeepSeek V4.1 Flash", "Compressor state ownership" (per-token KV and
// gate score of the same width, pooling softmax, BF16 rounding before RMSNorm)
// and "Serving-owned full RoPE tables" (group-start rotation); "DeepSeek
// V4-Flash, MTP point", "What is quantized" (INT8 on write, amax floored at
// 1e-4, scaled to 127).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include <algorithm>

#include "csa_internal.cuh"
#include "lowbit.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int kMaxRatio = 128;  // HCA

// ---------------------------------------------------------------------------
// Long chunks on the tensor cores: logits[t, d] = sum_k x[t, k] w_gate[k, d].
// One CTA per 128-row x 128-column tile of logits.  x tiles (K-major) and
// w_gate tiles (read as they lie, N-major: 64 columns of one k per 128-byte
// row) arrive by TMA into a 4-stage ring of 64-wide K chunks; one elected
// thread issues M = 128, N = 128, K = 16 BF16 MMAs into TMEM; four warps read
// the FP32 tile back (lane = row) and store it.
// ---------------------------------------------------------------------------
constexpr int GG_THREADS = 128;
constexpr int GG_M = 128, GG_N = 128, GG_K = 64, GG_STAGES = 4;
constexpr int GG_A_BYTES = GG_M * GG_K * 2;   // 16 KB
constexpr int GG_B_BYTES = GG_N * GG_K * 2;   // 16 KB: two 64-column groups of 8 KB
constexpr int GG_STAGE = GG_A_BYTES + GG_B_BYTES;
constexpr int GG_SMEM = GG_STAGES * GG_STAGE + 1024 + 256;

__global__ void __launch_bounds__(GG_THREADS, 1)
    gate_gemm_tc_kernel(float *__restrict__ logits, int n_rows, int dx, int d,
                        const __grid_constant__ CUtensorMap xmap,
                        const __grid_constant__ CUtensorMap wmap, uint32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + GG_STAGES * GG_STAGE);
  uint64_t *empty = full + GG_STAGES;
  uint64_t *acc_full = empty + GG_STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.y * GG_M, col0 = blockIdx.x * GG_N;
  const int n_k = dx / GG_K;
  if (tid == 0) {
    for (int i = 0; i < GG_STAGES; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, GG_N);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (warp == 0) {
    if (lane == 0)
      for (int kc = 0; kc < n_k && ok; ++kc) {
        const int st = kc % GG_STAGES;
        if (kc >= GG_STAGES && !tc::mbar_wait(&empty[st], ((kc / GG_STAGES) - 1) & 1)) {
          ok = false;
          break;
        }
        uint8_t *A = sm + st * GG_STAGE, *B = A + GG_A_BYTES;
        tc::mbar_arrive_expect_tx(&full[st], GG_STAGE);
        tc::tma_load_2d(A, &xmap, kc * GG_K, row0, &full[st]);
        tc::tma_load_2d(B, &wmap, col0, kc * GG_K, &full[st]);
        tc::tma_load_2d(B + GG_B_BYTES / 2, &wmap, col0 + 64, kc * GG_K, &full[st]);
      }
  } else if (warp == 1) {
    // A K-major, B N-major (w_gate rows are k)
    constexpr uint32_t idesc = tc::idesc_bf16_f32(GG_M, GG_N) | (1u << 16);
    for (int kc = 0; kc < n_k && ok; ++kc) {
      const int st = kc % GG_STAGES;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[st], (kc / GG_STAGES) & 1));
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t A = tc::smem_u32(sm + st * GG_STAGE), B = A + GG_A_BYTES;
#pragma unroll
      for (int k16 = 0; k16 < GG_K / 16; ++k16)
        tc::mma_ss_elect(tmem, tc::desc_sw128(A + k16 * 32),
                         tc::desc_sw128_mn(B + k16 * 2048, GG_B_BYTES / 2, 1024), idesc,
                         (kc | k16) != 0 ? 1u : 0u);
      tc::mma_commit_elect(&empty[st]);
    }
    tc::mma_commit_elect(acc_full);
  }
  __syncwarp();
  // ---- epilogue: lane = row, 128 FP32 columns
  if (!tc::mbar_wait(acc_full, 0)) {
    ok = false;
    if (tid == 0) flag(status, CSA_DEV_TIMEOUT);
  }
  tc::tc_fence_after();
  const int row = row0 + warp * 32 + lane;
#pragma unroll 1
  for (int c32 = 0; c32 < GG_N / 32; ++c32) {
    float v[32];
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c32 * 32, v);
    if (ok && row < n_rows) {
      float4 *dst = reinterpret_cast<float4 *>(logits + (long long)row * d + col0 + c32 * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, GG_N);
}

PFN_cuTensorMapEncodeTiled_v12000 gg_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

// 2D BF16 map [outer, inner] (row stride inner * 2 bytes), box {64, box_outer},
// 128-byte swizzle.
bool gg_map(CUtensorMap *map, const void *base, long long inner, long long outer, int box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = gg_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// The gate GEMM wants K in 64s, N in 128s and 16-byte-aligned operands, which
// the compressor's argument checks guarantee (d in {128, 512}, dx % 64 == 0).
cudaError_t launch_gate_gemm_tc(const csa_compress_args &a, float *logits, cudaStream_t s) {
  CUtensorMap xmap, wmap;
  memset(&xmap, 0, sizeof(xmap));
  memset(&wmap, 0, sizeof(wmap));
  if (!gg_map(&xmap, a.x, a.dx, a.n_rows, GG_M) || !gg_map(&wmap, a.w_gate, a.d, a.dx, GG_K))
    return cudaErrorInvalidValue;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(gate_gemm_tc_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, GG_SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const dim3 grid(a.d / GG_N, (a.n_rows + GG_M - 1) / GG_M);
  return launch_kernel(gate_gemm_tc_kernel, grid, dim3(GG_THREADS), (size_t)GG_SMEM, s, 0, false,
                       logits, a.n_rows, a.dx, a.d, xmap, wmap, a.status_dev);
}

// Output rows of the BF16 and INT8 publications through the pool's strides
// (bytes; the host makes them explicit), and the row's FP32 scale slot.
__device__ __forceinline__ __nv_bfloat16 *bf16_out_row(const csa_compress_args &a,
                                                      long long row) {
  return reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(a.cmp_pool) +
                                           pool_offset(row, a.pool_page_stride, a.pool_row_stride));
}
__device__ __forceinline__ int8_t *int8_out_row(const csa_compress_args &a, long long row) {
  return a.idx_pool + pool_offset(row, a.pool_page_stride, a.pool_row_stride);
}
__device__ __forceinline__ float *scale_out_slot(const csa_compress_args &a, long long row) {
  return reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.idx_scale_pool) +
                                   (row >> 7) * a.scale_page_stride + (row & 127) * 4);
}

// ---------------------------------------------------------------------------
// Long chunks, pooling: one CTA per row that closes a group (thread = channel)
// takes the group's logits, softmax over its r rows per channel, the pooled
// value and the BF16 / RMSNorm / RoPE / INT8 epilogue.
// ---------------------------------------------------------------------------
// Low-bit publication ("DeepSeek V4.1 Flash", production cache ABI; the
// rounding rules are the ones include/csa.h states) of channel d (value y)
// of pool row dst_row.  Called by every lane of a warp whose lanes hold
// consecutive channels, groups of G lanes aligned to G; `live` marks lanes
// that hold a channel.  G == 32: E8M0 scales; G == 16: E4M3 scales.
template <int G>
__device__ __forceinline__ void publish_fp4(const csa_compress_args &a, long long dst_row, int d,
                                            float y, bool live) {
  float v = live ? fabsf(y) : 0.f;
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  float scale;
  uint32_t sbyte;
  if constexpr (G == 32) {
    const int e = lowbit::e8m0_exponent(v);
    scale = lowbit::pow2f(e);
    sbyte = (uint32_t)(e + 127);
  } else {
    sbyte = lowbit::e4m3_scale_byte(v);
    scale = lowbit::e4m3_value(sbyte);
  }
  const uint32_t code = scale > 0.f ? lowbit::e2m1_code(__fdiv_rn(y, scale)) : 0u;
  const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
  const int D = a.d;
  if (live && (d & 1) == 0)
    static_cast<uint8_t *>(a.cmp_pool)[dst_row * (D / 2) + d / 2] = (uint8_t)(code | (hi << 4));
  if (live && d % G == 0) a.scale_pool[dst_row * (D / G) + d / G] = (uint8_t)sbyte;
}

// MXFP8 publication (the FP8 index plane read as MXFP8): one E4M3 code per
// channel, one E8M0 scale per group of 32 lanes (same calling rules as
// publish_fp4).
__device__ __forceinline__ void publish_mxfp8(const csa_compress_args &a, long long dst_row, int d,
                                              float y, bool live) {
  float v = live ? fabsf(y) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int e = lowbit::e8m0_exponent_448(v);
  const uint32_t code = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(y, lowbit::pow2f(e)),
                                                        __NV_SATFINITE, __NV_E4M3);
  const int D = a.d;
  if (live) static_cast<uint8_t *>(a.cmp_pool)[dst_row * D + d] = (uint8_t)code;
  if (live && d % 32 == 0) a.scale_pool[dst_row * (D / 32) + d / 32] = (uint8_t)(e + 127);
}

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

// One CTA per group-closing row (d threads, one channel each).  With a state
// ring, predecessors before the chunk start come from the ring: their kv row
// and their gate score (ape included) as the ring stores them.  The pooled
// window is the group's r tokens, or with `overlap` the previous group's too
// (n = min(p + 1, 2r) tokens ending at p), token q's score taking
// ape[q % r].
__device__ __forceinline__ void pool_row(const csa_compress_args &a,
                                         const float *__restrict__ logits, const int t, const int b,
                                         const int p) {
  __shared__ float ys[512];
  __shared__ float red[32];
  const int r = a.ratio, D = a.d;
  if (b >= a.n_req) {
    if (threadIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const float *ring = nullptr;  // this request's ring block
  if (a.state_cache) {
    const int blk = a.state_block_table[b];
    if (blk < 0) return;  // the request's compressor is disabled
    if (blk >= a.n_state_blocks) {
      if (threadIdx.x == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
      return;
    }
    ring = a.state_cache + (long long)blk * a.state_capacity * 2 * D;
  }
  // token j of the window (position p - n + 1 + j): row t - n + 1 + j of
  // this chunk, or (a position before the chunk start) the ring
  const int n = a.overlap ? min(p + 1, 2 * r) : r;
  __shared__ uint8_t in_chunk[kMaxRatio];
  __shared__ int s_complete;
  if (threadIdx.x == 0) s_complete = 1;
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int s = t - n + 1 + j;
    const bool here = s >= 0 && a.row_req[s] == b && a.positions[s] == p - n + 1 + j;
    in_chunk[j] = here;
    if (!here && !ring) s_complete = 0;
  }
  __syncthreads();
  if (!s_complete) return;  // the group is not complete in this chunk (uniform)
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
  const int t0 = t - n + 1, q0 = p - n + 1;
  const uint16_t *kv = static_cast<const uint16_t *>(a.kv);
  // gate score and kv value of token j for this channel
  auto token = [&](int j, float &lg, float &v) {
    if (in_chunk[j]) {
      lg = logits[(long long)(t0 + j) * D + d] + a.ape[((q0 + j) % r) * D + d];
      v = bf16_bits_to_float(kv[(long long)(t0 + j) * D + d]);
    } else {
      const float *slot = ring + (long long)((q0 + j) % a.state_capacity) * 2 * D;
      v = slot[d];
      lg = slot[D + d];
    }
  };

  // pooling softmax over the n tokens of the window, per channel, in one
  // pass over batches of 8 tokens (their loads in flight together; the
  // running maximum moves once per batch)
  float mx = -INFINITY, s = 0.f, y = 0.f;
  for (int j0 = 0; j0 < n; j0 += 8) {
    float lg[8], v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lg[i] = -INFINITY;
      v[i] = 0.f;
      if (j0 + i < n) token(j0 + i, lg[i], v[i]);
    }
    float mb = lg[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mb = fmaxf(mb, lg[i]);
    const float mn = fmaxf(mx, mb);
    const float c = expf(mx - mn);  // 0 for the first batch
    s *= c;
    y *= c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float e = expf(lg[i] - mn);  // 0 past the group's end
      s += e;
      y = fmaf(e, v[i], y);
    }
    mx = mn;
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
    bf16_out_row(a, dst_row)[d] = __float2bfloat16_rn(y);
  } else if (a.out_mode == CSA_OUT_FP4_E4M3) {
    publish_fp4<16>(a, dst_row, d, y, true);
  } else if (a.out_mode == CSA_OUT_FP4_E8M0) {
    publish_fp4<32>(a, dst_row, d, y, true);
  } else if (a.out_mode == CSA_OUT_MXFP8) {
    publish_mxfp8(a, dst_row, d, y, true);
  } else {
    float amax = block_max(fabsf(y), red);
    float scale = fmaxf(amax, 1e-4f) / 127.0f;
    float q = rintf(y / scale);
    q = fminf(fmaxf(q, -127.f), 127.f);
    int8_out_row(a, dst_row)[d] = static_cast<int8_t>(q);
    if (d == 0) *scale_out_slot(a, dst_row) = scale;
  }
}

// One CTA per row (long groups: HCA's ratio 128).
__global__ void compress_pool_kernel(csa_compress_args a, const float *__restrict__ logits) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int t = blockIdx.x;
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || p < 0 || (p % a.ratio) != a.ratio - 1) return;
  pool_row(a, logits, t, b, p);
}

// Short groups: a chunk's group-closing rows are one in every r, so a CTA
// takes rows_per_cta = r consecutive rows (their requests and positions
// loaded at once) and pools those that close a group.
constexpr int kPoolRows = 4;
__global__ void compress_pool_rows_kernel(csa_compress_args a, const float *__restrict__ logits,
                                          int rows_per_cta) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  __shared__ int rb[kPoolRows], rq[kPoolRows];
  const int t0 = blockIdx.x * rows_per_cta;
  const int m = min(rows_per_cta, a.n_rows - t0);
  if ((int)threadIdx.x < m) {
    rb[threadIdx.x] = a.row_req[t0 + threadIdx.x];
    rq[threadIdx.x] = a.positions[t0 + threadIdx.x];
  }
  __syncthreads();
  for (int i = 0; i < m; ++i) {
    const int b = rb[i], p = rq[i];
    if (b < 0 || p < 0 || (p % a.ratio) != a.ratio - 1) continue;  // uniform over the CTA
    pool_row(a, logits, t0 + i, b, p);
    __syncthreads();  // the row's shared state is no longer read
  }
}

// Long groups (HCA's ratio 128) without a row-wide statistic (no RMSNorm, no
// INT8 amax): one CTA per (group-closing row, 64-channel slice), 8 token
// lanes per channel.  Lane j takes tokens j, j + 8, ... of the group (their
// ring or chunk loads all in flight), keeps an online softmax of its share,
// and the 8 partial (max, sum, weighted sum) merge in shared memory; lanes 0
// then round, rotate and publish their 64 channels exactly as the per-row
// kernel does.  The per-row kernel walks the r tokens with one thread per
// channel, 8 tokens per round trip: 16 round trips for a 128-token group.
constexpr int WP_CH = 64, WP_LANES = 8, WP_THREADS = WP_CH * WP_LANES;
constexpr int WP_TOK = 16;  // tokens per lane held in flight (ratio <= WP_LANES * WP_TOK)

__global__ void __launch_bounds__(WP_THREADS)
    compress_pool_wide_kernel(csa_compress_args a, const float *__restrict__ logits) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  __shared__ float pm[WP_LANES][WP_CH], ps[WP_LANES][WP_CH], py[WP_LANES][WP_CH];
  __shared__ float ys[WP_CH];
  __shared__ uint8_t in_chunk[kMaxRatio];
  __shared__ int s_complete;
  const int slice = blockIdx.y;
  const int r = a.ratio, D = a.d;
  const int c = threadIdx.x % WP_CH, lane = threadIdx.x / WP_CH, d = slice * WP_CH + c;
  const uint16_t *kv = static_cast<const uint16_t *>(a.kv);
  // rows in a grid stride (a short chunk: at most one row per CTA)
  for (int t = blockIdx.x; t < a.n_rows; t += gridDim.x) {
    const int b = a.row_req[t], p = a.positions[t];
    if (b < 0 || p < 0 || (p % r) != r - 1) continue;  // uniform over the CTA
    if (b >= a.n_req) {
      if (threadIdx.x == 0 && slice == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
      continue;
    }
    const float *ring = nullptr;
    if (a.state_cache) {
      const int blk = a.state_block_table[b];
      if (blk < 0) continue;
      if (blk >= a.n_state_blocks) {
        if (threadIdx.x == 0 && slice == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
        continue;
      }
      ring = a.state_cache + (long long)blk * a.state_capacity * 2 * D;
    }
    __syncthreads();  // the previous row's shared state is no longer read
    if (threadIdx.x == 0) s_complete = 1;
    __syncthreads();
    for (int j = threadIdx.x; j < r; j += blockDim.x) {
      const int s = t - r + 1 + j;
      const bool here = s >= 0 && a.row_req[s] == b && a.positions[s] == p - r + 1 + j;
      in_chunk[j] = here;
      if (!here && !ring) s_complete = 0;
    }
    __syncthreads();
    if (!s_complete) continue;
    const int g = p / r, page = g / kBlock;
    int phys = -1;
    if (page < a.max_blocks) phys = a.block_table[(long long)b * a.max_blocks + page];
    if (phys < 0 || phys >= a.n_blocks) {
      if (threadIdx.x == 0 && slice == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
      continue;
    }
    const long long dst_row = (long long)phys * kBlock + (g % kBlock);
    const int t0 = t - r + 1;
    float lg[WP_TOK], v[WP_TOK];
#pragma unroll
    for (int i = 0; i < WP_TOK; ++i) {
      const int j = lane + WP_LANES * i;
      lg[i] = -INFINITY;
      v[i] = 0.f;
      if (j < r) {
        if (in_chunk[j]) {
          lg[i] = logits[(long long)(t0 + j) * D + d] + a.ape[j * D + d];
          v[i] = bf16_bits_to_float(kv[(long long)(t0 + j) * D + d]);
        } else {
          const float *slot = ring + (long long)((p - r + 1 + j) % a.state_capacity) * 2 * D;
          v[i] = slot[d];
          lg[i] = slot[D + d];
        }
      }
    }
    float mx = lg[0];
#pragma unroll
    for (int i = 1; i < WP_TOK; ++i) mx = fmaxf(mx, lg[i]);
    float sum = 0.f, y = 0.f;
#pragma unroll
    for (int i = 0; i < WP_TOK; ++i) {
      const float e = lg[i] == -INFINITY ? 0.f : expf(lg[i] - mx);
      sum += e;
      y = fmaf(e, v[i], y);
    }
    pm[lane][c] = mx;
    ps[lane][c] = sum;
    py[lane][c] = y;
    __syncthreads();
    if (lane == 0) {  // threads 0 .. 63: two full warps, channels in order
      float m = -INFINITY;
#pragma unroll
      for (int l = 0; l < WP_LANES; ++l) m = fmaxf(m, pm[l][c]);
      float S = 0.f, Y = 0.f;
#pragma unroll
      for (int l = 0; l < WP_LANES; ++l) {
        const float f = pm[l][c] == -INFINITY ? 0.f : expf(pm[l][c] - m);
        S = fmaf(ps[l][c], f, S);
        Y = fmaf(py[l][c], f, Y);
      }
      y = round_bf16(Y / S);
      if (a.rotate) {
        const int pos = g * r;
        ys[c] = y;
        asm volatile("bar.sync 1, 64;" ::: "memory");
        if (pos >= a.rope_cap) {
          if (c == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
        } else if (d >= D - kRopeDim) {
          const int i = (d - (D - kRopeDim)) >> 1;
          const float cs = a.rope_cos[(long long)pos * kRopeHalf + i];
          const float sn = a.rope_sin[(long long)pos * kRopeHalf + i];
          y = (d & 1) == 0 ? ys[c] * cs - ys[c + 1] * sn : ys[c - 1] * sn + ys[c] * cs;
        }
      }
      if (a.out_mode == CSA_OUT_BF16)
        bf16_out_row(a, dst_row)[d] = __float2bfloat16_rn(y);
      else if (a.out_mode == CSA_OUT_FP4_E4M3)
        publish_fp4<16>(a, dst_row, d, y, true);
      else if (a.out_mode == CSA_OUT_FP4_E8M0)
        publish_fp4<32>(a, dst_row, d, y, true);
      else
        publish_mxfp8(a, dst_row, d, y, true);
    }
  }
}

int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Short chunks only: a long chunk's grid would be mostly rows that close no
// group (measured: the per-row kernel is faster there, its idle CTAs cheaper
// than the wide kernel's row scan).
bool pool_wide(const csa_compress_args &a) {
  return a.n_rows <= 256 && !a.overlap && a.ratio > 16 && a.ratio <= WP_LANES * WP_TOK && !a.gamma &&
         a.out_mode != CSA_OUT_INT8 && a.d % WP_CH == 0;
}

// Ring writes of the state: row t among the last state_capacity rows of its
// request's chunk stores its kv row (FP32) and its gate score (ape included)
// in slot p % state_capacity.  Runs after the pooling kernel, so every ring
// read of the call precedes every write.  One CTA per row, d threads.
__device__ __forceinline__ void state_row(const csa_compress_args &a,
                                          const float *__restrict__ logits, const int t,
                                          const int d) {
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || b >= a.n_req || p < 0) return;
  const int blk = a.state_block_table[b];
  if (blk < 0 || blk >= a.n_state_blocks) return;  // flagged by the pooling kernel
  const int cap = a.state_capacity, D = a.d;
  if (t + cap < a.n_rows && a.row_req[t + cap] == b) return;  // not among the last cap rows
  float *slot = a.state_cache + ((long long)blk * cap + p % cap) * 2 * D;
  slot[d] = bf16_bits_to_float(static_cast<const uint16_t *>(a.kv)[(long long)t * D + d]);
  slot[D + d] = logits[(long long)t * D + d] + a.ape[(p % a.ratio) * D + d];
}

__global__ void compress_state_kernel(csa_compress_args a, const float *__restrict__ logits) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  state_row(a, logits, blockIdx.x, threadIdx.x);
}

// The ring writes of a layer's two compressors in one grid (blockIdx.y picks
// the compressor; each reads its own logits from its workspace).
__global__ void compress_state_pair_kernel(const __grid_constant__ csa_compress_args a,
                                           const __grid_constant__ csa_compress_args b) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const csa_compress_args *x = blockIdx.y == 0 ? &a : &b;
  if ((int)blockIdx.x >= x->n_rows || (int)threadIdx.x >= x->d) return;
  state_row(*x, static_cast<const float *>(x->workspace), blockIdx.x, threadIdx.x);
}

// Gate logits of a short chunk, row by row (the tensor-core GEMM's 128-row
// tiles would be mostly empty): one CTA per (16-column slice, row) stages its
// W_gate slice and the row's x, sums the K range split over its threads and
// writes logits[t, c] = x_t . w_gate[:, c] (FP32, ape not added).
constexpr int GR_THREADS = 256, GR_COLS = 16;
__global__ void __launch_bounds__(GR_THREADS) gate_rows_kernel(csa_compress_args a, float *logits) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t gr_smem[];
  constexpr int PARTS = GR_THREADS / GR_COLS;
  const int dx = a.dx, D = a.d, tid = threadIdx.x;
  const int c0 = blockIdx.x * GR_COLS, t = blockIdx.y;
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || b >= a.n_req || p < 0) return;  // no group or ring write reads this row
  uint16_t *Ws = reinterpret_cast<uint16_t *>(gr_smem);   // [dx][GR_COLS]
  uint16_t *Xs = Ws + (size_t)dx * GR_COLS;               // [dx]
  float *part = reinterpret_cast<float *>(Xs + dx);       // [PARTS][GR_COLS]
  const uint16_t *wg = static_cast<const uint16_t *>(a.w_gate);
  const uint16_t *xg = static_cast<const uint16_t *>(a.x) + (long long)t * dx;
  for (int e = tid; e < dx * (GR_COLS / 8); e += GR_THREADS) {
    const int k = e / (GR_COLS / 8), q = e % (GR_COLS / 8);
    tc::cp_async16(Ws + k * GR_COLS + q * 8, wg + (long long)k * D + c0 + q * 8);
  }
  for (int e = tid; e < dx / 8; e += GR_THREADS) tc::cp_async16(Xs + e * 8, xg + e * 8);
  tc::cp_async_wait_all();
  __syncthreads();
  const int c = tid % GR_COLS, pr = tid / GR_COLS;
  float acc = 0.f;
  for (int k = pr * (dx / PARTS); k < (pr + 1) * (dx / PARTS); ++k)
    acc = fmaf(bf16_bits_to_float(Xs[k]), bf16_bits_to_float(Ws[k * GR_COLS + c]), acc);
  part[pr * GR_COLS + c] = acc;
  __syncthreads();
  if (tid < GR_COLS) {
    float l = 0.f;
    for (int q = 0; q < PARTS; ++q) l += part[q * GR_COLS + tid];
    logits[(long long)t * D + c0 + tid] = l;
  }
}

// ---------------------------------------------------------------------------
// Short chunks: one CTA per (group-end row, column tile) does the whole group.
// COLS = 16 for a BF16 slice of a wide row (no row-wide statistic needed:
// narrow slices spread the W_gate loads over many SMs), or COLS = d = 128 for
// the whole row (RMSNorm / INT8 amax inside the CTA).  Once the CTA knows its
// group, every input it needs is requested at once (W_gate slice and x rows
// into shared memory; the block-table entry, kv, ape, RoPE and gamma entries
// into registers), so the group costs one memory round trip after the row
// check rather than one per dependent read.
// ---------------------------------------------------------------------------
constexpr int FC_THREADS = 256;
constexpr int FC_MAX_W_BYTES = 128 * 1024;

// RMSNorm (whole-row variant), rotation at the group start and publication
// of one pooled row (y: this thread's channel c = threadIdx.x < COLS).
template <int COLS>
__device__ __forceinline__ void fused_tail(const csa_compress_args &a, float y, const int cb,
                                           const float gam, const float cs, const float sn,
                                           const bool rope_ok, const bool rot_here, float *ys,
                                           float *red, const long long dst_row) {
  const int D = a.d, tid = threadIdx.x, c = tid, d = cb * COLS + c;
  // row-wide statistics exist only in the whole-row variant (COLS == D)
  if (a.gamma && COLS == D) {
    float v = c < COLS ? y * y : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    __syncthreads();
    float ss = 0.f;
    for (int i = 0; i < FC_THREADS / 32; ++i) ss += red[i];
    __syncthreads();
    if (c < COLS) y = round_bf16(y * rsqrtf(ss / (float)D + a.rms_eps) * gam);
  }
  if (a.rotate) {
    if (c < COLS) ys[c] = y;
    __syncthreads();
    if (!rope_ok) {
      if (tid == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
    } else if (rot_here) {
      y = (d & 1) == 0 ? ys[c] * cs - ys[c + 1] * sn : ys[c - 1] * sn + ys[c] * cs;
    }
  }
  if (a.out_mode == CSA_OUT_BF16) {
    if (c < COLS) bf16_out_row(a, dst_row)[d] = __float2bfloat16_rn(y);
  } else if (a.out_mode == CSA_OUT_FP4_E4M3) {
    publish_fp4<16>(a, dst_row, d, y, c < COLS);
  } else if (a.out_mode == CSA_OUT_FP4_E8M0) {
    publish_fp4<32>(a, dst_row, d, y, c < COLS);
  } else if (a.out_mode == CSA_OUT_MXFP8) {
    publish_mxfp8(a, dst_row, d, y, c < COLS);
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
      int8_out_row(a, dst_row)[d] = static_cast<int8_t>(q);
    }
    if (tid == 0) *scale_out_slot(a, dst_row) = scale;
  }
}

template <int COLS>
__device__ __forceinline__ void fused_group(const csa_compress_args &a, const int cb, const int t,
                                            uint8_t *fc_smem) {
  constexpr int PARTS = FC_THREADS / COLS;
  const int dx = a.dx, D = a.d, r = a.ratio, tid = threadIdx.x;
  uint16_t *Ws = reinterpret_cast<uint16_t *>(fc_smem);               // [dx][COLS]
  uint16_t *Xs = Ws + (size_t)dx * COLS;                               // [r][dx]
  float *part = reinterpret_cast<float *>(Xs + 4 * dx);               // [PARTS][4][COLS]
  float *ys = part + PARTS * 4 * COLS;                                 // [COLS]
  float *red = ys + COLS;                                              // [32]
  const int c0 = cb * COLS;
  // does row t close a group of r consecutive positions of one request?
  int bj[4], pj[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tj = max(t - j, 0);
    bj[j] = j < r ? a.row_req[tj] : 0;
    pj[j] = j < r ? a.positions[tj] : 0;
  }
  const int b = bj[0], p = pj[0];
  if (b < 0 || p < 0 || (p % r) != r - 1 || t < r - 1) return;
#pragma unroll
  for (int j = 1; j < 4; ++j)
    if (j < r && (bj[j] != b || pj[j] != p - j)) return;
  if (b >= a.n_req) {
    if (tid == 0 && cb == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int g = p / r, page = g / kBlock, t0 = t - r + 1;
  // ---- every input of the group in flight at once
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
  const int phys = page < a.max_blocks ? a.block_table[(long long)b * a.max_blocks + page] : -1;
  const int c = tid, d = c0 + c;
  const int pos = g * r;  // RoPE position: the group start
  const bool rope_ok = pos < a.rope_cap;
  const bool rot_here = a.rotate && rope_ok && c < COLS && d >= D - kRopeDim;
  const uint16_t *kvg = static_cast<const uint16_t *>(a.kv);
  uint16_t kvj[4] = {0, 0, 0, 0};
  float apej[4] = {0.f, 0.f, 0.f, 0.f};
  float cs = 1.f, sn = 0.f, gam = 1.f;
  if (c < COLS) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < r) {
        kvj[j] = kvg[(long long)(t0 + j) * D + d];
        apej[j] = a.ape[j * D + d];
      }
    if (rot_here) {
      const int i = (d - (D - kRopeDim)) >> 1;
      cs = a.rope_cos[(long long)pos * kRopeHalf + i];
      sn = a.rope_sin[(long long)pos * kRopeHalf + i];
    }
    if (a.gamma && COLS == D) gam = bf16_bits_to_float(static_cast<const uint16_t *>(a.gamma)[d]);
  }
  tc::cp_async_wait_all();
  __syncthreads();
  if (phys < 0 || phys >= a.n_blocks) {  // the same for every thread of the CTA
    if (tid == 0 && cb == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
    return;
  }
  // ---- logits: thread (column c, part) sums its K range for the r rows
  {
    const int cc = tid % COLS, pr = tid / COLS;
    const int k_lo = pr * (dx / PARTS), k_hi = pr == PARTS - 1 ? dx : k_lo + dx / PARTS;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = k_lo; k < k_hi; ++k) {
      const float w = bf16_bits_to_float(Ws[k * COLS + cc]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < r) acc[j] = fmaf(bf16_bits_to_float(Xs[j * dx + k]), w, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[(pr * 4 + j) * COLS + cc] = acc[j];
  }
  __syncthreads();
  // ---- softmax over the r positions of each channel, pooled kv, BF16 round
  float y = 0.f;
  if (c < COLS) {
    float lg[4];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < r) {
        float l = apej[j];
        for (int pr = 0; pr < PARTS; ++pr) l += part[(pr * 4 + j) * COLS + c];
        lg[j] = l;
        mx = fmaxf(mx, l);
      }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < r) {
        const float e = expf(lg[j] - mx);
        s += e;
        y = fmaf(e, bf16_bits_to_float(kvj[j]), y);
      }
    y = round_bf16(y / s);
  }
  fused_tail<COLS>(a, y, cb, gam, cs, sn, rope_ok, rot_here, ys, red,
                   (long long)phys * kBlock + (g % kBlock));
}

// The short-chunk kernel with a state ring: row t's CTA computes its own gate
// logit when the row is among the last state_capacity rows of its request
// (into the workspace, FP32 without ape, for the ring-write kernel that runs
// after every read of the call), and when t closes a group it pools the
// window's tokens: rows of this chunk from x and kv, earlier positions from
// the ring (kv row and score with ape, as stored).  The window is the r
// tokens of the group, or with `overlap` the n = min(p + 1, 2r) tokens
// ending at p; n <= FR_NJ.
constexpr int FR_NJ = 8;

template <int COLS>
__device__ __forceinline__ void fused_group_ring(const csa_compress_args &a, const int cb,
                                                 const int t, uint8_t *fc_smem) {
  constexpr int PARTS = FC_THREADS / COLS;
  const int dx = a.dx, D = a.d, r = a.ratio, tid = threadIdx.x;
  uint16_t *Ws = reinterpret_cast<uint16_t *>(fc_smem);               // [dx][COLS]
  uint16_t *Xs = Ws + (size_t)dx * COLS;                               // [FR_NJ][dx]
  float *part = reinterpret_cast<float *>(Xs + FR_NJ * dx);           // [PARTS][FR_NJ][COLS]
  float *ys = part + PARTS * FR_NJ * COLS;                             // [COLS]
  float *red = ys + COLS;                                              // [32]
  const int c0 = cb * COLS;
  const int b = a.row_req[t], p = a.positions[t];
  if (b < 0 || p < 0) return;
  const bool closing = (p % r) == r - 1;
  if (b >= a.n_req) {
    if (closing && tid == 0 && cb == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int blk = a.state_block_table[b];
  if (blk < 0) return;  // the request's compressor is disabled
  if (blk >= a.n_state_blocks) {
    if (closing && tid == 0 && cb == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
    return;
  }
  const int cap = a.state_capacity;
  const bool writer = !(t + cap < a.n_rows && a.row_req[t + cap] == b);
  if (!closing && !writer) return;
  const int n = closing ? (a.overlap ? min(p + 1, 2 * r) : r) : 1;
  const int t0 = t - n + 1, q0 = p - n + 1;
  // bit j: token j of the window (position q0 + j) is row t0 + j of this chunk
  uint32_t here = 0;
#pragma unroll
  for (int j = 0; j < FR_NJ; ++j) {
    if (j >= n) break;
    const int sj = t0 + j;
    if (sj >= 0 && a.row_req[sj] == b && a.positions[sj] == q0 + j) here |= 1u << j;
  }
  const float *ring = a.state_cache + (long long)blk * cap * 2 * D;
  // ---- every input in flight at once
  const uint16_t *wg = static_cast<const uint16_t *>(a.w_gate);
  const uint16_t *xg = static_cast<const uint16_t *>(a.x);
  for (int e = tid; e < dx * (COLS / 8); e += FC_THREADS) {
    const int k = e / (COLS / 8), q = e % (COLS / 8);
    tc::cp_async16(Ws + k * COLS + q * 8, wg + (long long)k * D + c0 + q * 8);
  }
  for (int e = tid; e < n * (dx / 8); e += FC_THREADS) {
    const int j = e / (dx / 8), q = e % (dx / 8);
    if ((here >> j) & 1u) tc::cp_async16(Xs + j * dx + q * 8, xg + (long long)(t0 + j) * dx + q * 8);
  }
  const int g = p / r, page = g / kBlock;
  int phys = -1;
  if (closing && page < a.max_blocks) phys = a.block_table[(long long)b * a.max_blocks + page];
  const int c = tid, d = c0 + c;
  const int pos = g * r;  // RoPE position: the group start
  const bool rope_ok = pos < a.rope_cap;
  const bool rot_here = a.rotate && rope_ok && c < COLS && d >= D - kRopeDim;
  const uint16_t *kvg = static_cast<const uint16_t *>(a.kv);
  // per token: its kv value and the part of its score known before the dot
  // product (ape for a chunk row, the whole stored score for a ring slot)
  float kvj[FR_NJ], basej[FR_NJ];
  float cs = 1.f, sn = 0.f, gam = 1.f;
#pragma unroll
  for (int j = 0; j < FR_NJ; ++j) {
    kvj[j] = 0.f;
    basej[j] = -INFINITY;
  }
  if (c < COLS && closing) {
#pragma unroll
    for (int j = 0; j < FR_NJ; ++j) {
      if (j >= n) break;
      if ((here >> j) & 1u) {
        kvj[j] = bf16_bits_to_float(kvg[(long long)(t0 + j) * D + d]);
        basej[j] = a.ape[((q0 + j) % r) * D + d];
      } else {
        const float *slot = ring + (long long)((q0 + j) % cap) * 2 * D;
        kvj[j] = slot[d];
        basej[j] = slot[D + d];
      }
    }
    if (rot_here) {
      const int i = (d - (D - kRopeDim)) >> 1;
      cs = a.rope_cos[(long long)pos * kRopeHalf + i];
      sn = a.rope_sin[(long long)pos * kRopeHalf + i];
    }
    if (a.gamma && COLS == D) gam = bf16_bits_to_float(static_cast<const uint16_t *>(a.gamma)[d]);
  }
  tc::cp_async_wait_all();
  __syncthreads();
  bool publish = closing;
  if (closing && (phys < 0 || phys >= a.n_blocks)) {  // the same for every thread of the CTA
    if (tid == 0 && cb == 0) flag(a.status_dev, CSA_DEV_BAD_BLOCK);
    publish = false;
    if (!writer) return;
  }
  // ---- logits of the window's chunk rows: thread (column, part) sums its K range
  {
    const int cc = tid % COLS, pr = tid / COLS;
    const int k_lo = pr * (dx / PARTS), k_hi = pr == PARTS - 1 ? dx : k_lo + dx / PARTS;
    float acc[FR_NJ];
#pragma unroll
    for (int j = 0; j < FR_NJ; ++j) acc[j] = 0.f;
    for (int k = k_lo; k < k_hi; ++k) {
      const float w = bf16_bits_to_float(Ws[k * COLS + cc]);
#pragma unroll
      for (int j = 0; j < FR_NJ; ++j)
        if ((here >> j) & 1u) acc[j] = fmaf(bf16_bits_to_float(Xs[j * dx + k]), w, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < FR_NJ; ++j)
      if ((here >> j) & 1u) part[(pr * FR_NJ + j) * COLS + cc] = acc[j];
  }
  __syncthreads();
  float y = 0.f;
  if (c < COLS) {
    float lg[FR_NJ];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < FR_NJ; ++j) {
      lg[j] = -INFINITY;
      if (j >= n) continue;
      if ((here >> j) & 1u) {
        float l = 0.f;
        for (int pr = 0; pr < PARTS; ++pr) l += part[(pr * FR_NJ + j) * COLS + c];
        if (j == n - 1 && writer) static_cast<float *>(a.workspace)[(long long)t * D + d] = l;
        lg[j] = l + basej[j];
      } else {
        lg[j] = basej[j];
      }
      mx = fmaxf(mx, lg[j]);
    }
    if (publish) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < FR_NJ; ++j) {
        if (j >= n) continue;
        const float e = expf(lg[j] - mx);
        sum += e;
        y = fmaf(e, kvj[j], y);
      }
      y = round_bf16(y / sum);
    }
  }
  if (!publish) return;  // uniform over the CTA
  fused_tail<COLS>(a, y, cb, gam, cs, sn, rope_ok, rot_here, ys, red,
                   (long long)phys * kBlock + (g % kBlock));
}

template <int COLS, bool RING>
__device__ __forceinline__ void fused_dispatch(const csa_compress_args &a, const int cb,
                                               const int t, uint8_t *fc_smem) {
  if constexpr (RING)
    fused_group_ring<COLS>(a, cb, t, fc_smem);
  else
    fused_group<COLS>(a, cb, t, fc_smem);
}

template <int COLS, bool RING>
__global__ void __launch_bounds__(FC_THREADS)
    compress_fused_kernel(const __grid_constant__ csa_compress_args a) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t fc_smem[];
  fused_dispatch<COLS, RING>(a, blockIdx.x, blockIdx.y, fc_smem);
}

// Two compressors of one layer (the main KV compressor and the index-key
// compressor read the same rows) in one grid: column tiles [0, n_a) serve the
// first, the rest the second.
template <int CA, int CB, bool RING>
__global__ void __launch_bounds__(FC_THREADS)
    compress_fused_pair_kernel(const __grid_constant__ csa_compress_args a,
                               const __grid_constant__ csa_compress_args b, int n_a) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t fc_smem[];
  const int x = blockIdx.x, t = blockIdx.y;
  if (x < n_a) {
    if (t < a.n_rows) fused_dispatch<CA, RING>(a, x, t, fc_smem);
  } else if (t < b.n_rows) {
    fused_dispatch<CB, RING>(b, x - n_a, t, fc_smem);
  }
}

template <int COLS, bool RING>
size_t fused_smem(const csa_compress_args &a) {
  const size_t nj = RING ? FR_NJ : 4;
  return (size_t)a.dx * COLS * 2 + nj * (size_t)a.dx * 2 +
         (FC_THREADS / COLS) * nj * COLS * 4 + COLS * 4 + 32 * 4;
}

// the short-chunk column tile for this call, or 0 when it takes the long path
// (with a ring: windows of at most FR_NJ tokens; without one: no overlap)
int fused_cols(const csa_compress_args &a) {
  if (a.n_rows > 256 || a.ratio > 4) return 0;
  if (a.state_cache ? (a.overlap ? 2 : 1) * a.ratio > FR_NJ : a.overlap) return 0;
  if (a.d == 128 && (size_t)a.dx * 128 * 2 <= FC_MAX_W_BYTES) return 128;
  // the 16-column tiles of d = 512 publish BF16 or E4M3-scaled groups of 16
  if (a.d == 512 && (a.out_mode == CSA_OUT_BF16 || a.out_mode == CSA_OUT_FP4_E4M3) && !a.gamma &&
      (size_t)a.dx * 16 * 2 <= FC_MAX_W_BYTES)
    return 16;
  return 0;
}

// The dynamic shared-memory limit is raised once per kernel and device
// (CB == 0: the single-compressor kernel of column tile CA).
template <int CA, int CB, bool RING>
cudaError_t allow_fused_smem() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e;
  if constexpr (CB == 0)
    e = cudaFuncSetAttribute(compress_fused_kernel<CA, RING>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, FC_MAX_W_BYTES + 32 * 1024);
  else
    e = cudaFuncSetAttribute(compress_fused_pair_kernel<CA, CB, RING>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, FC_MAX_W_BYTES + 32 * 1024);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <int COLS, bool RING>
cudaError_t launch_fused(const csa_compress_args &a, cudaStream_t s) {
  cudaError_t e = allow_fused_smem<COLS, 0, RING>();
  if (e != cudaSuccess) return e;
  launch_begin(CSA_K_COMPRESS_FUSED, s);
  e = launch_kernel(compress_fused_kernel<COLS, RING>, dim3(a.d / COLS, a.n_rows),
                    dim3(FC_THREADS), fused_smem<COLS, RING>(a), s, 0, false, a);
  launch_end(CSA_K_COMPRESS_FUSED, s);
  if (e == cudaSuccess && RING) {  // ring writes after every read of the call
    launch_begin(CSA_K_COMPRESS_POOL, s);
    e = launch_kernel(compress_state_kernel, dim3(a.n_rows), dim3(a.d), 0, s, 0, false, a,
                      static_cast<const float *>(a.workspace));
    launch_end(CSA_K_COMPRESS_POOL, s);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int CA, int CB, bool RING>
cudaError_t launch_fused_pair(const csa_compress_args &a, const csa_compress_args &b,
                              cudaStream_t s) {
  cudaError_t e = allow_fused_smem<CA, CB, RING>();
  if (e != cudaSuccess) return e;
  const int n_a = a.d / CA, n_b = b.d / CB;
  const size_t sa = fused_smem<CA, RING>(a), sb = fused_smem<CB, RING>(b);
  const int rows = a.n_rows > b.n_rows ? a.n_rows : b.n_rows;
  launch_begin(CSA_K_COMPRESS_FUSED, s);
  e = launch_kernel(compress_fused_pair_kernel<CA, CB, RING>, dim3(n_a + n_b, rows),
                    dim3(FC_THREADS), sa > sb ? sa : sb, s, 0, false, a, b, n_a);
  launch_end(CSA_K_COMPRESS_FUSED, s);
  if (e == cudaSuccess && RING) {  // both rings' writes after every read of the call
    launch_begin(CSA_K_COMPRESS_POOL, s);
    e = launch_kernel(compress_state_pair_kernel, dim3(rows, 2), dim3(a.d > b.d ? a.d : b.d), 0,
                      s, 0, false, a, b);
    launch_end(CSA_K_COMPRESS_POOL, s);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const csa_compress_args &a, float *logits, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  // short chunks (decode): one fused kernel per call (and the ring writes)
  const int cols = fused_cols(a);
  if (a.state_cache) {
    if (cols == 128) return launch_fused<128, true>(a, s);
    if (cols == 16) return launch_fused<16, true>(a, s);
  } else {
    if (cols == 128) return launch_fused<128, false>(a, s);
    if (cols == 16) return launch_fused<16, false>(a, s);
  }
  if (a.dx % GG_K != 0 || a.d % GG_N != 0 || (reinterpret_cast<uintptr_t>(logits) & 15u) != 0)
    return cudaErrorInvalidValue;
  cudaError_t e;
  launch_begin(CSA_K_COMPRESS_GATE, s);
  if (a.n_rows <= 256) {
    // a short chunk with a state ring: gate logits row by row
    const size_t smem = (size_t)a.dx * GR_COLS * 2 + (size_t)a.dx * 2 +
                        (GR_THREADS / GR_COLS) * GR_COLS * 4;
    e = launch_kernel(gate_rows_kernel, dim3(a.d / GR_COLS, a.n_rows), dim3(GR_THREADS), smem, s,
                      0, false, a, logits);
  } else {
    e = launch_gate_gemm_tc(a, logits, s);
  }
  launch_end(CSA_K_COMPRESS_GATE, s);
  if (e != cudaSuccess) return e;
  launch_begin(CSA_K_COMPRESS_POOL, s);
  if (pool_wide(a))
    e = launch_kernel(compress_pool_wide_kernel, dim3(std::min(a.n_rows, 2 * device_sm_count()),
                                                      a.d / WP_CH),
                      dim3(WP_THREADS), 0, s, 0, false, a, static_cast<const float *>(logits));
  else if (a.ratio <= kPoolRows)
    e = launch_kernel(compress_pool_rows_kernel, dim3((a.n_rows + a.ratio - 1) / a.ratio),
                      dim3(a.d), 0, s, 0, false, a, static_cast<const float *>(logits), a.ratio);
  else
    e = launch_kernel(compress_pool_kernel, dim3(a.n_rows), dim3(a.d), 0, s, 0, false, a,
                      static_cast<const float *>(logits));
  launch_end(CSA_K_COMPRESS_POOL, s);
  if (e == cudaSuccess && a.state_cache) {
    launch_begin(CSA_K_COMPRESS_POOL, s);
    e = launch_kernel(compress_state_kernel, dim3(a.n_rows), dim3(a.d), 0, s, 0, false, a,
                      static_cast<const float *>(logits));
    launch_end(CSA_K_COMPRESS_POOL, s);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_compress_pair(const csa_compress_args &a, float *logits_a,
                                 const csa_compress_args &b, float *logits_b, cudaStream_t s) {
  const int ca = a.n_rows > 0 ? fused_cols(a) : -1, cb = b.n_rows > 0 ? fused_cols(b) : -1;
  if (!a.state_cache && !b.state_cache) {
    if (ca == 16 && cb == 128) return launch_fused_pair<16, 128, false>(a, b, s);
    if (ca == 128 && cb == 16) return launch_fused_pair<128, 16, false>(a, b, s);
    if (ca == 128 && cb == 128) return launch_fused_pair<128, 128, false>(a, b, s);
    if (ca == 16 && cb == 16) return launch_fused_pair<16, 16, false>(a, b, s);
  } else if (a.state_cache && b.state_cache) {
    // the layer's main (d = 512) and index-key (d = 128) compressors
    if (ca == 16 && cb == 128) return launch_fused_pair<16, 128, true>(a, b, s);
    if (ca == 128 && cb == 128) return launch_fused_pair<128, 128, true>(a, b, s);
  }
  const cudaError_t e = launch_compress(a, logits_a, s);
  return e != cudaSuccess ? e : launch_compress(b, logits_b, s);
}

}  // namespace csa
