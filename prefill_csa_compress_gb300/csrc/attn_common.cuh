// Pieces shared by the two attention kernels (k_attn.cu: decode, split over a
// thread-block cluster; k_attn_prefill.cu: persistent prefill).  Both run the
// same tile: 128 candidates on the MMA's M side, the 64 heads on N,
//   S^T[c, h]  = K[c, :] . q_h              (A = gathered tile, K-major)
//   O^T[d, h] += sum_c K[c, d] P[c, h]      (A = same tile read MN-major)
// with S^T in TMEM columns [0, 64) and O^T (four 128-channel tiles) in
// [64, 320).  Softmax threads are (candidate c = TMEM lane, half of the heads).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace attn {

constexpr int CT = 128;  // candidates per tile
constexpr int S_COL = 0, O_COL = 64;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // move the running max only past a 2^8 growth

// shared-memory layout of a tile (1024-byte aligned base)
constexpr int OFF_Q = 0;                   // 8 chunks x (64 heads x 128 B), K-major swizzled
constexpr int OFF_KV = OFF_Q + 8 * 8192;   // 8 chunks x (128 cands x 128 B), K-major swizzled
constexpr int OFF_P = OFF_KV + 8 * 16384;  // P^T, MN-major: 128 cands x 64 heads
constexpr int OFF_MISC = OFF_P + 16384;

__device__ __forceinline__ uint32_t pack2(float x, float y) {
  __nv_bfloat162 v = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t *>(&v);
}

// P^T row c (one candidate): 64 heads as 8 swizzled 16-byte chunks.
__device__ __forceinline__ uint8_t *prow_chunk(uint8_t *P, int c, int j) {
  return P + (c >> 3) * 1024 + (c & 7) * 128 + ((j ^ (c & 7)) << 4);
}

// Column-wise reduction of x[0..31] over the 32 lanes (reduce-scatter):
// afterwards lane l holds the reduction of column l.
template <bool MAX>
__device__ __forceinline__ float warp_col_reduce32(const float (&x)[32]) {
  const int lane = threadIdx.x & 31;
  float a[16];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float keep = up ? x[16 + i] : x[i], send = up ? x[i] : x[16 + i];
      const float o = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  float b[8];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float keep = up ? a[8 + i] : a[i], send = up ? a[i] : a[8 + i];
      const float o = __shfl_xor_sync(0xffffffffu, send, 8);
      b[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  float c[4];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float keep = up ? b[4 + i] : b[i], send = up ? b[i] : b[4 + i];
      const float o = __shfl_xor_sync(0xffffffffu, send, 4);
      c[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  float d[2];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float keep = up ? c[2 + i] : c[i], send = up ? c[i] : c[2 + i];
      const float o = __shfl_xor_sync(0xffffffffu, send, 2);
      d[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  const bool up = lane & 1;
  const float keep = up ? d[1] : d[0], send = up ? d[0] : d[1];
  const float o = __shfl_xor_sync(0xffffffffu, send, 1);
  return MAX ? fmaxf(keep, o) : keep + o;
}

__device__ __forceinline__ void load32(const float *src, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = reinterpret_cast<const float4 *>(src)[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
}

// 2^t on the FMA pipe, for t <= 8 (keeps part of a tile's exponentials off
// the special-function unit, which bounds the softmax): t = n + f with n the
// nearest integer and f in [-1/2, 1/2]; 2^f is the degree-4 polynomial that
// interpolates it at the five Chebyshev nodes of [-1/2, 1/2] (relative error
// below 4e-6 in FP32 Horner form) and n is added to its exponent.  t is
// clamped at -125, so results below 2^-125 come out as 2^-125.
__device__ __forceinline__ float exp2_fma(float t) {
  t = fmaxf(t, -125.f);
  const float r = t + 12582912.f;  // 1.5 * 2^23: n in the low mantissa bits of r
  const float f = t - (r - 12582912.f);
  float p = 0.00966636837f;
  p = fmaf(p, f, 0.0559219755f);
  p = fmaf(p, f, 0.240223497f);
  p = fmaf(p, f, 0.693121016f);
  p = fmaf(p, f, 1.f);
  return __int_as_float(__float_as_int(p) + (__float_as_int(r) << 23));
}

// 2^t on the special-function unit (PTX ex2.approx.ftz).
__device__ __forceinline__ float exp2_sfu(float t) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

// Per-head softmax state of a row, in shared memory.
struct SoftState {
  alignas(16) float m[kHeads];     // running reference per head (log2 domain)
  alignas(16) float corr[kHeads];  // factor of the last move of the reference
  alignas(16) float red[4][kHeads];
};

// Softmax of one tile by the 256 threads of named barrier `bar` (thread =
// candidate c = qd*32 + lane, heads h0..h0+31), from this thread's raw
// logits x (S^T row c).  Moves the running reference of heads whose logits
// grew past 2^8 (rescaling the n_mt O^T tiles at TMEM column o_col unless this
// is the row's first tile, and this warp's partial denominators `lacc`), and
// writes P^T as BF16.  `ready()` runs (in every thread) before O^T or P is
// touched.  On return x holds the FP32 probabilities of this thread's
// candidate; the caller makes P visible to the MMA (fence, barrier) and adds
// the column sums of x to lacc.
template <typename Ready>
__device__ __forceinline__ void softmax_vals(uint32_t tmem, uint32_t o_col, int n_mt, int qd, int h0,
                                             bool valid, float sl2, bool first, SoftState *st,
                                             uint8_t *Ps, int bar, float &lacc, float (&x)[32],
                                             Ready &&ready) {
  const int lane = threadIdx.x & 31, c = qd * 32 + lane;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] *= sl2;
  float mref[32];
  load32(st->m + h0, mref);
  bool exceed = false;
  if (valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j) exceed |= x[j] > mref[j] + kRescaleLog2;
  }
  if (tc::bar_or(bar, 256, exceed)) {
    if (!valid) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = -INFINITY;
    }
    const float mx = warp_col_reduce32<true>(x);
    const int h = h0 + lane;
    st->red[qd][h] = mx;
    tc::bar_sync(bar, 256);
    const float mt = fmaxf(fmaxf(st->red[0][h], st->red[1][h]), fmaxf(st->red[2][h], st->red[3][h]));
    const float mo = st->m[h];
    float mn = mo, corr = 1.f;
    if (mo == -INFINITY) {
      mn = mt;
    } else if (mt > mo + kRescaleLog2) {
      mn = mt;
      corr = exp2f(mo - mt);
    }
    tc::bar_sync(bar, 256);
    if (qd == 0) {
      st->m[h] = mn;
      st->corr[h] = corr;
    }
    lacc *= corr;  // every warp's partial denominator of head h moves with it
    tc::bar_sync(bar, 256);
    load32(st->m + h0, mref);
    ready();
    if (!first) {
      float cr[32];
      load32(st->corr + h0, cr);
      bool any = false;
#pragma unroll
      for (int j = 0; j < 32; ++j) any |= cr[j] != 1.f;
      if (__any_sync(0xffffffffu, any)) {
        tc::tc_fence_after();
#pragma unroll 1
        for (int m4 = 0; m4 < n_mt; ++m4) {
          float v[32];
          const uint32_t addr = tmem + lane_off + o_col + m4 * 64 + h0;
          tc::tmem_ld32(addr, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= cr[j];
          tc::tmem_st32(addr, v);
        }
      }
    }
  } else {
    ready();
  }
  // P = 2^(x - m) as BF16 into the MN-major P^T rows (a valid candidate's
  // logits are at most m + 2^3 here, and its heads' references are finite:
  // any finite logit exceeds a reference of -inf); one in four
  // exponentials on the FMA pipe
  if (valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float t = x[j] - mref[j];
      x[j] = (j & 3) == 3 ? exp2_fma(t) : exp2_sfu(t);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 0.f;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4 *>(prow_chunk(Ps, c, (h0 >> 3) + q)) =
        make_uint4(pack2(x[8 * q], x[8 * q + 1]), pack2(x[8 * q + 2], x[8 * q + 3]),
                   pack2(x[8 * q + 4], x[8 * q + 5]), pack2(x[8 * q + 6], x[8 * q + 7]));
}

// The same, reading S^T from TMEM columns [0, 64) (O^T: four tiles at O_COL).
__device__ __forceinline__ void softmax_tile(uint32_t tmem, int qd, int h0, bool valid, float sl2,
                                             bool first, SoftState *st, uint8_t *Ps, int bar,
                                             float &lacc, float (&x)[32]) {
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  tc::tc_fence_after();
  tc::tmem_ld32(tmem + lane_off + S_COL + h0, x);
  softmax_vals(tmem, O_COL, 4, qd, h0, valid, sl2, first, st, Ps, bar, lacc, x, [] {});
}

// Rotate the RoPE chunk of the 64 q rows (the 128-byte swizzled K-major
// chunk holding channels 448..511, 128 bytes per head) by the row position's
// 32 cosines `cs` and sines `sn` (global or shared memory).
__device__ __forceinline__ void rope_q_rows(uint8_t *chunk, const float *cs, const float *sn,
                                            int tid, int nthreads) {
  for (int e = tid; e < kHeads * 8; e += nthreads) {
    const int h = e >> 3, jj = e & 7;
    uint4 *slot = reinterpret_cast<uint4 *>(chunk + h * 128 + ((jj ^ (h & 7)) << 4));
    const uint4 x4 = *slot;
    uint32_t w[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int pair = jj * 4 + q;
      const float c = cs[pair], s = sn[pair];
      const float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
      w[q] = pack2(x0 * c - x1 * s, x0 * s + x1 * c);
    }
    *slot = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster barrier, whole or split (arrive early, wait where it matters).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// Address of shared-memory address `la` (this CTA) in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr_u32(uint32_t la, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(la), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
  return peer_addr_u32(tc::smem_u32(p), rank);
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
// The tile's two contractions, issued by one warp (one elected lane).
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t kv, uint32_t qq, int kc) {
  constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, kHeads);
#pragma unroll
  for (int s = 0; s < 4; ++s)
    tc::mma_ss_elect(tmem + S_COL, tc::desc_sw128(kv + kc * 16384 + s * 32),
                     tc::desc_sw128(qq + kc * 8192 + s * 32), idesc_qk, (kc | s) != 0 ? 1u : 0u);
}

__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t kv, uint32_t pp, int mt,
                                         bool accumulate) {
  constexpr uint32_t idesc_pv = tc::idesc_bf16_f32_mn(128, kHeads);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    tc::mma_ss_elect(tmem + O_COL + mt * 64,
                     tc::desc_sw128_mn(kv + 2 * mt * 16384 + ks * 2048, 16384, 1024),
                     tc::desc_sw128_mn(pp + ks * 2048, 16384, 1024), idesc_pv,
                     (accumulate || ks > 0) ? 1u : 0u);
}

// Host: 2D BF16 tensor map [rows, 512] with a row stride of 1024 bytes, box
// {64 channels, box_rows}, 128-byte swizzle (the q rows of query rows).
bool encode_rows_map(CUtensorMap *map, const void *base, long long rows, int box_rows);

}  // namespace attn
}  // namespace csa
