// Shared-KV sparse attention with an attention sink on the tcgen05 tensor
// cores.  Candidates of a query row are its selected compressed entries
// followed by its raw causal window; each candidate row is both key and value.
//
// Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2),
// "二阶段 CP 总体算法" (Stage-2 sparse attention with sinks, softmax_scale,
// ori_win_left = 127; outputs out and lse), "9.1" (candidate list = window KV
// and selected compressed KV) and "7. Window KV Halo" (window includes self).
//
// GB300 mapping.  Every contraction is an M=128 tcgen05.mma with the 128
// CANDIDATES of a tile on the M side and the 64 heads on the N side:
//   S^T[c, h] = K[c, :] . q_h          (A = gathered tile, K-major; B = q, K-major)
//   O^T[d, h] += sum_c K[c, d] P[c, h]  (A = the same tile read MN-major; B = P^T, MN-major)
// so the gathered tile is staged once in shared memory and serves as key and
// as value.  The tile is gathered row by row with cp.async straight into the
// 128-byte-swizzled layout the MMA reads.  Softmax statistics per head reduce
// across TMEM lanes through a small shared transpose; the running maximum is
// only moved (and O^T rescaled in TMEM) when it grows by more than 2^8, so the
// common case never touches the accumulator.  Decode splits a row's
// candidates over CTAs (one 128-candidate tile each) and merges the partial
// softmaxes in a second kernel; prefill keeps a row in one CTA and writes the
// output directly.
#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int AT_THREADS = 128;
constexpr int CT = 128;  // candidates per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // move the running max only past a 2^8 growth

constexpr int OFF_Q = 0;                      // 64 heads x 512 bf16, K-major: 8 chunks x 8 KB
constexpr int OFF_KV = OFF_Q + 8 * 8192;      // 128 cands x 512 bf16: 8 chunks x 16 KB
constexpr int OFF_P = OFF_KV + 8 * 16384;     // P^T, MN-major: 128 cands x 64 heads bf16
constexpr int OFF_MISC = OFF_P + 16384;
constexpr int ATTN_SMEM = OFF_MISC + 4096 + 1024;
constexpr uint32_t ATTN_TMEM_COLS = 512;      // S^T: cols [0,64); O^T tile m: [64+64m, 128+64m)
constexpr int REC_FLOATS = kHeads * kHeadDim + 2 * kHeads;  // partial record per (row, split)

struct AttnMisc {
  uint64_t bar_qk;
  uint64_t bar_pv;
  uint32_t tmem_base;
  int any_rescale;
  const uint16_t *rowp[CT];
  float m_ref[kHeads];  // running reference (log2 domain)
  float l_acc[kHeads];
  float corr[kHeads];
  float red[2][kHeads];
  float red4[4][kHeads];
};

__device__ __forceinline__ const uint16_t *candidate_row(const csa_attn_args &a, int t, int b,
                                                        int p, int V, int gi) {
  if (gi < a.topk) {
    const int c = a.topk_idx[(long long)t * a.topk + gi];
    if (c < 0) return nullptr;
    if (c >= V) {
      flag(a.status_dev, CSA_DEV_BAD_INDEX);
      return nullptr;
    }
    const long long row =
        page_row(a.cmp_block_table, a.cmp_max_blocks, a.cmp_n_blocks, b, c, a.status_dev);
    return row < 0 ? nullptr : static_cast<const uint16_t *>(a.cmp_pool) + row * kHeadDim;
  }
  const int pp = p - a.window + 1 + (gi - a.topk);
  if (pp < 0) return nullptr;
  if (pp >= a.kv_len[b]) {
    flag(a.status_dev, CSA_DEV_BAD_POS);
    return nullptr;
  }
  const long long row =
      page_row(a.kv_block_table, a.kv_max_blocks, a.kv_n_blocks, b, pp, a.status_dev);
  return row < 0 ? nullptr : static_cast<const uint16_t *>(a.kv_pool) + row * kHeadDim;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// P^T buffer: row c (one candidate) holds 64 heads as 8 swizzled 16-byte chunks.
__device__ __forceinline__ uint8_t *prow_chunk(uint8_t *P, int c, int j) {
  return P + (c >> 3) * 1024 + (c & 7) * 128 + ((j ^ (c & 7)) << 4);
}

__device__ __forceinline__ float p_at(const uint8_t *P, int c, int h) {
  const uint16_t v = *reinterpret_cast<const uint16_t *>(
      P + (c >> 3) * 1024 + (c & 7) * 128 + (((h >> 3) ^ (c & 7)) << 4) + (h & 7) * 2);
  return bf16_bits_to_float(v);
}

// Column sums of x[0..63] over the 32 lanes of a warp by a butterfly
// reduce-scatter: afterwards lane l holds the warp sums of columns 2l, 2l+1.
__device__ __forceinline__ float2 warp_colsum64(const float (&x)[64]) {
  const int lane = threadIdx.x & 31;
  float a[32];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float send = up ? x[i] : x[32 + i];
      a[i] = (up ? x[32 + i] : x[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  float b[16];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? a[i] : a[16 + i];
      b[i] = (up ? a[16 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  float c[8];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = up ? b[i] : b[8 + i];
      c[i] = (up ? b[8 + i] : b[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  float d[4];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = up ? c[i] : c[4 + i];
      d[i] = (up ? c[4 + i] : c[i]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
  }
  const bool up = lane & 1;
  const float s0 = (up ? d[2] : d[0]) + __shfl_xor_sync(0xffffffffu, up ? d[0] : d[2], 1);
  const float s1 = (up ? d[3] : d[1]) + __shfl_xor_sync(0xffffffffu, up ? d[1] : d[3], 1);
  return make_float2(s0, s1);
}

__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, uint32_t *status) {
  if (tc::mbar_wait(bar, parity)) return true;
  flag(status, CSA_DEV_TIMEOUT);
  return false;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_tc_kernel(csa_attn_args a, int n_splits, int tiles_per_split, float *__restrict__ partials) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t *Qs = sm + OFF_Q;
  uint8_t *KVs = sm + OFF_KV;
  uint8_t *Ps = sm + OFF_P;
  AttnMisc *M = reinterpret_cast<AttnMisc *>(sm + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t = blockIdx.y, split = blockIdx.x;
  const int b = a.row_req[t];
  if (b < 0) return;
  if (b >= a.n_req) {
    if (tid == 0 && split == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int p = a.row_pos[t];
  const int V = min(visible_count(p, a.ratio, a.n_cmp[b]), a.cmp_max_blocks * kBlock);
  const int n_cand = a.topk + a.window;
  const int g_begin = split * tiles_per_split * CT;
  const int g_end = min(n_cand, g_begin + tiles_per_split * CT);

  if (tid == 0) {
    tc::mbar_init(&M->bar_qk, 1);
    tc::mbar_init(&M->bar_pv, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(&M->tmem_base, ATTN_TMEM_COLS);
  if (tid < kHeads) {
    M->m_ref[tid] = -INFINITY;
    M->l_acc[tid] = 0.f;
  }

  // ---- q rotated at p (FP32), rounded to BF16, K-major swizzled
  bool rot = a.rope_cos != nullptr && p >= 0;
  if (rot && p >= a.rope_cap) {
    rot = false;
    if (tid == 0 && split == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
  }
  const uint16_t *qg = static_cast<const uint16_t *>(a.q) + (long long)t * kHeads * kHeadDim;
  // all 4096 16-byte pieces in flight at once, straight into the swizzled layout
  for (int e = tid; e < kHeads * (kHeadDim / 8); e += AT_THREADS) {
    const int h = e >> 6, u = e & 63, kc = u >> 3, jj = u & 7;
    tc::cp_async16(Qs + kc * 8192 + h * 128 + ((jj ^ (h & 7)) << 4), qg + h * kHeadDim + u * 8);
  }
  tc::cp_async_wait_all();
  if (rot) {  // rotate the last 64 channels in place (each thread its own pieces)
    for (int e = tid; e < kHeads * (kHeadDim / 8); e += AT_THREADS) {
      const int h = e >> 6, u = e & 63, kc = u >> 3, jj = u & 7;
      if (u * 8 < kHeadDim - kRopeDim) continue;
      uint4 *slot = reinterpret_cast<uint4 *>(Qs + kc * 8192 + h * 128 + ((jj ^ (h & 7)) << 4));
      const uint4 x = *slot;
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pair = (u * 8 - (kHeadDim - kRopeDim)) / 2 + q;
        const float c = a.rope_cos[(long long)p * kRopeHalf + pair];
        const float s = a.rope_sin[(long long)p * kRopeHalf + pair];
        const float x0 = bf16_lo(w[q]), x1 = bf16_hi(w[q]);
        w[q] = pack2(x0 * c - x1 * s, x0 * s + x1 * c);
      }
      *slot = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = M->tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const float sl2 = a.softmax_scale * kLog2e;
  uint32_t ph_qk = 0, ph_pv = 0;
  int n_done = 0;  // tiles accumulated into O^T
  bool ok = true;

  for (int g0 = g_begin; g0 < g_end && ok; g0 += CT) {
    // ---- candidate rows of this tile
    {
      const int gi = g0 + tid;
      M->rowp[tid] = gi < g_end ? candidate_row(a, t, b, p, V, gi) : nullptr;
    }
    const int n_valid = __syncthreads_count(M->rowp[tid] != nullptr);
    if (n_valid == 0) continue;
    // ---- gather into the swizzled tile (the previous PV has completed)
#pragma unroll 4
    for (int q = 0; q < 64; ++q) {
      const int unit = q * AT_THREADS + tid;
      const int c = unit >> 6, u = unit & 63, kc = u >> 3, jj = u & 7;
      uint8_t *dst = KVs + kc * 16384 + c * 128 + ((jj ^ (c & 7)) << 4);
      const uint16_t *src = M->rowp[c];
      if (src)
        tc::cp_async16(dst, src + u * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    tc::cp_async_wait_all();
    tc::fence_async_shared();
    __syncthreads();

    // ---- S^T = K q^T
    if (tid == 0) {
      tc::tc_fence_after();
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, kHeads);
      const uint32_t kv = tc::smem_u32(KVs), qq = tc::smem_u32(Qs);
      for (int kc = 0; kc < 8; ++kc)
#pragma unroll
        for (int s = 0; s < 4; ++s)
          tc::mma_bf16(tmem, tc::desc_sw128(kv + kc * 16384 + s * 32),
                       tc::desc_sw128(qq + kc * 8192 + s * 32), idesc, (kc | s) != 0);
      tc::mma_commit(&M->bar_qk);
    }
    ok = wait_or_flag(&M->bar_qk, ph_qk, a.status_dev);
    ph_qk ^= 1;
    tc::tc_fence_after();

    // ---- logits of this thread's candidate (log2 domain)
    const bool valid = M->rowp[tid] != nullptr;
    float x[kHeads];
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_base, v);
#pragma unroll
      for (int h = 0; h < 32; ++h) x[h] = valid ? v[h] * sl2 : -INFINITY;
      tc::tmem_ld32(tmem + lane_base + 32, v);
#pragma unroll
      for (int h = 0; h < 32; ++h) x[32 + h] = valid ? v[h] * sl2 : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4 *>(prow_chunk(Ps, tid, j)) =
          make_uint4(pack2(x[8 * j], x[8 * j + 1]), pack2(x[8 * j + 2], x[8 * j + 3]),
                     pack2(x[8 * j + 4], x[8 * j + 5]), pack2(x[8 * j + 6], x[8 * j + 7]));
    __syncthreads();
    {
      const int h = tid & 63, half = tid >> 6;
      float mx = -INFINITY;
      for (int c = half * 64; c < half * 64 + 64; ++c) mx = fmaxf(mx, p_at(Ps, c, h));
      M->red[half][h] = mx;
      if (tid == 0) M->any_rescale = 0;
    }
    __syncthreads();
    if (tid < kHeads) {
      const int h = tid;
      const float mt = fmaxf(M->red[0][h], M->red[1][h]);
      const float mo = M->m_ref[h];
      float corr = 1.f;
      if (mo == -INFINITY) {
        M->m_ref[h] = mt;  // first finite tile sets the reference
      } else if (mt > mo + kRescaleLog2) {
        M->m_ref[h] = mt;
        corr = exp2f(mo - mt);
      }
      M->corr[h] = corr;
      M->l_acc[h] *= corr;
      if (corr != 1.f && n_done > 0) M->any_rescale = 1;
    }
    __syncthreads();
    if (M->any_rescale) {  // rare: bring O^T to the new reference
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          const uint32_t addr = tmem + lane_base + 64 + mt * 64 + hh * 32;
          tc::tmem_ld32(addr, v);
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] *= M->corr[hh * 32 + h];
          tc::tmem_st32(addr, v);
        }
      tc::tc_fence_before();
    }
    // ---- P = 2^(x - m), BF16, MN-major rows
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      const float m = M->m_ref[h];
      x[h] = (m == -INFINITY) ? 0.f : exp2f(x[h] - m);
    }
    __syncthreads();  // all column reads of the previous P contents are done
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4 *>(prow_chunk(Ps, tid, j)) =
          make_uint4(pack2(x[8 * j], x[8 * j + 1]), pack2(x[8 * j + 2], x[8 * j + 3]),
                     pack2(x[8 * j + 4], x[8 * j + 5]), pack2(x[8 * j + 6], x[8 * j + 7]));
    tc::fence_async_shared();
    {
      // FP32 denominators: per-head sums of the unrounded probabilities
      const float2 s2 = warp_colsum64(x);
      const int lane = tid & 31;
      M->red4[warp][2 * lane] = s2.x;
      M->red4[warp][2 * lane + 1] = s2.y;
    }
    __syncthreads();
    // ---- O^T += V^T P^T (4 dim tiles of 128)
    if (tid == 0) {
      tc::tc_fence_after();
      constexpr uint32_t idesc = tc::idesc_bf16_f32_mn(128, kHeads);
      const uint32_t kv = tc::smem_u32(KVs), pp = tc::smem_u32(Ps);
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + 64 + mt * 64,
                       tc::desc_sw128_mn(kv + 2 * mt * 16384 + ks * 2048, 16384, 1024),
                       tc::desc_sw128_mn(pp + ks * 2048, 16384, 1024), idesc,
                       (n_done > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(&M->bar_pv);
    }
    if (tid < kHeads)
      M->l_acc[tid] += (M->red4[0][tid] + M->red4[1][tid]) + (M->red4[2][tid] + M->red4[3][tid]);
    ok = wait_or_flag(&M->bar_pv, ph_pv, a.status_dev) && ok;
    ph_pv ^= 1;
    tc::tc_fence_after();
    ++n_done;
    ok = __syncthreads_and(ok);  // a timed-out wait ends the row for the whole CTA
  }
  __syncthreads();

  // ---- epilogue: thread = output channel lane of each 128-channel tile
  if (n_splits == 1) {
    if (tid < kHeads) {
      const int h = tid;
      const float s2 = a.sink ? a.sink[h] * kLog2e : -INFINITY;
      float m = M->m_ref[h], l = n_done ? M->l_acc[h] : 0.f;
      if (m == -INFINITY) {
        m = s2;
        l = 0.f;
      }
      const float L = (m == -INFINITY) ? 0.f : l + exp2f(s2 - m);
      M->corr[h] = L > 0.f ? 1.f / L : 0.f;  // reuse as 1/L
      if (a.lse) a.lse[(long long)t * kHeads + h] = L > 0.f ? (m + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    const bool inv = a.inv_rope_out && a.rope_cos != nullptr && p >= 0 && p < a.rope_cap;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + (long long)t * kHeads * kHeadDim;
    for (int mt = 0; mt < 4; ++mt) {
      const int d = mt * 128 + tid;
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        if (n_done) {
          tc::tmem_ld32(tmem + lane_base + 64 + mt * 64 + hh * 32, v);
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          float o = v[h] * M->corr[hh * 32 + h];
          if (inv && d >= kHeadDim - kRopeDim) {
            const float other = __shfl_xor_sync(0xffffffffu, o, 1);
            const int pair = (d - (kHeadDim - kRopeDim)) >> 1;
            const float c = a.rope_cos[(long long)p * kRopeHalf + pair];
            const float s = a.rope_sin[(long long)p * kRopeHalf + pair];
            o = (d & 1) ? (-other * s + o * c) : (o * c + other * s);
          }
          out[(hh * 32 + h) * kHeadDim + d] = __float2bfloat16_rn(o);
        }
      }
    }
  } else {
    float *rec = partials + ((long long)t * n_splits + split) * REC_FLOATS;
    for (int mt = 0; mt < 4; ++mt)
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        if (n_done) {
          tc::tmem_ld32(tmem + lane_base + 64 + mt * 64 + hh * 32, v);
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) rec[(hh * 32 + h) * kHeadDim + mt * 128 + tid] = v[h];
      }
    if (tid < kHeads) {
      rec[kHeads * kHeadDim + tid] = n_done ? M->m_ref[tid] : -INFINITY;
      rec[kHeads * kHeadDim + kHeads + tid] = n_done ? M->l_acc[tid] : 0.f;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, ATTN_TMEM_COLS);
}

// Merge a row's split partials with the sink.  One CTA per (head, row);
// each thread owns four consecutive output channels.
__global__ void __launch_bounds__(128) attn_combine_kernel(csa_attn_args a, int n_splits,
                                                           const float *__restrict__ partials) {
  __shared__ float wsplit[64];
  __shared__ float sL, sM;
  const int h = blockIdx.x, t = blockIdx.y;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;
  const int p = a.row_pos[t];
  const float *rec0 = partials + (long long)t * n_splits * REC_FLOATS;
  if (threadIdx.x == 0) {
    const float s2 = a.sink ? a.sink[h] * kLog2e : -INFINITY;
    float mx = s2;
    for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, rec0[s * REC_FLOATS + kHeads * kHeadDim + h]);
    float L = 0.f;
    if (mx != -INFINITY) {
      L = exp2f(s2 - mx);
      for (int s = 0; s < n_splits; ++s) {
        const float ms = rec0[s * REC_FLOATS + kHeads * kHeadDim + h];
        const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
        if (s < 64) wsplit[s] = w;
        L += w * rec0[s * REC_FLOATS + kHeads * kHeadDim + kHeads + h];
      }
    }
    sL = L;
    sM = mx;
    if (a.lse) a.lse[(long long)t * kHeads + h] = L > 0.f ? (mx + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  const float invL = sL > 0.f ? 1.f / sL : 0.f;
  const int d = threadIdx.x * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sL > 0.f) {
    for (int s = 0; s < n_splits; ++s) {
      float w;
      if (s < 64) {
        w = wsplit[s];
      } else {
        const float ms = rec0[s * REC_FLOATS + kHeads * kHeadDim + h];
        w = ms == -INFINITY ? 0.f : exp2f(ms - sM);
      }
      if (w == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4 *>(rec0 + s * REC_FLOATS + h * kHeadDim + d);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  float o[4] = {acc.x * invL, acc.y * invL, acc.z * invL, acc.w * invL};
  if (a.inv_rope_out && a.rope_cos != nullptr && p >= 0 && p < a.rope_cap &&
      d >= kHeadDim - kRopeDim) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int pair = (d + 2 * q - (kHeadDim - kRopeDim)) >> 1;
      const float c = a.rope_cos[(long long)p * kRopeHalf + pair];
      const float s = a.rope_sin[(long long)p * kRopeHalf + pair];
      const float x0 = o[2 * q], x1 = o[2 * q + 1];
      o[2 * q] = x0 * c + x1 * s;
      o[2 * q + 1] = -x0 * s + x1 * c;
    }
  }
  __nv_bfloat162 *out = reinterpret_cast<__nv_bfloat162 *>(
      static_cast<__nv_bfloat16 *>(a.out) + ((long long)t * kHeads + h) * kHeadDim + d);
  out[0] = __floats2bfloat162_rn(o[0], o[1]);
  out[1] = __floats2bfloat162_rn(o[2], o[3]);
}

}  // namespace

int attn_record_floats() { return REC_FLOATS; }

cudaError_t launch_attn(const csa_attn_args &a, int n_splits, int tiles_per_split,
                        float *partials, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, ATTN_SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(n_splits, a.n_rows);
  const int kid = n_splits == 1 ? CSA_K_ATTN_PREFILL : CSA_K_ATTN_PARTIAL;
  launch_begin(kid, s);
  attn_tc_kernel<<<grid, AT_THREADS, ATTN_SMEM, s>>>(a, n_splits, tiles_per_split, partials);
  launch_end(kid, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_splits == 1) return e;
  launch_begin(CSA_K_ATTN_COMBINE, s);
  attn_combine_kernel<<<dim3(kHeads, a.n_rows), 128, 0, s>>>(a, n_splits, partials);
  launch_end(CSA_K_ATTN_COMBINE, s);
  return cudaGetLastError();
}

}  // namespace csa
