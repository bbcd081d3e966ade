// Decode shared-KV sparse attention with an attention sink, the candidates of
// a row split over several CTAs.  Candidates of a query row are its selected
// compressed entries followed by its raw causal window; each candidate row is
// both key and value.
//
// Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2),
// "二阶段 CP 总体算法" (Stage-2 sparse attention with sinks, softmax_scale,
// ori_win_left = 127; outputs out and lse), "9.1" (candidate list = window KV
// and selected compressed KV) and "7. Window KV Halo" (window includes self).
//
// GB300 mapping.  A row's 128-candidate tiles are dealt to S CTAs (one tile
// each while the grid fits one CTA per SM, S <= 17).  Each CTA loads the row's
// q with TMA while it gathers its first tile with cp.async (q and the gather
// overlap), runs the tile's two contractions on tcgen05 (see attn_common.cuh)
// and a softmax whose running maximum only moves past a 2^8 growth.  The
// partial softmaxes merge through the workspace (L2): every CTA stores its
// O^T / l as BF16 (512 contiguous bytes per warp store) with its per-head
// maximum and denominator, the S CTAs of the row meet at a counter (bounded
// wait; the grid fits the GPU, so all of them are resident), and each then
// weighs the S partials of its own slice of the output channels and writes
// it.  Barrier initialisation and the tensor-memory allocation run before the
// kernel waits for its predecessor in the stream.
#include <algorithm>
#include <cstring>

#include "attn_common.cuh"
#include "lowbit.cuh"

namespace csa {
namespace {

using namespace attn;

constexpr int AD_THREADS = 256;
constexpr int AD_BAR = 1;  // named barrier over all 256 threads (the softmax's)
constexpr int AD_MAX_SPLITS = 17;  // (topk <= 2048 + window 128) / 128 tiles

struct AdMisc {
  uint64_t q_full, mma_bar, done_bar;
  uint32_t tmem_base;
  int flag;
  SoftState st;
  const uint8_t *src[CT];   // pool row of each candidate of the tile, or null
  alignas(16) float w[AD_MAX_SPLITS][kHeads];   // references, then merge weights, per partial
  alignas(16) float lq[AD_MAX_SPLITS][kHeads];  // denominators per partial
  alignas(16) float red_l[4][kHeads];
  alignas(16) float f_self[kHeads];       // this CTA's share of each head's output
  alignas(16) float rope[2 * kRopeHalf];  // cos, sin at the row's position
};
constexpr int AD_SMEM = OFF_MISC + (int)sizeof(AdMisc) + 1024;
static_assert(AD_SMEM <= 227 * 1024, "shared memory");

// The output channels d in [chan_lo(r), chan_lo(r + 1)) are merged by CTA r:
// whole 16-channel groups, so that every output row piece starts on a 32-byte
// sector and RoPE pairs stay together.
__device__ __forceinline__ int chan_lo(uint32_t r, uint32_t S) {
  return 16 * (int)((kHeadDim / 16 * r) / S);
}

// Workspace of a call with `items` (row, group of 64 heads) pairs split S
// ways: the BF16 partials (8 head groups x 512 channels of 16-byte units per
// split), the per-head reference and denominator of each split, and two
// counters per item (arrivals, departures), which must read zero before the
// first call and are left at zero by every call that completes.
struct AdWs {
  uint4 *part;
  float *stat;
  uint32_t *ctr;
};
__host__ __device__ __forceinline__ long long ad_ws_bytes(long long items, long long S) {
  return items * S * (8 * kHeadDim * 16 + 2 * kHeads * 4) + items * 8;
}
__device__ __forceinline__ AdWs ad_ws(void *ws, long long items, long long S) {
  uint8_t *b = static_cast<uint8_t *>(ws);
  AdWs w;
  w.part = reinterpret_cast<uint4 *>(b);
  w.stat = reinterpret_cast<float *>(b + items * S * (8 * kHeadDim * 16));
  w.ctr = reinterpret_cast<uint32_t *>(b + items * S * (8 * kHeadDim * 16 + 2 * kHeads * 4));
  return w;
}

// The S CTAs of an item meet once their partials are in the workspace:
// thread 0 counts this CTA in (after a release fence) and waits, at most a
// second, until the count equals S exactly (a counter that did not start at
// zero makes the wait run out rather than pass early); false, with
// CSA_DEV_TIMEOUT flagged, when it gives up.
__device__ bool split_barrier(uint32_t *ctr, uint32_t S, uint32_t *status, int *s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int ok = 1;
    if (atomicAdd(ctr, 1u) + 1u != S) {
      const uint64_t t0 = tc::global_ns();
      while (*reinterpret_cast<volatile uint32_t *>(ctr) != S) {
        if (tc::global_ns() - t0 > 1000000000ull) {
          ok = 0;
          flag(status, CSA_DEV_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Counts this CTA out; the last of the S to leave (every one has passed the
// barrier) puts both counters back to zero for the next call.
__device__ __forceinline__ void split_depart(uint32_t *ctr, uint32_t S) {
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(ctr + 1, 1u) + 1u == S) {
    ctr[0] = 0u;
    ctr[1] = 0u;
    __threadfence();
  }
}

// Pool row of candidate j of row t (its list: top-k entries, then the
// window), or null when absent; data errors raise their flag.
__device__ __forceinline__ const uint8_t *candidate_row(const csa_attn_args &a, int t, int b,
                                                        int p, int V, int kvl, int j) {
  if (j < a.topk) {
    // dense visibility (no selection): compressed entry j itself
    const int c = a.topk_idx ? a.topk_idx[(long long)t * a.topk + j] : (j < V ? j : -1);
    if (!a.topk_idx && j == 0 && V > a.topk) flag(a.status_dev, CSA_DEV_BAD_INDEX);
    if (c < 0) return nullptr;
    if (c >= V) {
      flag(a.status_dev, CSA_DEV_BAD_INDEX);
      return nullptr;
    }
    const long long row =
        page_row(a.cmp_block_table, a.cmp_max_blocks, a.cmp_n_blocks, b, c, a.status_dev);
    return row < 0 ? nullptr
                   : static_cast<const uint8_t *>(a.cmp_pool) +
                         pool_offset(row, a.cmp_page_stride, a.cmp_row_stride);
  }
  if (j >= a.topk + a.window) return nullptr;
  const int pp = p - a.window + 1 + (j - a.topk);
  if (pp < 0) return nullptr;
  if (pp >= kvl) {
    flag(a.status_dev, CSA_DEV_BAD_POS);
    return nullptr;
  }
  const long long row =
      page_row(a.kv_block_table, a.kv_max_blocks, a.kv_n_blocks, b, pp, a.status_dev);
  return row < 0 ? nullptr
                 : static_cast<const uint8_t *>(a.kv_pool) +
                       pool_offset(row, a.kv_page_stride, a.kv_row_stride);
}

// Gather of tile g when a pool holds a low-bit format ("DeepSeek V4.1 Flash",
// production cache ABI: FP4 compressed KV with E4M3 scales per 16 channels,
// MXFP8 window KV): unit = (candidate row, 32-channel slab), 16 consecutive
// threads per row.  Every low-bit unit's codes and scales are loaded before
// any is converted; each slab becomes 64 bytes of BF16 (exact) in the
// 128-byte-swizzled tile.  BF16 rows and absent rows go through cp.async
// (zero fill) as in the plain gather.  The conversion loops stay rolled: a
// decode CTA runs this code once or twice, cold, so its size costs more
// than its instruction count.
constexpr int LB_UNITS = CT * (kHeadDim / 32) / AD_THREADS;  // 8 per thread

// One slab's four 16-byte pieces: FP4 (kind 2: codes in c0, two E4M3 scale
// bytes in sc) or MXFP8 (kind 3: codes in c0, c1, one E8M0 byte in sc).
__device__ __forceinline__ void convert_slab(int kind, uint4 c0, uint4 c1, uint32_t sc, int r,
                                             int slab, uint8_t *KVs) {
  uint8_t *base = KVs + (slab >> 1) * 16384 + r * 128;
  const float e8 = lowbit::pow2f((int)(sc & 0xFFu) - 127);
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    const uint4 c = q < 2 ? c0 : c1;
    const bool lo = (q & 1) == 0;
    uint4 v;
    if (kind == 2) {
      const uint4 cc = c0;
      const uint32_t w = q == 0 ? cc.x : q == 1 ? cc.y : q == 2 ? cc.z : cc.w;
      v = lowbit::e2m1x8_e4m3_to_bf16x8(w, (sc >> (8 * (q >> 1))) & 0xFFu);
    } else {
      v = lowbit::e4m3x8_e8m0_to_bf16x8(lo ? make_uint2(c.x, c.y) : make_uint2(c.z, c.w), e8);
    }
    const int piece = (slab & 1) * 4 + q;
    *reinterpret_cast<uint4 *>(base + ((piece ^ (r & 7)) << 4)) = v;
  }
}

__device__ __forceinline__ void gather_lowbit(const csa_attn_args &a, const AdMisc *M,
                                              uint8_t *KVs, int g, int tid) {
  uint4 c0[LB_UNITS], c1[LB_UNITS];
  uint32_t sc[LB_UNITS];
  int kind[LB_UNITS];  // 0: cp.async (BF16 or absent), 2: FP4 + E4M3, 3: MXFP8
#pragma unroll
  for (int i = 0; i < LB_UNITS; ++i) {
    const int u = i * AD_THREADS + tid, r = u >> 4, slab = u & 15;
    const uint8_t *row = M->src[r];
    const int fmt = g * CT + r < a.topk ? a.cmp_fmt : a.kv_fmt;
    kind[i] = !row ? 0 : (fmt == CSA_FMT_FP4_E4M3 ? 2 : (fmt == CSA_FMT_MXFP8 ? 3 : 0));
    c0[i] = c1[i] = make_uint4(0u, 0u, 0u, 0u);
    sc[i] = 0u;
    if (kind[i] == 2) {
      const long long ri = (row - static_cast<const uint8_t *>(a.cmp_pool)) / (kHeadDim / 2);
      c0[i] = *reinterpret_cast<const uint4 *>(row + slab * 16);
      sc[i] = *reinterpret_cast<const uint16_t *>(a.cmp_scale_pool + ri * (kHeadDim / 16) + slab * 2);
    } else if (kind[i] == 3) {
      const long long ri = (row - static_cast<const uint8_t *>(a.kv_pool)) / kHeadDim;
      c0[i] = *reinterpret_cast<const uint4 *>(row + slab * 32);
      c1[i] = *reinterpret_cast<const uint4 *>(row + slab * 32 + 16);
      sc[i] = a.kv_scale_pool[ri * (kHeadDim / 32) + slab];
    }
  }
#pragma unroll
  for (int i = 0; i < LB_UNITS; ++i) {
    const int u = i * AD_THREADS + tid, r = u >> 4, slab = u & 15;
    if (kind[i] != 0) {
      convert_slab(kind[i], c0[i], c1[i], sc[i], r, slab, KVs);
    } else {
      // BF16 row (or absent: zero fill): the slab's four 16-byte pieces
      const uint8_t *row = M->src[r];
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int piece = (slab & 1) * 4 + q;
        uint8_t *dst = KVs + (slab >> 1) * 16384 + r * 128 + ((piece ^ (r & 7)) << 4);
        tc::cp_async16_zfill(dst, row ? row + slab * 64 + q * 16 : static_cast<const uint8_t *>(a.kv_pool),
                             row != nullptr);
      }
    }
  }
}

// LOWBIT: a pool holds a low-bit format (its gather is a separate
// instantiation, so that the BF16 kernel carries none of its code).
template <bool LOWBIT>
__global__ void __launch_bounds__(AD_THREADS, 1)
    attn_decode_kernel(csa_attn_args a, int tiles_per_split,
                       const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t *Qs = sm + OFF_Q;
  uint8_t *KVs = sm + OFF_KV;
  uint8_t *Ps = sm + OFF_P;
  AdMisc *M = reinterpret_cast<AdMisc *>(sm + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s = blockIdx.x, S = gridDim.x;

  // ---- set-up that reads no global memory, overlapping the previous kernel
  if (tid == 0) {
    tc::mbar_init(&M->q_full, 1);
    tc::mbar_init(&M->mma_bar, 1);
    tc::mbar_init(&M->done_bar, 1);
    tc::mbar_fence_init();
  }
  if (tid < kHeads) M->st.m[tid] = -INFINITY;
  if (warp == 0) tc::tmem_alloc(&M->tmem_base, TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = M->tmem_base;
  tc::griddep_wait();
  tc::griddep_launch_dependents();

  // blockIdx.y = (row, group of 64 heads); heads past n_heads are computed
  // from padding (their columns are independent of the others) and never stored
  const int HG = (a.n_heads + kHeads - 1) / kHeads;
  const int t = blockIdx.y / HG, h_lo = (blockIdx.y % HG) * kHeads;
  const int nh = min(kHeads, a.n_heads - h_lo);
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) {  // the same for every CTA of the item: none waits
    if (b >= 0 && tid == 0 && s == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
    return;
  }
  const int p = a.row_pos[t];
  const int V = min(visible_count(p, a.ratio, a.n_cmp[b]), a.cmp_max_blocks * kBlock);
  const int kvl = a.kv_len[b];
  const int n_tiles = (a.topk + a.window + CT - 1) / CT;
  const int g_begin = (int)s * tiles_per_split;
  const int g_end = min(n_tiles, g_begin + tiles_per_split);
  const uint32_t kv = tc::smem_u32(KVs), qq = tc::smem_u32(Qs), pp = tc::smem_u32(Ps);

  // q of the row by TMA, in flight while the first tile is gathered
  const bool has_tiles = g_begin < g_end;
  if (has_tiles && tid == 0) {
    tc::mbar_arrive_expect_tx(&M->q_full, 8 * 8192);
    for (int kc = 0; kc < 8; ++kc)
      tc::tma_load_2d(Qs + kc * 8192, &qmap, kc * 64, t * a.n_heads + h_lo, &M->q_full);
  }
  bool rot = a.rope_cos != nullptr && p >= 0;
  if (rot && p >= a.rope_cap) {
    rot = false;
    if (tid == 0 && s == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
  }
  // the row's RoPE entries and the sink logit of head tid % 64, read up front
  const float sink_h = (tid & (kHeads - 1)) < nh && a.sink
                           ? a.sink[h_lo + (tid & (kHeads - 1))] * kLog2e
                           : -INFINITY;
  if (rot && tid < 2 * kRopeHalf)
    M->rope[tid] = tid < kRopeHalf ? a.rope_cos[(long long)p * kRopeHalf + tid]
                                   : a.rope_sin[(long long)p * kRopeHalf + tid - kRopeHalf];
  const int qd = warp & 3, h0 = (warp >> 2) * 32, c = qd * 32 + lane;
  const int sub = lane >> 3, piece = lane & 7;  // gather: rows 32 i + 4 warp + sub, 16-byte piece
  const float sl2 = a.softmax_scale * kLog2e;
  float lacc = 0.f;  // this warp's partial denominator of head h0 + lane
  bool first = true, ok = true, q_ready = false;
  uint32_t phase = 0;

  for (int g = g_begin; g < g_end && ok; ++g) {
    // ---- candidate rows of this tile
    if (tid < CT) M->src[tid] = candidate_row(a, t, b, p, V, kvl, g * CT + tid);
    if (__syncthreads_count(tid < CT && M->src[tid] != nullptr) == 0) continue;
    const bool valid = M->src[c] != nullptr;
    // ---- gather the tile into the swizzled layout (the previous P.V is done)
    if constexpr (LOWBIT) {
      gather_lowbit(a, M, KVs, g, tid);
    } else {
      const uint8_t *src[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) src[i] = M->src[32 * i + 4 * warp + sub];
      // a candidate row's eight 128-byte pieces are requested back to back
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 32 * i + 4 * warp + sub;
        uint8_t *dst = KVs + r * 128 + ((piece ^ (r & 7)) << 4);
        for (int kc = 0; kc < 8; ++kc) {
          const uint8_t *gsrc = src[i] ? src[i] + kc * 128 + piece * 16
                                       : static_cast<const uint8_t *>(a.kv_pool);
          tc::cp_async16_zfill(dst + kc * 16384, gsrc, src[i] != nullptr);
        }
      }
    }
    if (!q_ready) {
      // q landed meanwhile: rotate its last 64 channels at p
      if (!tc::mbar_wait(&M->q_full, 0)) {
        ok = false;
        flag(a.status_dev, CSA_DEV_TIMEOUT);
      }
      if (rot) rope_q_rows(Qs + 7 * 8192, M->rope, M->rope + kRopeHalf, tid, AD_THREADS);
      q_ready = true;
    }
    tc::cp_async_wait_all();
    tc::fence_async_shared();
    __syncthreads();

    // ---- S^T = K q^T
    if (warp == 0) {
      tc::tc_fence_after();
      for (int kc = 0; kc < 8; ++kc) issue_qk(tmem, kv, qq, kc);
      tc::mma_commit_elect(&M->mma_bar);
    }
    if (!tc::mbar_wait(&M->mma_bar, phase)) ok = false;
    phase ^= 1;

    // ---- softmax; P^T to shared memory
    float x[32];
    softmax_tile(tmem, qd, h0, valid, sl2, first, &M->st, Ps, AD_BAR, lacc, x);
    tc::fence_async_shared();
    tc::tc_fence_before();
    tc::bar_sync(AD_BAR, AD_THREADS);

    // ---- O^T += V^T P^T
    if (warp == 0) {
      tc::tc_fence_after();
      for (int mt = 0; mt < 4; ++mt) issue_pv(tmem, kv, pp, mt, !first);
      tc::mma_commit_elect(&M->mma_bar);
    }
    lacc += warp_col_reduce32<false>(x);
    if (!tc::mbar_wait(&M->mma_bar, phase)) ok = false;
    phase ^= 1;
    tc::tc_fence_after();
    first = false;
    ok = __syncthreads_and(ok);
    if (!ok && tid == 0) flag(a.status_dev, CSA_DEV_TIMEOUT);
  }
  if (has_tiles && !q_ready) tc::mbar_wait(&M->q_full, 0, 50000000ull);  // no tile had candidates
  if (!ok && warp == 0) {
    // nothing of ours may still run on TMEM when it is read or released
    tc::mma_commit_elect(&M->done_bar);
    tc::mbar_wait(&M->done_bar, 0, 100000000ull);
  }

  // ---- this CTA's partial into the workspace: O^T / l as BF16 (normalised
  // by this CTA's own denominator, so BF16 keeps it to 2^-9 relative whatever
  // the magnitudes), 16-byte unit (hb, d) holding heads 8 hb .. 8 hb + 7 of
  // channel d (the 32 lanes of a warp store 512 contiguous bytes), and its
  // per-head reference and denominator.
  const AdWs W = ad_ws(a.workspace, gridDim.y, S);
  uint4 *part = W.part + ((long long)blockIdx.y * S + s) * (8 * kHeadDim);
  float *stat = W.stat + ((long long)blockIdx.y * S + s) * (2 * kHeads);
  M->red_l[qd][h0 + lane] = lacc;
  __syncthreads();
  if (tid < kHeads) {
    const float l = (M->red_l[0][tid] + M->red_l[1][tid]) + (M->red_l[2][tid] + M->red_l[3][tid]);
    M->f_self[tid] = !first && l > 0.f ? 1.f / l : 0.f;
    stat[tid] = first ? -INFINITY : M->st.m[tid];
    stat[kHeads + tid] = first ? 0.f : l;
  }
  __syncthreads();
  {
    float f[32];
    load32(M->f_self + h0, f);
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    tc::tc_fence_after();
#pragma unroll 1
    for (int m4 = 0; m4 < 4; ++m4) {
      float v[32];
      if (first) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      } else {
        tc::tmem_ld32(tmem + lane_off + O_COL + m4 * 64 + h0, v);
      }
      const int d = m4 * 128 + qd * 32 + lane;
#pragma unroll
      for (int cgrp = 0; cgrp < 4; ++cgrp) {
        const int hb = (h0 >> 3) + cgrp;
        part[hb * kHeadDim + d] =
            make_uint4(pack2(v[8 * cgrp + 0] * f[8 * cgrp + 0], v[8 * cgrp + 1] * f[8 * cgrp + 1]),
                       pack2(v[8 * cgrp + 2] * f[8 * cgrp + 2], v[8 * cgrp + 3] * f[8 * cgrp + 3]),
                       pack2(v[8 * cgrp + 4] * f[8 * cgrp + 4], v[8 * cgrp + 5] * f[8 * cgrp + 5]),
                       pack2(v[8 * cgrp + 6] * f[8 * cgrp + 6], v[8 * cgrp + 7] * f[8 * cgrp + 7]));
      }
    }
  }

  // ---- the S CTAs of the row meet: every partial is in the workspace
  ok = split_barrier(W.ctr + 2 * blockIdx.y, S, a.status_dev, &M->flag) && ok;

  // ---- merge weights: every partial's statistics into shared memory at once
  // (independent loads), then each head's maximum and denominator over the S
  // partials (thread = (head, quarter of the partials)); w[q][h] becomes the
  // weight of partial q
  {
    constexpr int PER = (AD_MAX_SPLITS * 2 * kHeads + AD_THREADS - 1) / AD_THREADS;
    const float *st_row = W.stat + (long long)blockIdx.y * S * (2 * kHeads);
    const int n_st = (int)S * 2 * kHeads;
    float v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + u * AD_THREADS;
      v[u] = e < n_st && ok ? __ldcg(st_row + e) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + u * AD_THREADS;
      if (e < n_st) {
        const int q = e / (2 * kHeads), k = e % (2 * kHeads);
        if (k < kHeads)
          M->w[q][k] = ok ? v[u] : -INFINITY;
        else
          M->lq[q][k - kHeads] = v[u];
      }
    }
  }
  __syncthreads();
  {
    const int h = tid & (kHeads - 1), jq = tid >> 6;
    float mx = -INFINITY;
    for (uint32_t q = jq; q < S; q += 4) mx = fmaxf(mx, M->w[q][h]);
    M->red_l[jq][h] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(M->red_l[0][h], M->red_l[1][h]), fmaxf(M->red_l[2][h], M->red_l[3][h]));
    const float s2 = sink_h;
    mx = fmaxf(mx, s2);
    float part_l = 0.f;
    if (mx != -INFINITY)
      for (uint32_t q = jq; q < S; q += 4) {
        const float mq = M->w[q][h];
        const float e = mq == -INFINITY ? 0.f : exp2_sfu(mq - mx) * M->lq[q][h];
        M->w[q][h] = e;
        part_l += e;
      }
    __syncthreads();
    M->red_l[jq][h] = part_l;
    __syncthreads();
    float L = (M->red_l[0][h] + M->red_l[1][h]) + (M->red_l[2][h] + M->red_l[3][h]);
    if (mx != -INFINITY) L += exp2_sfu(s2 - mx);
    const float inv_L = L > 0.f ? 1.f / L : 0.f;
    for (uint32_t q = jq; q < S; q += 4) M->w[q][h] = mx == -INFINITY ? 0.f : M->w[q][h] * inv_L;
    if (jq == 0 && s == 0 && a.lse && h < nh)
      a.lse[(long long)t * a.n_heads + h_lo + h] = L > 0.f ? (mx + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();

  // ---- this CTA's channels: warp w sums heads 8 w .. 8 w + 7 over the S
  // partials, 32 consecutive channels per step (a RoPE pair sits in an
  // even/odd lane pair), and stores them (64 contiguous bytes per head)
  {
    const int d0 = chan_lo(s, S), dn = chan_lo(s + 1, S) - d0;
    const bool inv = a.inv_rope_out && rot;
    const int hb = warp;
    const uint4 *parts = W.part + (long long)blockIdx.y * S * (8 * kHeadDim) + hb * kHeadDim;
    __nv_bfloat16 *out =
        static_cast<__nv_bfloat16 *>(a.out) + ((long long)t * a.n_heads + h_lo) * kHeadDim;
    for (int dl0 = 0; dl0 < dn; dl0 += 32) {  // the same trip count in every lane
      const int dl = dl0 + lane;
      const bool live = dl < dn;  // dn is a multiple of 16: RoPE pairs live together
      const int d = d0 + (live ? dl : 0);
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // every partial's unit requested before any is used (one L2 round trip)
      uint4 v[AD_MAX_SPLITS];
#pragma unroll
      for (int u = 0; u < AD_MAX_SPLITS; ++u)
        v[u] = u < (int)S ? __ldcg(parts + (long long)u * (8 * kHeadDim) + d)
                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < AD_MAX_SPLITS; ++u) {
        if (u >= (int)S) break;
        const float4 w0 = *reinterpret_cast<const float4 *>(&M->w[u][hb * 8]);
        const float4 w1 = *reinterpret_cast<const float4 *>(&M->w[u][hb * 8 + 4]);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[2 * i] = fmaf(wv[2 * i], __uint_as_float(wd[i] << 16), o[2 * i]);
          o[2 * i + 1] = fmaf(wv[2 * i + 1], __uint_as_float(wd[i] & 0xFFFF0000u), o[2 * i + 1]);
        }
      }
      if (inv) {
        // inverse rotation of the RoPE channel pairs (partner: the neighbouring lane)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float other = __shfl_xor_sync(0xffffffffu, o[i], 1);
          if (d >= kHeadDim - kRopeDim) {
            const int pair = (d - (kHeadDim - kRopeDim)) >> 1;
            const float cs = M->rope[pair], sn = M->rope[kRopeHalf + pair];
            o[i] = (d & 1) == 0 ? o[i] * cs + other * sn : -other * sn + o[i] * cs;
          }
        }
      }
      if (live && ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (hb * 8 + i < nh) out[(hb * 8 + i) * kHeadDim + d] = __float2bfloat16_rn(o[i]);
      }
    }
  }
  split_depart(W.ctr + 2 * blockIdx.y, S);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// Opt the kernel into its shared memory, once per device.
cudaError_t prepare_kernel() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AD_SMEM);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

}  // namespace

// Splits per (row, head group): as many CTAs as the row has tiles while the
// whole grid fits one CTA per SM (its CTAs wait for one another, so all of a
// row's must be resident at once); with more items than SMs, one CTA per item.
void attn_decode_geometry(const csa_attn_args &a, int *n_splits, int *tiles_per_split) {
  const int tiles = (a.topk + a.window + CT - 1) / CT;
  const long long items = (long long)a.n_rows * ((a.n_heads + kHeads - 1) / kHeads);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();  // no device (a size query on a host without one): one split
    sms = 1;
  }
  const long long fit = items > 0 ? sms / items : 1;
  const int S = (int)std::max(1ll, std::min<long long>(tiles, fit));
  const int tps = (tiles + S - 1) / S;
  *tiles_per_split = tps;
  *n_splits = (tiles + tps - 1) / tps;
}

size_t attn_decode_workspace(const csa_attn_args &a) {
  if (a.n_rows <= 0) return 0;
  int S = 1, tps = 1;
  attn_decode_geometry(a, &S, &tps);
  const long long items = (long long)a.n_rows * ((a.n_heads + kHeads - 1) / kHeads);
  return (size_t)ad_ws_bytes(items, S);
}

cudaError_t launch_attn_decode(const csa_attn_args &a, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  if (!encode_rows_map(&qmap, a.q, (long long)a.n_rows * a.n_heads, kHeads))
    return cudaErrorInvalidValue;
  cudaError_t e = prepare_kernel();
  if (e != cudaSuccess) return e;
  int n_splits, tps;
  attn_decode_geometry(a, &n_splits, &tps);
  launch_begin(CSA_K_ATTN_DECODE, s);
  const bool lowbit = a.kv_fmt == CSA_FMT_MXFP8 || a.cmp_fmt == CSA_FMT_FP4_E4M3;
  e = launch_kernel(lowbit ? attn_decode_kernel<true> : attn_decode_kernel<false>,
                    dim3(n_splits, a.n_rows * ((a.n_heads + kHeads - 1) / kHeads)), dim3(AD_THREADS),
                    (size_t)AD_SMEM, s, 0, false, a, tps, qmap);
  launch_end(CSA_K_ATTN_DECODE, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
