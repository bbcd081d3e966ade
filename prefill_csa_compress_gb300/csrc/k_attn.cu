// Decode shared-KV sparse attention with an attention sink, the candidates of
// a row split over the CTAs of one thread-block cluster.  Candidates of a
// query row are its selected compressed entries followed by its raw causal
// window; each candidate row is both key and value.
//
// Source: "Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2),
// "二阶段 CP 总体算法" (Stage-2 sparse attention with sinks, softmax_scale,
// ori_win_left = 127; outputs out and lse), "9.1" (candidate list = window KV
// and selected compressed KV) and "7. Window KV Halo" (window includes self).
//
// GB300 mapping.  A row's 128-candidate tiles are dealt to the S CTAs of a
// cluster (S <= 16, one CTA per SM).  Each CTA loads the row's q with TMA while
// it gathers its first tile with cp.async (q and the gather overlap), runs the
// tile's two contractions on tcgen05 (see attn_common.cuh) and a softmax whose
// running maximum only moves past a 2^8 growth.  The partial softmaxes merge
// through distributed shared memory: every CTA parks its O^T (FP32) and its
// per-head maximum and denominator in its own shared memory, and after a
// cluster barrier CTA r normalises the r-th slice of the output by reading
// the matching slices of all S partials -- no partial ever reaches HBM and no
// second kernel runs.
#include <cstring>

#include "attn_common.cuh"

namespace csa {
namespace {

using namespace attn;

constexpr int AD_THREADS = 256;
constexpr int AD_BAR = 1;  // named barrier over all 256 threads (the softmax's)
constexpr int AD_MAX_CLUSTER = 16;

struct AdMisc {
  uint64_t q_full, mma_bar, done_bar, recv_bar;
  uint32_t tmem_base;
  int pad;
  SoftState st;
  const uint16_t *src[CT];  // pool row of each candidate of the tile, or null
  alignas(16) float m_all[AD_MAX_CLUSTER][kHeads];  // every CTA's reference per head (log2)
  alignas(16) float l_all[AD_MAX_CLUSTER][kHeads];  // every CTA's denominator per head
  alignas(16) float red_l[4][kHeads];
  alignas(16) float w_all[AD_MAX_CLUSTER][kHeads];  // scale of each CTA's partial
  alignas(16) float inv_L[kHeads];
  alignas(16) float inv_l[kHeads];  // 1 / this CTA's denominator per head
};
constexpr int AD_SMEM = OFF_MISC + (int)sizeof(AdMisc) + 1024;
static_assert(AD_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier: arrive early, wait where it matters.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
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


// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory to the
// shared memory of CTA `rank`, completing on that CTA's mbarrier.
__device__ __forceinline__ void bulk_to_peer(const void *src, uint32_t dst_local, uint32_t bytes,
                                             uint64_t *bar_local, uint32_t rank) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(peer_addr_u32(dst_local, rank)),
      "r"(tc::smem_u32(src)), "r"(bytes), "r"(peer_addr(bar_local, rank))
      : "memory");
}

// Pool row of candidate j of row t (its list: top-k entries, then the
// window), or null when absent; data errors raise their flag.
__device__ __forceinline__ const uint16_t *candidate_row(const csa_attn_args &a, int t, int b,
                                                         int p, int V, int kvl, int j) {
  if (j < a.topk) {
    const int c = a.topk_idx[(long long)t * a.topk + j];
    if (c < 0) return nullptr;
    if (c >= V) {
      flag(a.status_dev, CSA_DEV_BAD_INDEX);
      return nullptr;
    }
    const long long row =
        page_row(a.cmp_block_table, a.cmp_max_blocks, a.cmp_n_blocks, b, c, a.status_dev);
    return row < 0 ? nullptr : static_cast<const uint16_t *>(a.cmp_pool) + row * kHeadDim;
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
  return row < 0 ? nullptr : static_cast<const uint16_t *>(a.kv_pool) + row * kHeadDim;
}

__global__ void __launch_bounds__(AD_THREADS, 1)
    attn_decode_kernel(csa_attn_args a, int tiles_per_split,
                       const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t *Qs = sm + OFF_Q;
  uint8_t *KVs = sm + OFF_KV;
  uint8_t *Ps = sm + OFF_P;
  // once the tiles are done: this CTA's normalised partial O[h][d] / l[h] (BF16)
  uint16_t *Os = reinterpret_cast<uint16_t *>(KVs);
  AdMisc *M = reinterpret_cast<AdMisc *>(sm + OFF_MISC);
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y;
  const uint32_t s = cluster_rank(), S = gridDim.x;
  const int b = a.row_req[t];
  if (b < 0) return;  // every CTA of the cluster serves the same row
  if (b >= a.n_req) {
    if (tid == 0 && s == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
    return;
  }
  const int p = a.row_pos[t];
  const int V = min(visible_count(p, a.ratio, a.n_cmp[b]), a.cmp_max_blocks * kBlock);
  const int kvl = a.kv_len[b];
  const int n_tiles = (a.topk + a.window + CT - 1) / CT;
  const int g_begin = (int)s * tiles_per_split;
  const int g_end = min(n_tiles, g_begin + tiles_per_split);

  if (tid == 0) {
    tc::mbar_init(&M->q_full, 1);
    tc::mbar_init(&M->mma_bar, 1);
    tc::mbar_init(&M->done_bar, 1);
    tc::mbar_init(&M->recv_bar, 1);
    tc::mbar_fence_init();
  }
  if (tid < kHeads) M->st.m[tid] = -INFINITY;
  // every CTA of the cluster must have started before any of them touches a
  // peer's shared memory: the matching wait comes before the first remote store
  cluster_arrive_relaxed();
  if (warp == 0) tc::tmem_alloc(&M->tmem_base, TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = M->tmem_base;
  const uint32_t kv = tc::smem_u32(KVs), qq = tc::smem_u32(Qs), pp = tc::smem_u32(Ps);

  // q of the row by TMA, in flight while the first tile is gathered
  const bool has_tiles = g_begin < g_end;
  if (has_tiles && tid == 0) {
    tc::mbar_arrive_expect_tx(&M->q_full, 8 * 8192);
    for (int kc = 0; kc < 8; ++kc)
      tc::tma_load_2d(Qs + kc * 8192, &qmap, kc * 64, t * kHeads, &M->q_full);
  }
  bool rot = a.rope_cos != nullptr && p >= 0;
  if (rot && p >= a.rope_cap) {
    rot = false;
    if (tid == 0 && s == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
  }

  // the sink logit of head tid, read now rather than at the merge
  const float sink2 = tid < kHeads && a.sink ? a.sink[tid] * kLog2e : -INFINITY;
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
    {
      const uint16_t *src[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) src[i] = M->src[32 * i + 4 * warp + sub];
      for (int kc = 0; kc < 8; ++kc) {
        uint8_t *dst = KVs + kc * 16384;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 32 * i + 4 * warp + sub;
          const uint16_t *gsrc = src[i] ? src[i] + kc * 64 + piece * 8
                                        : static_cast<const uint16_t *>(a.kv_pool);
          tc::cp_async16_zfill(dst + r * 128 + ((piece ^ (r & 7)) << 4), gsrc, src[i] != nullptr);
        }
      }
    }
    if (!q_ready) {
      // q landed meanwhile: rotate its last 64 channels at p
      if (!tc::mbar_wait(&M->q_full, 0)) {
        ok = false;
        flag(a.status_dev, CSA_DEV_TIMEOUT);
      }
      if (rot) rope_q_tile(Qs, a, p, tid, AD_THREADS);
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
    // nothing of ours may still run on TMEM when it is released
    tc::mma_commit_elect(&M->done_bar);
    tc::mbar_wait(&M->done_bar, 0, 100000000ull);
  }

  // ---- this CTA's partial: its per-head reference and denominator go to
  // every CTA of the cluster (remote stores, ordered by the cluster barrier);
  // O^T / l stays here as BF16 O[h][d] (normalised, so BF16 keeps it to
  // 2^-9 relative whatever the magnitudes)
  M->red_l[qd][h0 + lane] = lacc;
  __syncthreads();
  if (tid < kHeads) {
    const float l = (M->red_l[0][tid] + M->red_l[1][tid]) + (M->red_l[2][tid] + M->red_l[3][tid]);
    M->inv_l[tid] = !first && l > 0.f ? 1.f / l : 0.f;
  }
  cluster_wait();
  for (int e = tid; e < kHeads * (int)S; e += AD_THREADS) {
    const int h = e % kHeads;
    const uint32_t q = e / kHeads;
    const float m = first ? -INFINITY : M->st.m[h];
    const float l =
        first ? 0.f : (M->red_l[0][h] + M->red_l[1][h]) + (M->red_l[2][h] + M->red_l[3][h]);
    st_peer_f32(peer_addr(&M->m_all[s][h], q), m);
    st_peer_f32(peer_addr(&M->l_all[s][h], q), l);
  }
  __syncthreads();
  // output slices: CTA r normalises units [slice_lo(r), slice_lo(r + 1)) of
  // 8 channels; peers send it their part of that slice into its (now free) q
  // buffer, one region per sender (regions of senders above r move down one,
  // so S - 1 regions of kUnits / S + 1 units fit in the 64 KB)
  constexpr int kUnits = kHeads * kHeadDim / 8;
  auto slice_lo = [&](uint32_t r) { return (int)((long long)kUnits * r / S); };
  const int u0 = slice_lo(s), u1 = slice_lo(s + 1);
  const uint32_t region = (uint32_t)(kUnits / S + 1) * 16;  // bytes per sender
  if (tid == 0) tc::mbar_arrive_expect_tx(&M->recv_bar, (uint32_t)(u1 - u0) * 16 * (S - 1));
  if (first) {
    // no candidates here: a zero partial, so that peers may read it unmasked
    for (int e = tid; e < kHeads * kHeadDim / 8; e += AD_THREADS)
      reinterpret_cast<uint4 *>(Os)[e] = make_uint4(0u, 0u, 0u, 0u);
  } else {
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    float il[32];
    load32(M->inv_l + h0, il);
#pragma unroll 1
    for (int m4 = 0; m4 < 4; ++m4) {
      float v[32];
      tc::tmem_ld32(tmem + lane_off + O_COL + m4 * 64 + h0, v);
      const int d = m4 * 128 + qd * 32 + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        Os[(h0 + j) * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j] * il[j]));
    }
  }
  tc::fence_async_shared();  // the parked partial is read by the bulk copies
  tc::tc_fence_before();
  cluster_sync();
  if (tid == 0)
    for (uint32_t r = 0; r < S; ++r) {
      if (r == s) continue;
      const int lo = slice_lo(r), hi = slice_lo(r + 1);
      const uint32_t slot = s < r ? s : s - 1;
      bulk_to_peer(Os + (size_t)lo * 8, tc::smem_u32(Qs) + slot * region, (uint32_t)(hi - lo) * 16,
                   &M->recv_bar, r);
    }

  // ---- merge weights: one thread per head, from the statistics every CTA sent
  if (tid < kHeads) {
    const int h = tid;
    const float s2 = sink2;
    float mx = s2;
    for (uint32_t q = 0; q < S; ++q) mx = fmaxf(mx, M->m_all[q][h]);
    float L = 0.f;
    if (mx != -INFINITY) {
      L = exp2f(s2 - mx);
      for (uint32_t q = 0; q < S; ++q) {
        const float mq = M->m_all[q][h];
        const float w = mq == -INFINITY ? 0.f : exp2f(mq - mx);
        M->w_all[q][h] = w * M->l_all[q][h];  // the partial was parked divided by l
        L += w * M->l_all[q][h];
      }
    } else {
      for (uint32_t q = 0; q < S; ++q) M->w_all[q][h] = 0.f;
    }
    M->inv_L[h] = L > 0.f ? 1.f / L : 0.f;
    if (s == 0 && a.lse)
      a.lse[(long long)t * kHeads + h] = L > 0.f ? (mx + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();

  // ---- this CTA's slice of the output, 8 channels per step: its own part
  // from the parked partial, the peers' parts from the receive regions
  if (S > 1 && !tc::mbar_wait(&M->recv_bar, 0)) flag(a.status_dev, CSA_DEV_TIMEOUT);
  const bool inv = a.inv_rope_out && a.rope_cos != nullptr && p >= 0 && p < a.rope_cap;
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + (long long)t * kHeads * kHeadDim;
  for (int u = u0 + tid; u < u1; u += AD_THREADS) {
    const int h = u / (kHeadDim / 8), d = (u % (kHeadDim / 8)) * 8;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (uint32_t q = 0; q < S; ++q) {
      const uint32_t slot = q < s ? q : q - 1;
      const uint4 v = q == s ? reinterpret_cast<const uint4 *>(Os)[u]
                             : *reinterpret_cast<const uint4 *>(Qs + slot * region + (u - u0) * 16);
      const float w = M->w_all[q][h];
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[2 * i] = fmaf(w, __uint_as_float(wd[i] << 16), o[2 * i]);
        o[2 * i + 1] = fmaf(w, __uint_as_float(wd[i] & 0xFFFF0000u), o[2 * i + 1]);
      }
    }
    const float il = M->inv_L[h];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= il;
    if (inv && d >= kHeadDim - kRopeDim) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pair = (d + 2 * i - (kHeadDim - kRopeDim)) >> 1;
        const float cs = a.rope_cos[(long long)p * kRopeHalf + pair];
        const float sn = a.rope_sin[(long long)p * kRopeHalf + pair];
        const float x0 = o[2 * i], x1 = o[2 * i + 1];
        o[2 * i] = x0 * cs + x1 * sn;
        o[2 * i + 1] = -x0 * sn + x1 * cs;
      }
    }
    *reinterpret_cast<uint4 *>(out + h * kHeadDim + d) =
        make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
  }
  // this CTA's outgoing copies have landed once every peer is through its wait
  cluster_sync();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// Largest cluster the decode kernel may use on this device (16 where the
// device schedules it, else the portable 8).
int max_cluster() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 8;
  if (!cached[dev]) {
    int best = 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(AD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = AD_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 16;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, attn_decode_kernel, &cfg) == cudaSuccess && n > 0)
      best = 16;
    cudaGetLastError();  // a refused query leaves no error behind
    cached[dev] = best;
  }
  return cached[dev];
}

// Opt the kernel into its shared memory, once per device.
cudaError_t prepare_kernel() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(
      attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

}  // namespace

void attn_decode_geometry(const csa_attn_args &a, int *n_splits, int *tiles_per_split) {
  const int tiles = (a.topk + a.window + CT - 1) / CT;
  const int mc = prepare_kernel() == cudaSuccess ? max_cluster() : 8;
  const int tps = (tiles + mc - 1) / mc;
  *tiles_per_split = tps;
  *n_splits = (tiles + tps - 1) / tps;
}

cudaError_t launch_attn_decode(const csa_attn_args &a, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  if (!encode_rows_map(&qmap, a.q, (long long)a.n_rows * kHeads, kHeads))
    return cudaErrorInvalidValue;
  cudaError_t e = prepare_kernel();
  if (e != cudaSuccess) return e;
  int n_splits, tps;
  attn_decode_geometry(a, &n_splits, &tps);
  launch_begin(CSA_K_ATTN_DECODE, s);
  e = launch_kernel(attn_decode_kernel, dim3(n_splits, a.n_rows), dim3(AD_THREADS),
                    (size_t)AD_SMEM, s, n_splits, false, a, tps, qmap);
  launch_end(CSA_K_ATTN_DECODE, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
