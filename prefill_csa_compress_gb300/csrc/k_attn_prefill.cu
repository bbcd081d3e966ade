// Prefill shared-KV sparse attention with an attention sink: a persistent,
// warp-specialised tcgen05 pipeline.  Same function as the split kernel in
// k_attn.cu ("Hyper-Parallel ... DeepSeek V4 CP" (gitcode issue #2),
// "二阶段 CP 总体算法": Stage-2 sparse attention with sinks, softmax_scale and
// ori_win_left = 127, outputs out and lse; "9.1": the candidates are the
// selected compressed entries followed by the raw causal window; "7. Window KV
// Halo": the window includes the query's own position).
//
// One CTA per SM walks query rows; per row the candidates are processed in
// tiles of 128 with the candidates on the MMA's M side and the 64 heads on N:
//   S^T[c, h]  = K[c, :] . q_h              (A = gathered tile, K-major)
//   O^T[d, h] += sum_c K[c, d] P[c, h]      (A = same tile read MN-major)
// Roles:
//   warp 0      producer: resolves each tile's candidates to pool-row
//               addresses (a two-slot table in shared memory) and loads each
//               row's q with TMA;
//   warp 1      MMA issuer (one elected lane);
//   warps 2..9  softmax, gather and epilogue; thread = (candidate, half of the
//               heads).  Right after handing tile i's P to the MMA they gather
//               tile i+1 with 16-byte cp.async straight into the
//               128-byte-swizzled layout (eight lanes per 128-byte row slice,
//               so each warp request covers whole sectors): warps 2m, 2m+1
//               refill the 128-channel pair m as soon as tile i's P.V has
//               finished reading it and mark it landed on their own, and the
//               MMA starts QK^T on each pair as it lands.  The running maximum per head only moves (and O^T is
//               rescaled in TMEM) when a tile's logits exceed it by more than
//               2^8; checking that costs one barrier reduction per tile.  FP32
//               denominators come from a warp reduce-scatter.  At the end of a
//               row they normalise O^T out of TMEM and store the output.
// TMEM: S^T in columns [0, 64), O^T (four 128-channel tiles) in [64, 320).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "attn_common.cuh"

namespace csa {
namespace {

constexpr int AP_THREADS = 320;
constexpr int AP_PROD_WARP = 0;
constexpr int AP_MMA_WARP = 1;
constexpr int AP_SOFT0 = 2;   // first softmax warp
constexpr int AP_SOFT = 256;  // softmax / gather / epilogue threads (warps 2..9)
constexpr int AP_BAR = 1;     // their named barrier
using namespace attn;

struct ApRow {
  int t, p, b;
  int h_lo;        // first head of the item's group of 64 heads
  uint32_t tiles;  // bit g: tile g of the row's candidate list is processed
};

struct ApMisc {
  uint64_t q_full, q_rot, q_empty, s_full, p_full, o_full, o_empty, mma_done;
  uint64_t kv_full[4];   // one per pair of chunks, arrived by the two warps that copy it
  uint64_t kv_empty[4];  // one per pair of chunks (one 128-channel tile of P.V)
  uint64_t tab_full[2];   // the producer filled the tile's address table
  uint64_t tab_empty[2];  // the gatherers have read it
  uint32_t tmem_base;
  int abort;
  ApRow row[2];
  int32_t tbl[64];            // the row's compressed-page table (up to 64 pages)
  const uint16_t *src[2][CT];  // pool row of each candidate of the tile, or null
  SoftState st;
  alignas(16) float inv_s[kHeads];
  alignas(16) float red_l[4][kHeads];
};
constexpr int AP_SMEM = OFF_MISC + (int)sizeof(ApMisc) + 1024;
static_assert(AP_SMEM <= 227 * 1024, "shared memory");

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool ap_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                        uint32_t *status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_ns();
  for (uint32_t i = 1;; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (tc::global_ns() - t0 > 2000000000ull) {
        *abort = 1;
        flag(status, CSA_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Softmax of one tile (thread = candidate c = qd*32 + lane, heads h0..h0+31)
// that speculates that no logit moves the running reference: P is computed
// with the current reference and the block-wide "exceeded" test rides on the
// barrier that hands P to the MMA.  On a row's first tile, or when some
// valid logit exceeded its reference by more than 2^8, the tile reloads its
// logits (S^T stays in TMEM until P is handed over) and takes the reference
// move of softmax_vals, which rewrites P.  Returns past that final barrier
// with P stored and fenced for the MMA; x holds this thread's probabilities.
__device__ __forceinline__ void softmax_tile_spec(uint32_t tmem, int qd, int h0, bool valid,
                                                  float sl2, bool first, SoftState *st,
                                                  uint8_t *Ps, int bar, float &lacc,
                                                  float (&x)[32]) {
  const int lane = threadIdx.x & 31, c = qd * 32 + lane;
  const uint32_t s_addr = tmem + ((uint32_t)(qd * 32) << 16) + S_COL + h0;
  tc::tc_fence_after();
  tc::tmem_ld32(s_addr, x);
  if (!first) {
    float mref[32];
    load32(st->m + h0, mref);
    bool exceed = false;
    if (valid) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float t = x[j] * sl2 - mref[j];
        exceed |= t > kRescaleLog2;
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
    tc::fence_async_shared();
    tc::tc_fence_before();
    if (!tc::bar_or(bar, 256, exceed)) return;
    tc::tc_fence_after();
    tc::tmem_ld32(s_addr, x);
  }
  softmax_vals(tmem, O_COL, 4, qd, h0, valid, sl2, first, st, Ps, bar, lacc, x, [] {});
  tc::fence_async_shared();
  tc::tc_fence_before();
  tc::bar_sync(bar, 256);
}

__global__ void __launch_bounds__(AP_THREADS, 1)
    attn_prefill_kernel(csa_attn_args a, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t *Qs = sm + OFF_Q;
  uint8_t *KVs = sm + OFF_KV;
  uint8_t *Ps = sm + OFF_P;
  ApMisc *M = reinterpret_cast<ApMisc *>(sm + OFF_MISC);
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_cand = a.topk + a.window;
  volatile int *abort = &M->abort;

  if (tid == 0) {
    tc::mbar_init(&M->q_full, 1);
    tc::mbar_init(&M->q_rot, 1);
    tc::mbar_init(&M->q_empty, 1);
    tc::mbar_init(&M->s_full, 1);
    tc::mbar_init(&M->p_full, 1);
    tc::mbar_init(&M->o_full, 1);
    tc::mbar_init(&M->o_empty, 1);
    tc::mbar_init(&M->mma_done, 1);
    for (int i = 0; i < 4; ++i) tc::mbar_init(&M->kv_full[i], 64);
    for (int i = 0; i < 4; ++i) tc::mbar_init(&M->kv_empty[i], 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&M->tab_full[i], 32);
      tc::mbar_init(&M->tab_empty[i], AP_SOFT / 32);
    }
    M->abort = 0;
    tc::mbar_fence_init();
  }
  if (tid < kHeads) M->st.m[tid] = -INFINITY;
  if (warp == AP_MMA_WARP) tc::tmem_alloc(&M->tmem_base, TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = M->tmem_base;

  // The items this CTA serves: w = blockIdx.x + i * gridDim.x, item w being
  // row w / HG with its group w % HG of 64 heads (heads past n_heads are
  // computed from padding -- every head's column is independent -- and never
  // stored), for rows with a valid request.
  const int HG = (a.n_heads + kHeads - 1) / kHeads;
  const int n_items = a.n_rows * HG;
  auto next_row = [&](int w) {
    for (w += gridDim.x; w < n_items; w += gridDim.x) {
      const int b = a.row_req[w / HG];
      if (b >= 0 && b < a.n_req) return w;
    }
    return n_items;
  };
  const int first_row = next_row((int)blockIdx.x - (int)gridDim.x);

  if (warp == AP_PROD_WARP) {
    // ================================================================ producer
    uint32_t row_it = 0, tile_it = 0, q_loads = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
      const int t = w / HG, h_lo = (w % HG) * kHeads;
      const int b = a.row_req[t];
      if (b < 0) continue;
      if (b >= a.n_req) {
        if (lane == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
        continue;
      }
      if (!ok) break;
      const int p = a.row_pos[t];
      const int V = min(visible_count(p, a.ratio, a.n_cmp[b]), a.cmp_max_blocks * kBlock);
      const int kvl = a.kv_len[b];
      // the row's selection, or (no selection: dense visibility) entries 0 .. V-1
      const int32_t *sel = a.topk_idx ? a.topk_idx + (long long)t * a.topk : nullptr;
      if (!sel && V > a.topk && lane == 0) flag(a.status_dev, CSA_DEV_BAD_INDEX);
      // the row's compressed-page table, read once (tables of up to 64 pages)
      const bool cache_tbl = a.cmp_max_blocks <= 64;
      __syncwarp();
      if (cache_tbl)
        for (int i = lane; i < a.cmp_max_blocks; i += 32)
          M->tbl[i] = a.cmp_block_table[(long long)b * a.cmp_max_blocks + i];
      // tiles holding at least one candidate; out-of-range entries are flagged once
      uint32_t mine = 0;
      for (int j0 = 0; j0 < a.topk; j0 += 16 * 32) {
        int c[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = j0 + 32 * u + lane;
          c[u] = j < a.topk ? (sel ? sel[j] : (j < V ? j : -1)) : -1;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = j0 + 32 * u + lane;
          if (c[u] >= 0 && c[u] < V) mine |= 1u << (j / CT);
          if (c[u] >= V) flag(a.status_dev, CSA_DEV_BAD_INDEX);
        }
      }
      for (int j = a.topk + lane; j < n_cand; j += 32) {
        const int pp = p - a.window + 1 + (j - a.topk);
        if (pp >= 0 && pp < kvl) mine |= 1u << (j / CT);
        if (pp >= kvl) flag(a.status_dev, CSA_DEV_BAD_POS);
      }
      uint32_t tiles = __reduce_or_sync(0xffffffffu, mine);
      if (!tiles) tiles = 1u << ((n_cand - 1) / CT);  // an all-empty tile still yields out = 0
      __syncwarp();
      for (uint32_t mm = tiles; mm && ok; mm &= mm - 1) {
        const int g0 = (__ffs(mm) - 1) * CT;
        const int slot = tile_it & 1;
        ok = __all_sync(0xffffffffu, ap_wait(&M->tab_empty[slot], ((tile_it >> 1) & 1) ^ 1, abort,
                                             a.status_dev));
        if (!ok) break;
        int c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = g0 + 32 * u + lane;
          c[u] = j < a.topk ? (sel ? sel[j] : (j < V ? j : -1)) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = g0 + 32 * u + lane;
          long long row = -1;
          const void *pool = a.kv_pool;
          long long ps = a.kv_page_stride, rs = a.kv_row_stride;
          if (j < a.topk) {
            pool = a.cmp_pool;
            ps = a.cmp_page_stride;
            rs = a.cmp_row_stride;
            if (c[u] >= 0 && c[u] < V) {
              if (cache_tbl) {
                const int phys = M->tbl[c[u] / kBlock];
                if (phys >= 0 && phys < a.cmp_n_blocks)
                  row = (long long)phys * kBlock + (c[u] % kBlock);
                else
                  flag(a.status_dev, CSA_DEV_BAD_BLOCK);
              } else {
                row = page_row(a.cmp_block_table, a.cmp_max_blocks, a.cmp_n_blocks, b, c[u],
                               a.status_dev);
              }
            }
          } else if (j < n_cand) {
            const int pp = p - a.window + 1 + (j - a.topk);
            if (pp >= 0 && pp < kvl)
              row = page_row(a.kv_block_table, a.kv_max_blocks, a.kv_n_blocks, b, pp,
                             a.status_dev);
          }
          M->src[slot][32 * u + lane] =
              row < 0 ? nullptr
                      : reinterpret_cast<const uint16_t *>(static_cast<const uint8_t *>(pool) +
                                                           pool_offset(row, ps, rs));
        }
        tc::mbar_arrive(&M->tab_full[slot]);
        if (mm == tiles) {
          // the row's q, once the previous row's last QK^T has read its own
          ok = __all_sync(0xffffffffu, ap_wait(&M->q_empty, (row_it & 1) ^ 1, abort, a.status_dev));
          if (ok && lane == 0) {
            ApRow &R = M->row[row_it & 1];
            R.t = t;
            R.p = p;
            R.b = b;
            R.h_lo = h_lo;
            R.tiles = tiles;
            tc::mbar_arrive_expect_tx(&M->q_full, 8 * 8192);
            for (int kc = 0; kc < 8; ++kc)
              tc::tma_load_2d(Qs + kc * 8192, &qmap, kc * 64, t * a.n_heads + h_lo, &M->q_full);
          }
          if (ok) ++q_loads;
          __syncwarp();
        }
        ++tile_it;
      }
      ++row_it;
    }
    // a q load still in flight lands before the CTA retires
    if (!ok && q_loads) tc::mbar_wait(&M->q_full, (q_loads - 1) & 1, 50000000ull);
  } else if (warp == AP_MMA_WARP) {
    // ================================================================ MMA issuer
    const uint32_t kv = tc::smem_u32(KVs), qq = tc::smem_u32(Qs), pp = tc::smem_u32(Ps);
    uint32_t row_it = 0, tile_it = 0;
    bool ok = true;
    for (int t = first_row; t < n_items && ok; t = next_row(t)) {
      ok = __all_sync(0xffffffffu, ap_wait(&M->q_full, row_it & 1, abort, a.status_dev));
      if (!ok) break;
      const uint32_t tiles = M->row[row_it & 1].tiles;
      bool first = true;
      for (uint32_t mm = tiles; mm && ok; mm &= mm - 1) {
        const bool last = (mm & (mm - 1)) == 0;
        // QK^T pair by pair as the gather lands them: wait for the next
        // chunk pair, take every later pair that has landed as well, and
        // issue the batch behind one tcgen05 fence (a fence per chunk drains
        // the MMA pipe and halves its rate).
        for (int kp = 0; kp < 4 && ok;) {
          ok = __all_sync(0xffffffffu, ap_wait(&M->kv_full[kp], tile_it & 1, abort, a.status_dev));
          if (!ok) break;
          int ke = kp + 1;
          while (ke < 4 && __all_sync(0xffffffffu, tc::mbar_test_wait(&M->kv_full[ke], tile_it & 1)))
            ++ke;
          if (first && ke == 4)  // the row's q, rotated (its last chunk), before chunk 7
            ok = __all_sync(0xffffffffu, ap_wait(&M->q_rot, row_it & 1, abort, a.status_dev));
          if (!ok) break;
          tc::tc_fence_after();
          for (; kp < ke; ++kp) {
            issue_qk(tmem, kv, qq, 2 * kp);
            issue_qk(tmem, kv, qq, 2 * kp + 1);
          }
        }
        if (!ok) break;
        tc::mma_commit_elect(&M->s_full);
        if (last) tc::mma_commit_elect(&M->q_empty);
        if (first) {
          ok = __all_sync(0xffffffffu,
                          ap_wait(&M->o_empty, (row_it & 1) ^ 1, abort, a.status_dev));
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, ap_wait(&M->p_full, tile_it & 1, abort, a.status_dev));
        if (!ok) break;
        tc::tc_fence_after();
        for (int mt = 0; mt < 4; ++mt) {
          issue_pv(tmem, kv, pp, mt, !first);
          tc::mma_commit_elect(&M->kv_empty[mt]);
        }
        if (last) tc::mma_commit_elect(&M->o_full);
        first = false;
        ++tile_it;
      }
      ++row_it;
    }
    // every issued MMA has completed before TMEM is released
    tc::mma_commit_elect(&M->mma_done);
    tc::mbar_wait(&M->mma_done, 0, 100000000ull);
  } else {
    // ================================================================ softmax / gather / epilogue
    const int sw = warp - AP_SOFT0;         // 0..7
    const int qd = warp & 3;                // TMEM lane quarter of this warp
    const int h0 = (sw >> 2) * 32;          // first head of this thread's half
    const int c = qd * 32 + lane;           // candidate = TMEM lane
    const int stid = sw * 32 + lane;        // 0..255
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float sl2 = a.softmax_scale * kLog2e;
    // gather: this thread copies 16-byte piece `piece` of rows
    // 8 j + 4 (sw & 1) + sub (j < 16) of chunk pair sw / 2
    const int sub = lane >> 3, piece = lane & 7;
    uint32_t row_it = 0, tile_it = 0;
    bool ok = true;

    // Gather tile `it` (its address table in slot it & 1) into the KV buffer.
    // Warps 2m and 2m+1 of the group copy chunk pair m (channels 128m ..
    // 128m + 127 of all 128 candidates) as soon as tile it - 1's P.V has
    // released it, wait for their own copies and mark the pair landed: QK^T
    // starts on the first pairs while the later ones are still in flight.
    // Returns this thread's candidate validity for the tile; `mid()` runs
    // while the copies fly.
    auto gather = [&](uint32_t it, auto &&mid) -> bool {
      const int slot = it & 1, grp = sw >> 1;
      const int r0 = (sw & 1) * 4 + sub;  // this thread's rows: r0 + 8 j
      bool good = ap_wait(&M->tab_full[slot], (it >> 1) & 1, abort, a.status_dev);
      const bool my_valid = M->src[slot][c] != nullptr;
      if (good) good = ap_wait(&M->kv_empty[grp], (it & 1) ^ 1, abort, a.status_dev);
      if (good) {
        uint8_t *dst = KVs + 2 * grp * 16384 + r0 * 128 + ((piece ^ r0) << 4);
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const uint16_t *row = M->src[slot][8 * j + r0];
          const uint16_t *g =
              row ? row + grp * 128 + piece * 8 : static_cast<const uint16_t *>(a.kv_pool);
          tc::cp_async16_zfill(dst + j * 1024, g, row != nullptr);
          tc::cp_async16_zfill(dst + j * 1024 + 16384, row ? g + 64 : g, row != nullptr);
        }
      }
      tc::cp_async_commit();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&M->tab_empty[slot]);
      mid();
      tc::cp_async_wait<0>();
      if (good) {
        tc::fence_async_shared();
        tc::mbar_arrive(&M->kv_full[grp]);
      }
      ok = ok && good;
      return my_valid;
    };

    // Wait for the q of row iteration `it`, rotate its last 64 channels at p
    // (FP32, rounded to BF16) in place and release it to the MMA.
    auto rope_row = [&](uint32_t it, ApRow &R) {
      ok = tc::bar_and(AP_BAR, AP_SOFT, ok && ap_wait(&M->q_full, it & 1, abort, a.status_dev));
      if (!ok) return;
      R = M->row[it & 1];
      bool rot = a.rope_cos != nullptr && R.p >= 0;
      if (rot && R.p >= a.rope_cap) {
        rot = false;
        if (stid == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
      }
      if (rot) {
        rope_q_rows(Qs + 7 * 8192, a.rope_cos + (long long)R.p * kRopeHalf,
                    a.rope_sin + (long long)R.p * kRopeHalf, stid, AP_SOFT);
        tc::fence_async_shared();
      }
      tc::bar_sync(AP_BAR, AP_SOFT);
      if (stid == 0) tc::mbar_arrive(&M->q_rot);
    };

    bool valid = false;
    ApRow R_next;
    if (first_row < n_items) {
      valid = gather(0, [] {});
      rope_row(0, R_next);
    }
    for (int t = first_row; t < n_items && ok; t = next_row(t)) {
      const ApRow R = R_next;
      bool first = true;
      float lacc = 0.f;  // this warp's partial denominator of head h0 + lane
      for (uint32_t mm = R.tiles; mm && ok; mm &= mm - 1) {
        ok = tc::bar_and(AP_BAR, AP_SOFT, ok && ap_wait(&M->s_full, tile_it & 1, abort, a.status_dev));
        if (!ok) break;
        float x[32];
        softmax_tile_spec(tmem, qd, h0, valid, sl2, first, &M->st, Ps, AP_BAR, lacc, x);
        if (stid == 0) tc::mbar_arrive(&M->p_full);
        // FP32 denominators (this warp's per-head sums of the unrounded
        // probabilities, lane l: head h0 + l) while the next tile is gathered
        auto colsum = [&] { lacc += warp_col_reduce32<false>(x); };
        const bool more = (mm & (mm - 1)) != 0 || next_row(t) < n_items;
        if (more)
          valid = gather(tile_it + 1, colsum);
        else
          colsum();
        first = false;
        ++tile_it;
      }
      if (!ok) break;
      // the next row's q is rotated before this row's epilogue, so that its
      // first QK^T does not wait for the output stores
      if (next_row(t) < n_items) {
        rope_row(row_it + 1, R_next);
        if (!ok) break;
      }

      // ---- epilogue: out = O^T / L, lse = log L, with the sink in L
      ok = tc::bar_and(AP_BAR, AP_SOFT, ap_wait(&M->o_full, row_it & 1, abort, a.status_dev));
      if (!ok) break;
      M->red_l[qd][h0 + lane] = lacc;
      tc::bar_sync(AP_BAR, AP_SOFT);
      const int nh = min(kHeads, a.n_heads - R.h_lo);  // stored heads of this item
      if (qd == 0) {
        const int h = h0 + lane;
        const float s2 = a.sink && h < nh ? a.sink[R.h_lo + h] * kLog2e : -INFINITY;
        float m = M->st.m[h];
        float l = (M->red_l[0][h] + M->red_l[1][h]) + (M->red_l[2][h] + M->red_l[3][h]);
        if (m == -INFINITY) {
          m = s2;
          l = 0.f;
        }
        const float L = (m == -INFINITY) ? 0.f : l + exp2f(s2 - m);
        M->inv_s[h] = L > 0.f ? 1.f / L : 0.f;
        if (a.lse && h < nh)
          a.lse[(long long)R.t * a.n_heads + R.h_lo + h] =
              L > 0.f ? (m + log2f(L)) * kLn2 : -INFINITY;
      }
      tc::bar_sync(AP_BAR, AP_SOFT);
      float inv[32];
      load32(M->inv_s + h0, inv);
      const bool inv_rope = a.inv_rope_out && a.rope_cos != nullptr && R.p >= 0 && R.p < a.rope_cap;
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) +
                           ((long long)R.t * a.n_heads + R.h_lo) * kHeadDim;
      tc::tc_fence_after();
      // the inverse rotation touches channels 448.. only: warps of lane
      // quarters 2 and 3 in the last slice (every branch below is warp-uniform
      // and sits outside the per-head loops)
      const bool rot_warp = inv_rope && qd >= 2;
      float cs = 1.f, sn = 0.f;
      if (rot_warp) {
        const int pair = (qd * 32 + lane - 64) >> 1;
        cs = a.rope_cos[(long long)R.p * kRopeHalf + pair];
        sn = a.rope_sin[(long long)R.p * kRopeHalf + pair];
      }
      const bool all_heads = h0 + 32 <= nh;
#pragma unroll 1
      for (int m4 = 0; m4 < 4; ++m4) {
        float v[32];
        tc::tmem_ld32(tmem + lane_off + O_COL + m4 * 64 + h0, v);
        const int d = m4 * 128 + qd * 32 + lane;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= inv[j];
        if (m4 == 3 && rot_warp) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            v[j] = (lane & 1) ? (-other * sn + v[j] * cs) : (v[j] * cs + other * sn);
          }
        }
        __nv_bfloat16 *o = out + h0 * kHeadDim + d;
        if (all_heads) {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j * kHeadDim] = __float2bfloat16_rn(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (h0 + j < nh) o[j * kHeadDim] = __float2bfloat16_rn(v[j]);
        }
      }
      tc::tc_fence_before();
      tc::bar_sync(AP_BAR, AP_SOFT);
      if (stid == 0) tc::mbar_arrive(&M->o_empty);
      if (qd == 0) M->st.m[h0 + lane] = -INFINITY;
      ++row_it;
    }
    tc::cp_async_wait<0>();
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == AP_MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

}  // namespace

namespace attn {
bool encode_rows_map(CUtensorMap *map, const void *base, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode || rows <= 0 || rows > 0x7FFFFFFFll) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}
}  // namespace attn

bool attn_prefill_supported(const csa_attn_args &a) { return a.topk + a.window <= 32 * CT; }

cudaError_t launch_attn_prefill(const csa_attn_args &a, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  if (!encode_rows_map(&qmap, a.q, (long long)a.n_rows * a.n_heads, kHeads))
    return cudaErrorInvalidValue;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AP_SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  const long long items = (long long)a.n_rows * ((a.n_heads + kHeads - 1) / kHeads);
  const int grid = items < sms ? (int)items : sms;
  launch_begin(CSA_K_ATTN_PREFILL, s);
  const cudaError_t e = launch_kernel(attn_prefill_kernel, dim3(grid), dim3(AP_THREADS),
                                      (size_t)AP_SMEM, s, 0, false, a, qmap);
  launch_end(CSA_K_ATTN_PREFILL, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
