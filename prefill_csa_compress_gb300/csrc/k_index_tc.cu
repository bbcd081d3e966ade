// Lightning-indexer scores on the 5th-generation tensor cores.
//
// score[t, c] = scale_c * sum_h w[t,h] * act(q_{t,h} . k_c) for every visible
// compressed entry c of row t ("Hyper-Parallel ... DeepSeek V4 CP", "10. ratio=4
// Global Top-k" and "10.3 Causal mask"; INT8 keys with an FP32 per-row scale,
// "DeepSeek V4-Flash, MTP point", "What is quantized").
//
// GB300 mapping.  The contraction runs with the KEYS as the MMA's M side: one
// 128-row key page is one M=128 tile, so TMEM lane r holds key r and its
// columns hold the dot products with the G rows x 64 heads of a row group
// (N = 64G).  The head reduction then happens inside one thread with no
// cross-lane traffic.  A CTA streams the pages of one request:
//   warp 12     bulk-copies each INT8 page (16 KB) and its scales into a ring,
//   warps 4..11 convert INT8 -> FP16 (exact, 10 instructions per 8 keys) into
//               the 128-byte-swizzled K-major layout (a ring of A tiles),
//   warp 13     issues tcgen05.mma (A = keys, B = queries) into a ring of
//               TMEM accumulators (all 512 columns),
//   warps 0..3  read TMEM and apply ReLU, the head weights and the key scale;
//               with warp 13 they also build the query operand at the start
//               of each pass while the first pages are already in flight.
// The queries enter the MMA as FP16: each (row, head) is scaled by a power of
// two that puts its largest |q| in [2^13, 2^14) (exact; the inverse factor is
// folded into that head's weight, since ReLU(2^e x) = 2^e ReLU(x)).  The RoPE
// half, rotated in FP32, is split into FP16 hi + lo parts so that the product
// keeps FP32-level accuracy (K = 64 + 64 + 64).
#include <cuda.h>
#include <cstring>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "csa_internal.cuh"
#include "lowbit.cuh"
#include "tc.cuh"

namespace csa {
namespace {

// warps 0..7: epilogue (two warps per TMEM sub-partition, split by row);
// warps 8..15: converters; warp 16: producer; warp 17: MMA issuer.  All
// warps but the producer build the query operand at the start of a pass.
constexpr int IT_THREADS = 576;
constexpr int IT_EPI = 256;       // epilogue threads
constexpr int IT_CONV = 256;      // converter threads
constexpr int IT_BUILD = 544;     // query builders: every warp but the producer
constexpr int W_CONV0 = 8, W_PROD = 16, W_MMA = 17;

template <int G>
struct IdxTc {
  // G == 2 (decode row pairs): the converted keys go to TMEM as the MMA's A
  // operand, which keeps shared memory for the page ring and the queries.
  // G == 4 (prefill): N = 256 fills TMEM with accumulators; A stays in smem.
  static constexpr bool ATMEM = G == 2;
  static constexpr int N = G * kHeads;            // MMA N
  static constexpr int NS = ATMEM ? 8 : 3;        // staging ring depth
  static constexpr int NA = 2;                    // converted A tiles
  static constexpr int NT = ATMEM ? 3 : 2;        // TMEM accumulator slots
  static constexpr int NSC = 8;                   // scale ring: > NA + NT tiles in flight
  static constexpr int A_COL = 0;                 // TMEM A tiles (64 columns each)
  static constexpr int ACC_COL = ATMEM ? NA * 64 : 0;
  static constexpr int B_CHUNK = N * 128;         // bytes of one 64-wide K chunk of B
  static constexpr int A_CHUNK = kBlock * 128;    // 16 KB
  static constexpr int A_BUF = 2 * A_CHUNK;       // 128 keys x 128 dims fp16
  static constexpr int PAGE = kBlock * kIdxDim;   // 16 KB of int8 keys
  static constexpr int OFF_B = 0;
  static constexpr int OFF_A = OFF_B + 3 * B_CHUNK;
  static constexpr int OFF_ST = OFF_A + (ATMEM ? 0 : NA * A_BUF);
  static constexpr int OFF_STSC = OFF_ST + NS * PAGE;
  static constexpr int OFF_SC = OFF_STSC + NS * kBlock * 4;
  static constexpr int OFF_W = OFF_SC + NSC * kBlock * 4;
  static constexpr int OFF_ROPE = OFF_W + G * kHeads * 4;   // per row: 32 cos, 32 sin
  static constexpr int OFF_GQ = OFF_ROPE + G * 64 * 4;      // reindex: looked-up blocks
  static constexpr int GQ_TILES = 16;                        // tiles per look-up batch
  static constexpr int OFF_MISC = OFF_GQ + GQ_TILES * (kBlock / 8) * 4;
  static constexpr int SMEM = OFF_MISC + 512 + 1024;        // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(NA + NT < NSC, "the scale ring must outlast the tiles in flight");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct IdxMisc {
  uint64_t st_full[8];
  uint64_t st_empty[8];
  uint64_t a_full[3];    // converters -> MMA
  uint64_t a_free[3];    // MMA commit -> converters (A tile may be overwritten)
  uint64_t acc_full[4];  // MMA commit -> epilogue
  uint64_t acc_empty[4]; // epilogue -> MMA (accumulator may be overwritten)
  uint32_t tmem_base;
  int st_ok[8];
  int t_ok[8];           // per scale slot: the page was valid
  volatile int abort;
  int row_t[4];
  int row_V[4];
  int row_on[4];
  int row_p[4];
  int cand_min;
};

__device__ __forceinline__ void set_abort(IdxMisc *m, uint32_t *status) {
  m->abort = 1;
  flag(status, CSA_DEV_TIMEOUT);
}

// 8 int8 -> 8 fp16, exactly: the offset-binary byte (v ^ 0x80) placed in the
// low mantissa bits of 1024.0 gives 1024 + 128 + v; subtracting 1152 leaves v.
__device__ __forceinline__ uint4 i8x8_to_f16x8(uint2 raw) {
  const uint32_t a = raw.x ^ 0x80808080u, b = raw.y ^ 0x80808080u;
  const uint32_t p[4] = {__byte_perm(a, 0x64646464u, 0x5140u), __byte_perm(a, 0x64646464u, 0x5342u),
                         __byte_perm(b, 0x64646464u, 0x5140u), __byte_perm(b, 0x64646464u, 0x5342u)};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&p[i]), bias);
    out[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Hint: bring the 128-byte line holding `p` into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void named_barrier(int id, int n_threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n_threads) : "memory");
}

// Reindex ("DeepSeek V4.1 Flash", hierarchical indexer): the number of
// leading entries of a candidate list c[0..n) that are strictly ascending
// blocks in [0, nb).  Entries after that prefix other than -1 raise
// CSA_DEV_BAD_INDEX.  Called by every thread of the CTA.
__device__ int candidate_prefix(const int32_t *c, int n, int nb, int *s_min, uint32_t *status) {
  if (threadIdx.x == 0) *s_min = n;
  __syncthreads();
  // every entry and its predecessor are loaded before any is tested (one
  // round trip for lists of up to PER * blockDim.x entries)
  constexpr int PER = 4;
  for (int j0 = 0; j0 < n; j0 += PER * (int)blockDim.x) {
    int x[PER], xp[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int j = j0 + threadIdx.x + r * blockDim.x;
      x[r] = j < n ? c[j] : 0;
      xp[r] = j > 0 && j < n ? c[j - 1] : -1;
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int j = j0 + threadIdx.x + r * blockDim.x;
      if (j < n && (x[r] < 0 || x[r] >= nb || x[r] <= xp[r])) {
        atomicMin(s_min, j);
        break;
      }
    }
  }
  __syncthreads();
  const int nv = *s_min;
  bool bad = false;
  for (int j0 = nv; j0 < n; j0 += PER * (int)blockDim.x) {
    int x[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int j = j0 + threadIdx.x + r * blockDim.x;
      x[r] = j < n ? c[j] : -1;
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) bad = bad || x[r] != -1;
  }
  if (bad) flag(status, CSA_DEV_BAD_INDEX);
  return nv;
}

template <int G, int HS>
__global__ void __launch_bounds__(IT_THREADS, 1)
    index_score_tc_kernel(csa_index_args a, float *__restrict__ scores, int cols, int n_groups,
                          int chunk_tiles, int units_per_group, uint32_t *zero_ctr,
                          const __grid_constant__ CUtensorMap keys_map, ScoreSel sel) {
  using C = IdxTc<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t *Bs = sm + C::OFF_B;
  uint8_t *As = sm + C::OFF_A;
  uint8_t *St = sm + C::OFF_ST;
  float *StSc = reinterpret_cast<float *>(sm + C::OFF_STSC);
  float *Sc = reinterpret_cast<float *>(sm + C::OFF_SC);
  float *Ws = reinterpret_cast<float *>(sm + C::OFF_W);
  float *Rope = reinterpret_cast<float *>(sm + C::OFF_ROPE);
  IdxMisc *M = reinterpret_cast<IdxMisc *>(sm + C::OFF_MISC);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  // ---- set-up that touches no global memory, overlapping the previous kernel
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      tc::mbar_init(&M->st_full[s], 1);
      tc::mbar_init(&M->st_empty[s], IT_CONV);
    }
    for (int j = 0; j < C::NA; ++j) {
      tc::mbar_init(&M->a_full[j], IT_CONV);
      tc::mbar_init(&M->a_free[j], 1);
    }
    for (int j = 0; j < C::NT; ++j) {
      tc::mbar_init(&M->acc_full[j], 1);
      tc::mbar_init(&M->acc_empty[j], IT_EPI);
    }
    M->abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == W_MMA) tc::tmem_alloc(&M->tmem_base, C::TMEM_COLS);
  tc::griddep_wait();
  tc::griddep_launch_dependents();

  const long long n_words = (long long)a.n_rows * kTopkCtlWords;
  for (int z = 0; z < 2; ++z) {
    uint32_t *ctr = z == 0 ? zero_ctr : sel.zero2;
    if (!ctr) continue;
    for (long long i = (long long)blockIdx.x * IT_THREADS + tid; i < n_words;
         i += (long long)gridDim.x * IT_THREADS)
      ctr[i] = 0u;
  }
  // reindex: a group is one row (rows do not share candidates), its tiles
  // hold 128 candidate entries (128 >> cb_shift blocks) each
  const bool reidx = sel.cand_in != nullptr;
  const int cb = 1 << sel.cb_shift;
  // The G slots of a group (64 MMA columns each) hold 64 heads of one row:
  // with up to 64 index heads a slot is a row (heads past n_heads are zero
  // queries with zero weights); with 65..128 heads a row takes two slots,
  // slot i holding heads 64 (i / RR) .. of row i % RR of the group.
  constexpr int RR = G / HS;                  // rows per group (HS: slots per row)
  const int RPG = reidx ? 1 : RR;             // rows per group actually used
  // FP4 index keys ("DeepSeek V4.1 Flash", production cache ABI): packed E2M1
  // with one E8M0 scale per 32 dims, copied linearly and decoded to FP16
  const bool fp4 = a.key_fmt == CSA_FMT_FP4_E8M0;
  // FP8 keys (the FP8 index plane, MXFP8: E4M3 codes with one E8M0 scale per
  // 32 dims): the INT8 page layout, decoded to FP16 like the FP4 keys
  const bool fp8 = a.key_fmt == CSA_FMT_MXFP8;
  const bool rope = a.rope_cos != nullptr;
  const int n_kchunks = rope ? 3 : 2;
  const int n_cap = a.max_blocks * kBlock;

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = M->tmem_base;

  uint32_t it = 0;  // running tile counter (same sequence in every role)
  const int n_units = n_groups * units_per_group;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int g = u / units_per_group;
    const int chunk = u % units_per_group;
    // requests present in the group, in order of first appearance
    int rb[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int r = i % RR;  // the slot's row in the group
      const int t = g * RPG + r;
      rb[i] = r < RPG && t < a.n_rows ? a.row_req[t] : -1;
      if (rb[i] >= a.n_req) {
        if (chunk == 0 && tid == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
        rb[i] = -1;
      }
    }
    for (int pi = 0; pi < G; ++pi) {
      const int b = rb[pi];
      bool first = b >= 0;
      if (!reidx)
        for (int j = 0; j < pi; ++j) first = first && rb[j] != b;
      if (!first) continue;

      // ---------------- pass start (all roles have finished the previous pass)
      __syncthreads();
      if (M->abort) break;
      int vmax = 0;
      unsigned on_mask = 0;  // rows of this pass
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int t = g * RPG + i % RR;
        int V = 0;
        const bool on = reidx ? i == pi : rb[i] == b;
        if (on) V = min(visible_count(a.row_pos[t], a.ratio, a.n_cmp[b]), n_cap);
        on_mask |= on ? 1u << i : 0u;
        vmax = max(vmax, V);
        if (tid == 0) {
          M->row_t[i] = t;
          M->row_V[i] = V;
          M->row_on[i] = on;
        }
      }
      const int32_t *cand = nullptr;
      if (reidx) {
        // the row's eligible entries: its valid candidate blocks, all fully
        // visible but the last, which may be cut by V
        const int t = g * RPG + pi, V = vmax;
        cand = sel.cand_in + (long long)t * sel.n_cand;
        const int nv = candidate_prefix(cand, sel.n_cand, (V + cb - 1) >> sel.cb_shift,
                                        &M->cand_min, a.status_dev);
        const int Vc = nv == 0 ? 0 : (nv - 1) * cb + min(cb, V - (cand[nv - 1] << sel.cb_shift));
        vmax = Vc;
        if (tid == 0) {
          M->row_V[pi] = Vc;
          if (chunk == 0 && sel.v_row) sel.v_row[t] = Vc;
        }
      }
      const int tiles_total = (vmax + kBlock - 1) / kBlock;
      const int tb = chunk * chunk_tiles;
      const int te = min(tiles_total, tb + chunk_tiles);
      if (tb >= te) continue;  // uniform across the CTA
      const int nt = te - tb;

      if (warp != W_PROD) {
        // ---------------- query operand (overlaps the first page copies)
        const int bt = warp < W_PROD ? tid : tid - 32;
        for (int e = bt; e < 16 * C::N; e += IT_BUILD) {
          const int n = e / 16, part = (e / 8) % 2, jj = e % 8;
          const int i = n / kHeads, hq = (i / RR) * kHeads + n % kHeads;  // head of the row
          if (((on_mask >> i) & 1u) && hq < a.n_heads)
            tc::cp_async16(Bs + part * C::B_CHUNK + n * 128 + ((jj ^ (n & 7)) << 4),
                           static_cast<const uint16_t *>(a.q_idx) +
                               ((long long)(g * RPG + i % RR) * a.n_heads + hq) * kIdxDim +
                               part * 64 + jj * 8);
        }
        // head weights, row positions and the rows' RoPE table entries
        for (int e = bt; e < G * (kHeads + 64); e += IT_BUILD) {
          const int i = e / (kHeads + 64), f = e % (kHeads + 64);
          const int t = g * RPG + i % RR;
          if (!((on_mask >> i) & 1u)) continue;
          const int p = a.row_pos[t];
          if (f < kHeads) {
            const int hq = (i / RR) * kHeads + f;
            Ws[i * kHeads + f] = hq < a.n_heads ? a.weights[(long long)t * a.n_heads + hq] : 0.f;
          } else if (rope && p >= 0 && p < a.rope_cap) {
            const int q = f - kHeads;  // 0..31 cos, 32..63 sin
            Rope[i * 64 + q] = q < 32 ? a.rope_cos[(long long)p * kRopeHalf + q]
                                      : a.rope_sin[(long long)p * kRopeHalf + q - 32];
          }
          if (f == 0) M->row_p[i] = p;
        }
        tc::cp_async_wait_all();
        named_barrier(1, IT_BUILD);
        // in place: scale the (row, head) by 2^e (its 16 pieces sit in 16
        // consecutive lanes), convert to FP16, and split the rotated half into
        // hi (chunk 1) + lo (chunk 2)
        for (int e0 = 0; e0 < 16 * C::N; e0 += IT_BUILD) {
          const int e = e0 + bt;
          const bool live = e < 16 * C::N;
          const int n = live ? e / 16 : 0, part = (e / 8) % 2, jj = e % 8;
          const int i = n / kHeads;
          const bool on = live && ((on_mask >> i) & 1u) && (i / RR) * kHeads + n % kHeads < a.n_heads;
          uint8_t *d = Bs + part * C::B_CHUNK + n * 128 + ((jj ^ (n & 7)) << 4);
          float x[8];
          float mx = 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) x[q] = 0.f;
          if (on) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(d);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              x[2 * q] = __uint_as_float(w[q] << 16);
              x[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(x[q]));
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (!live) continue;
          if (!on) {
            *reinterpret_cast<uint4 *>(d) = make_uint4(0, 0, 0, 0);
            if (part == 1) *reinterpret_cast<uint4 *>(d + C::B_CHUNK) = make_uint4(0, 0, 0, 0);
            if (part == 0 && jj == 0) Ws[n] = 0.f;
            continue;
          }
          // 2^ex puts the head's largest |q| in [2^13, 2^14); exact scaling
          int ex = 0;
          if (mx > 0.f) {
            const int E = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 126;  // mx in [2^(E-1), 2^E)
            ex = min(100, max(-100, 14 - E));
          }
          const float up = __uint_as_float((uint32_t)(127 + ex) << 23);
          if (part == 0 && jj == 0) Ws[n] *= __uint_as_float((uint32_t)(127 - ex) << 23);
          const int p = M->row_p[i];
          bool rot = part == 1 && rope && p >= 0;
          if (rot && p >= a.rope_cap) {
            rot = false;
            if ((n & 63) == 0 && jj == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
          }
          if (rot) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int pair = jj * 4 + q;
              const float c = Rope[i * 64 + pair], sn = Rope[i * 64 + 32 + pair];
              const float x0 = x[2 * q], x1 = x[2 * q + 1];
              x[2 * q] = x0 * c - x1 * sn;
              x[2 * q + 1] = x0 * sn + x1 * c;
            }
          }
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float y0 = x[2 * q] * up, y1 = x[2 * q + 1] * up;
            const __half2 hv = __floats2half2_rn(y0, y1);
            hw[q] = *reinterpret_cast<const uint32_t *>(&hv);
            lw[q] = pack_f16(y0 - __low2float(hv), y1 - __high2float(hv));
          }
          *reinterpret_cast<uint4 *>(d) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          if (part == 1)
            *reinterpret_cast<uint4 *>(d + C::B_CHUNK) =
                rot ? make_uint4(lw[0], lw[1], lw[2], lw[3]) : make_uint4(0, 0, 0, 0);
        }
        tc::fence_async_shared();
        named_barrier(1, IT_BUILD);
      }

      if (warp == W_PROD && reidx) {
        // ---------------- producer (reindex): lane jj looks up and copies
        // candidate block jj of each tile (cb rows of one page and their
        // scales); st_ok holds one bit per 8 rows that arrive
        const int nbt = kBlock >> sel.cb_shift;
        int *gq = reinterpret_cast<int *>(sm + C::OFF_GQ);
        for (int k = 0; k < nt; ++k) {
          if (k % C::GQ_TILES == 0) {
            // look up the blocks of the next GQ_TILES tiles at once: first every
            // candidate entry, then every block-table entry (two round trips)
            const int n_q = min(C::GQ_TILES, nt - k) * nbt;
            constexpr int QPL = C::GQ_TILES * (kBlock / 8) / 32;  // per lane
            int cv[QPL];
#pragma unroll
            for (int r = 0; r < QPL; ++r) {
              const int q = lane + 32 * r, j = (tb + k) * nbt + q;
              cv[r] = q < n_q && j * cb < vmax ? cand[j] : -1;
            }
            int ph[QPL];
#pragma unroll
            for (int r = 0; r < QPL; ++r)
              ph[r] = cv[r] >= 0 ? a.cmp_block_table[(long long)b * a.max_blocks +
                                                     ((cv[r] << sel.cb_shift) / kBlock)]
                                 : -1;
#pragma unroll
            for (int r = 0; r < QPL; ++r) {
              const int q = lane + 32 * r;
              if (q >= n_q) continue;
              int g_row = -1;
              if (cv[r] >= 0) {
                if (ph[r] >= 0 && ph[r] < a.n_blocks)
                  g_row = ph[r] * kBlock + ((cv[r] << sel.cb_shift) % kBlock);
                else
                  flag(a.status_dev, CSA_DEV_BAD_BLOCK);
              }
              gq[q] = g_row;
            }
            __syncwarp();
          }
          const uint32_t itk = it + k;
          const int s = itk % C::NS;
          int go = 0;
          if (lane == 0) {
            go = !M->abort;
            if (go && !tc::mbar_wait(&M->st_empty[s], ((itk / C::NS) & 1) ^ 1)) {
              set_abort(M, a.status_dev);
              go = 0;
            }
          }
          if (!__shfl_sync(0xffffffffu, go, 0)) break;
          const long long grow = lane < nbt ? gq[(k % C::GQ_TILES) * nbt + lane] : -1;
          const unsigned mask = __reduce_or_sync(
              0xffffffffu, grow >= 0 ? ((1u << (cb / 8)) - 1u) << (lane * cb / 8) : 0u);
          const int n_ok = __popc(__ballot_sync(0xffffffffu, grow >= 0));
          if (lane == 0) {
            M->st_ok[s] = (int)mask;
            if (n_ok)
              tc::mbar_arrive_expect_tx(&M->st_full[s], n_ok * cb * ((fp4 ? 64 : kIdxDim) + 4));
            else
              tc::mbar_arrive(&M->st_full[s]);
          }
          __syncwarp();
          if (grow >= 0 && fp4) {
            // FP4 keys: cb rows of 64 code bytes, cb words of scale bytes
            tc::bulk_g2s(St + s * C::PAGE + lane * cb * 64, a.idx_pool + grow * 64, cb * 64,
                         &M->st_full[s]);
            tc::bulk_g2s(StSc + s * kBlock + lane * cb, a.key_scale_pool + grow * 4, cb * 4,
                         &M->st_full[s]);
          } else if (grow >= 0) {
            uint8_t *dst = St + s * C::PAGE + lane * cb * kIdxDim;
            tc::tma_load_3d(dst, &keys_map, 0, (int)(grow & (kBlock - 1)), (int)(grow / kBlock),
                            &M->st_full[s]);
            tc::bulk_g2s(StSc + s * kBlock + lane * cb,
                         fp8 ? static_cast<const void *>(a.key_scale_pool + grow * 4)
                             : static_cast<const void *>(
                                   reinterpret_cast<const uint8_t *>(a.idx_scale_pool) +
                                   (grow / kBlock) * a.scale_page_stride + (grow & (kBlock - 1)) * 4),
                         cb * 4, &M->st_full[s]);
          }
        }
      } else if (warp == W_PROD) {
        // ---------------- producer: one page (and its scales) per tile
        if (lane == 0) {
          for (int k = 0; k < nt && !M->abort; ++k) {
            const uint32_t itk = it + k;
            const int s = itk % C::NS;
            if (!tc::mbar_wait(&M->st_empty[s], ((itk / C::NS) & 1) ^ 1)) {
              set_abort(M, a.status_dev);
              break;
            }
            const int tile = tb + k;
            const int phys = tile < a.max_blocks
                                 ? a.cmp_block_table[(long long)b * a.max_blocks + tile]
                                 : -1;
            const bool ok = phys >= 0 && phys < a.n_blocks;
            M->st_ok[s] = ok ? 0xFFFF : 0;
            if (ok && fp4) {
              // FP4 keys: 8 KB of codes and 512 bytes of scales per page
              tc::mbar_arrive_expect_tx(&M->st_full[s], kBlock * 64 + kBlock * 4);
              tc::bulk_g2s(St + s * C::PAGE, a.idx_pool + (long long)phys * kBlock * 64, kBlock * 64,
                           &M->st_full[s]);
              tc::bulk_g2s(StSc + s * kBlock, a.key_scale_pool + (long long)phys * kBlock * 4,
                           kBlock * 4, &M->st_full[s]);
            } else if (ok) {
              tc::mbar_arrive_expect_tx(&M->st_full[s], C::PAGE + kBlock * 4);
              // one page as a box of the [pages, 128, 128 B] key map (128-byte
              // swizzled rows for conflict-free row reads when A goes to TMEM);
              // keys and scales are read once: they leave L2 first
              const uint64_t once = tc::l2_evict_first();
              tc::tma_load_3d_hint(St + s * C::PAGE, &keys_map, 0, 0, phys, &M->st_full[s], once);
              tc::bulk_g2s_hint(StSc + s * kBlock,
                                fp8 ? static_cast<const void *>(a.key_scale_pool +
                                                                (long long)phys * kBlock * 4)
                                    : static_cast<const void *>(
                                          reinterpret_cast<const uint8_t *>(a.idx_scale_pool) +
                                          (long long)phys * a.scale_page_stride),
                                kBlock * 4, &M->st_full[s], once);
            } else {
              flag(a.status_dev, CSA_DEV_BAD_BLOCK);
              tc::mbar_arrive(&M->st_full[s]);
            }
          }
        }
        // The next unit's query rows, head weights, positions and RoPE rows
        // into L2 while this pass streams: its query build, which every role
        // waits for, then reads L2 instead of DRAM.  (Hints only: they read
        // nothing the kernel depends on.)
        __syncwarp();
        const int un = u + (int)gridDim.x;
        if (un < n_units && !M->abort) {
          const long long t0 = (long long)(un / units_per_group) * RPG;
          const int nr = (int)min((long long)RPG, (long long)a.n_rows - t0);
          if (nr > 0) {
            const uint8_t *qb = static_cast<const uint8_t *>(a.q_idx) + t0 * a.n_heads * kIdxDim * 2;
            const int qbytes = nr * a.n_heads * kIdxDim * 2;
            for (int off = lane * 128; off < qbytes; off += 32 * 128) prefetch_l2(qb + off);
            const uint8_t *wb = reinterpret_cast<const uint8_t *>(a.weights + t0 * a.n_heads);
            for (int off = lane * 128; off < nr * a.n_heads * 4; off += 32 * 128)
              prefetch_l2(wb + off);
            if (lane < nr) {
              const int p = a.row_pos[t0 + lane];
              if (rope && p >= 0 && p < a.rope_cap) {
                prefetch_l2(a.rope_cos + (long long)p * kRopeHalf);
                prefetch_l2(a.rope_sin + (long long)p * kRopeHalf);
              }
            }
          }
        }
      } else if (warp >= W_CONV0 && warp < W_PROD) {
        // ---------------- converters: int8 page -> fp16 A tile
        const int ct = tid - W_CONV0 * 32;
        for (int k = 0; k < nt; ++k) {
          const uint32_t itk = it + k;
          const int s = itk % C::NS, j = itk % C::NA, sc = itk % C::NSC;
          if (!tc::mbar_wait(&M->st_full[s], (itk / C::NS) & 1) ||
              !tc::mbar_wait(&M->a_free[j], ((itk / C::NA) & 1) ^ 1)) {
            set_abort(M, a.status_dev);
            break;
          }
          const int ok = M->st_ok[s];
          if constexpr (C::ATMEM) {
            // thread = one key row (TMEM lane) x one half of its 128 dims
            const int wq = (warp - W_CONV0) & 3, half = (warp - W_CONV0) >> 2;
            const int r = wq * 32 + lane;
            if (ok && fp4) {
              // FP4 keys (64 code bytes and 4 E8M0 bytes per row): this half's
              // 32 code bytes, each group scaled by 2^(E_g - R) into FP16
              const uint8_t *src = St + s * C::PAGE + r * 64 + half * 32;
              const uint32_t sb4 =
                  reinterpret_cast<const uint32_t *>(StSc)[s * kBlock + r];
              const int R = lowbit::e8m0_row_shift(sb4);
              uint32_t packed[32];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint2 w = *reinterpret_cast<const uint2 *>(src + c * 8);
                const __half2 sc2 = lowbit::e8m0_group_h2(sb4, half * 2 + (c >> 1), R);
                const uint4 lo = lowbit::e2m1x8_to_f16x8(w.x, sc2);
                const uint4 hi = lowbit::e2m1x8_to_f16x8(w.y, sc2);
                packed[8 * c + 0] = lo.x;
                packed[8 * c + 1] = lo.y;
                packed[8 * c + 2] = lo.z;
                packed[8 * c + 3] = lo.w;
                packed[8 * c + 4] = hi.x;
                packed[8 * c + 5] = hi.y;
                packed[8 * c + 6] = hi.z;
                packed[8 * c + 7] = hi.w;
              }
              tc::tmem_st32u(tmem + ((uint32_t)(wq * 32) << 16) + C::A_COL + j * 64 + half * 32,
                             packed);
              tc::tmem_wait_st();
              if (half == 0) Sc[sc * kBlock + r] = lowbit::pow2f(R);
            } else if (ok && fp8) {
              // FP8 keys: this half's four swizzled 16-byte chunks of E4M3
              // codes, each group scaled by 2^(E_g - R) into FP16
              const uint8_t *src = St + s * C::PAGE + r * 128;
              const uint32_t sb4 =
                  reinterpret_cast<const uint32_t *>(StSc)[s * kBlock + r];
              const int R = lowbit::e8m0_row_shift(sb4);
              uint32_t packed[32];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int cc = half * 4 + c;
                const uint4 raw = *reinterpret_cast<const uint4 *>(src + ((cc ^ (r & 7)) << 4));
                const __half2 sc2 = lowbit::e8m0_group_h2(sb4, cc >> 1, R);
                const uint4 lo = lowbit::e4m3x8_to_f16x8(make_uint2(raw.x, raw.y), sc2);
                const uint4 hi = lowbit::e4m3x8_to_f16x8(make_uint2(raw.z, raw.w), sc2);
                packed[8 * c + 0] = lo.x;
                packed[8 * c + 1] = lo.y;
                packed[8 * c + 2] = lo.z;
                packed[8 * c + 3] = lo.w;
                packed[8 * c + 4] = hi.x;
                packed[8 * c + 5] = hi.y;
                packed[8 * c + 6] = hi.z;
                packed[8 * c + 7] = hi.w;
              }
              tc::tmem_st32u(tmem + ((uint32_t)(wq * 32) << 16) + C::A_COL + j * 64 + half * 32,
                             packed);
              tc::tmem_wait_st();
              if (half == 0) Sc[sc * kBlock + r] = lowbit::pow2f(R);
            } else if (ok) {
              const uint8_t *src = St + s * C::PAGE + r * 128;
              uint32_t packed[32];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int cc = half * 4 + c;
                const uint4 raw = *reinterpret_cast<const uint4 *>(src + ((cc ^ (r & 7)) << 4));
                const uint4 lo = i8x8_to_f16x8(make_uint2(raw.x, raw.y));
                const uint4 hi = i8x8_to_f16x8(make_uint2(raw.z, raw.w));
                packed[8 * c + 0] = lo.x;
                packed[8 * c + 1] = lo.y;
                packed[8 * c + 2] = lo.z;
                packed[8 * c + 3] = lo.w;
                packed[8 * c + 4] = hi.x;
                packed[8 * c + 5] = hi.y;
                packed[8 * c + 6] = hi.z;
                packed[8 * c + 7] = hi.w;
              }
              tc::tmem_st32u(tmem + ((uint32_t)(wq * 32) << 16) + C::A_COL + j * 64 + half * 32,
                             packed);
              tc::tmem_wait_st();
              if (half == 0) Sc[sc * kBlock + r] = StSc[s * kBlock + r];
            }
            if (ct == 0) M->t_ok[sc] = ok;
            tc::tc_fence_before();
          } else {
          if (ok && fp4) {
            // FP4 keys: unit = (row, 8 dims): one code word and the row's
            // four E8M0 bytes
            const uint8_t *src = St + s * C::PAGE;
            const uint32_t *sbw = reinterpret_cast<const uint32_t *>(StSc) + s * kBlock;
            uint8_t *dst = As + j * C::A_BUF;
            uint32_t raw[8], sb4[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              raw[q] = *reinterpret_cast<const uint32_t *>(src + (unit >> 4) * 64 + (unit & 15) * 4);
              sb4[q] = sbw[unit >> 4];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              const int r = unit >> 4, jc = unit & 15;
              const int kc = jc >> 3, jj = jc & 7;
              const int R = lowbit::e8m0_row_shift(sb4[q]);
              *reinterpret_cast<uint4 *>(dst + kc * C::A_CHUNK + r * 128 + ((jj ^ (r & 7)) << 4)) =
                  lowbit::e2m1x8_to_f16x8(raw[q], lowbit::e8m0_group_h2(sb4[q], jc >> 2, R));
            }
            if (ct < kBlock) Sc[sc * kBlock + ct] = lowbit::pow2f(lowbit::e8m0_row_shift(sbw[ct]));
          } else if (ok && fp8) {
            // FP8 keys: unit = (row, 8 dims): two code words and the row's
            // four E8M0 bytes
            const uint8_t *src = St + s * C::PAGE;
            const uint32_t *sbw = reinterpret_cast<const uint32_t *>(StSc) + s * kBlock;
            uint8_t *dst = As + j * C::A_BUF;
            uint2 raw[8];
            uint32_t sb4[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              raw[q] = *reinterpret_cast<const uint2 *>(src + (unit >> 4) * 128 + (unit & 15) * 8);
              sb4[q] = sbw[unit >> 4];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              const int r = unit >> 4, jc = unit & 15;
              const int kc = jc >> 3, jj = jc & 7;
              const int R = lowbit::e8m0_row_shift(sb4[q]);
              *reinterpret_cast<uint4 *>(dst + kc * C::A_CHUNK + r * 128 + ((jj ^ (r & 7)) << 4)) =
                  lowbit::e4m3x8_to_f16x8(raw[q], lowbit::e8m0_group_h2(sb4[q], jc >> 2, R));
            }
            if (ct < kBlock) Sc[sc * kBlock + ct] = lowbit::pow2f(lowbit::e8m0_row_shift(sbw[ct]));
          } else if (ok) {
            const uint8_t *src = St + s * C::PAGE;
            uint8_t *dst = As + j * C::A_BUF;
            uint2 raw[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              raw[q] = *reinterpret_cast<const uint2 *>(src + (unit >> 4) * 128 + (unit & 15) * 8);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = q * IT_CONV + ct;
              const int r = unit >> 4, jc = unit & 15;
              const int kc = jc >> 3, jj = jc & 7;
              *reinterpret_cast<uint4 *>(dst + kc * C::A_CHUNK + r * 128 + ((jj ^ (r & 7)) << 4)) =
                  i8x8_to_f16x8(raw[q]);
            }
            if (ct < kBlock) Sc[sc * kBlock + ct] = StSc[s * kBlock + ct];
          }
          if (ct == 0) M->t_ok[sc] = ok;
          tc::fence_async_shared();
          }
          tc::mbar_arrive(&M->a_full[j]);
          tc::mbar_arrive(&M->st_empty[s]);
        }
      } else if (warp == W_MMA) {
        // ---------------- MMA issuer: the whole warp runs the loop with
        // warp-uniform operands; one elected lane issues
        constexpr uint32_t idesc = tc::idesc_f16_f32(128, C::N);
        const uint32_t a_base = tc::smem_u32(As), b_base = tc::smem_u32(Bs);
        uint64_t bd[12];
#pragma unroll
        for (int kc = 0; kc < 3; ++kc)
#pragma unroll
          for (int s16 = 0; s16 < 4; ++s16)
            bd[kc * 4 + s16] = tc::desc_sw128(b_base + kc * C::B_CHUNK + s16 * 32);
        for (int k = 0; k < nt; ++k) {
          const uint32_t itk = it + k;
          const int j = itk % C::NA, q4 = itk % C::NT;
          if (!tc::mbar_wait(&M->a_full[j], (itk / C::NA) & 1) ||
              !tc::mbar_wait(&M->acc_empty[q4], ((itk / C::NT) & 1) ^ 1)) {
            set_abort(M, a.status_dev);
            break;
          }
          tc::tc_fence_after();
          const uint32_t d = tmem + C::ACC_COL + q4 * C::N;
          if constexpr (C::ATMEM) {
            const uint32_t a_t = tmem + C::A_COL + j * 64;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              tc::mma_f16_ta_elect(d, a_t + (i < 4 ? 0 : 32) + (i & 3) * 8, bd[i], idesc, i != 0);
            if (n_kchunks == 3) {
#pragma unroll
              for (int i = 8; i < 12; ++i)
                tc::mma_f16_ta_elect(d, a_t + 32 + (i & 3) * 8, bd[i], idesc, 1u);
            }
          } else {
            const uint32_t a_off = a_base + j * C::A_BUF;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              tc::mma_ss_elect(d, tc::desc_sw128(a_off + (i < 4 ? 0 : C::A_CHUNK) + (i & 3) * 32),
                               bd[i], idesc, i != 0);
            if (n_kchunks == 3) {
#pragma unroll
              for (int i = 8; i < 12; ++i)
                tc::mma_ss_elect(d, tc::desc_sw128(a_off + C::A_CHUNK + (i & 3) * 32), bd[i],
                                 idesc, 1u);
            }
          }
          tc::mma_commit_elect(&M->a_free[j]);
          tc::mma_commit_elect(&M->acc_full[q4]);
          __syncwarp();
        }
      } else if (warp < W_CONV0) {
        // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 and
        // the rows rr with rr % 2 == w / 4 (a row's score sums its slots)
        const int r = (warp & 3) * 32 + lane;  // key within the tile
        const int i0 = warp >> 2;
        const uint64_t keep = tc::l2_evict_last();
        for (int k = 0; k < nt; ++k) {
          const uint32_t itk = it + k;
          const int q4 = itk % C::NT, sc = itk % C::NSC;
          if (!tc::mbar_wait(&M->acc_full[q4], (itk / C::NT) & 1)) {
            set_abort(M, a.status_dev);
            break;
          }
          tc::tc_fence_after();
          const bool ok = (M->t_ok[sc] >> (r >> 3)) & 1;
          const float scale = Sc[sc * kBlock + r];
          const int c = (tb + k) * kBlock + r;
          for (int rr = i0; rr < RR; rr += 2) {
            if (!M->row_on[rr]) continue;
            float sum = 0.f;
#pragma unroll 1
            for (int sl = 0; sl < HS; ++sl) {
              const int i = sl * RR + rr;
              float v[64];
              tc::tmem_ld64(tmem + ((uint32_t)((warp & 3) * 32) << 16) + C::ACC_COL + q4 * C::N +
                                i * kHeads,
                            v);
              const float4 *w4 = reinterpret_cast<const float4 *>(Ws + i * kHeads);
              float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
              for (int h4 = 0; h4 < 16; ++h4) {
                const float4 w = w4[h4];
                float x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  x[q] = a.relu ? fmaxf(v[4 * h4 + q], 0.f) : v[4 * h4 + q];
                acc0 = tc::ffma2(make_float2(w.x, w.y), make_float2(x[0], x[1]), acc0);
                acc1 = tc::ffma2(make_float2(w.z, w.w), make_float2(x[2], x[3]), acc1);
              }
              sum += (acc0.x + acc0.y) + (acc1.x + acc1.y);
            }
            const int i = rr;
            const bool vis = c < M->row_V[i];
            const float val = ok ? scale * sum : -INFINITY;
            // scores stay in L2 for the top-k that reads them next, instead of
            // being written back while the key stream still flows
            if (vis) tc::st_global_hint(scores + (long long)M->row_t[i] * cols + c, val, keep);
            if (sel.blk) {
              // level one: the maximum over each block's visible entries (a
              // block is cb consecutive lanes)
              float m = vis ? val : -INFINITY;
              for (int o = 1; o < cb; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
              if (vis && (lane & (cb - 1)) == 0)
                sel.blk[(long long)M->row_t[i] * sel.blk_cols + (c >> sel.cb_shift)] = m;
            }
          }
          tc::tc_fence_before();
          tc::mbar_arrive(&M->acc_empty[q4]);
        }
      }
      it += nt;
    }
  }

  // drain: wait (bounded) for copies still in flight, then free TMEM
  if (warp == W_PROD && lane == 0 && M->abort) {
    for (int k = 0; k < C::NS && k < (int)it; ++k) {
      const uint32_t itk = it - 1 - k;
      tc::mbar_wait(&M->st_full[itk % C::NS], (itk / C::NS) & 1, 100000000ull);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == W_MMA) tc::tmem_dealloc(tmem, C::TMEM_COLS);
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Tensor map of the INT8 (or FP8) key pool as a 3D [pages, 128 rows, 128
// bytes] array with the pool's page and row strides, `box_rows` rows (a page,
// or one candidate block) per box; 128-byte swizzle when the converters read
// rows of a swizzled tile (A in TMEM), none otherwise (a linear tile).
bool encode_keys_map(const csa_index_args &a, int box_rows, bool swizzle, CUtensorMap *map) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[3] = {(cuuint64_t)kIdxDim, (cuuint64_t)kBlock, (cuuint64_t)a.n_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)a.key_row_stride, (cuuint64_t)a.key_page_stride};
  const cuuint32_t box[3] = {(cuuint32_t)kIdxDim, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<int8_t *>(a.idx_pool), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G, int HS>
cudaError_t launch_tc(const csa_index_args &a, float *scores, int cols, uint32_t *zero_ctr,
                      cudaStream_t s, const ScoreSel &sel) {
  using C = IdxTc<G>;
  const bool reidx = sel.cand_in != nullptr;
  CUtensorMap keys_map;
  memset(&keys_map, 0, sizeof(keys_map));
  if (a.key_fmt != CSA_FMT_FP4_E8M0 &&
      !encode_keys_map(a, reidx ? 1 << sel.cb_shift : kBlock, C::ATMEM, &keys_map))
    return cudaErrorInvalidValue;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel<G, HS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const int sms = sm_count();
  constexpr int RR = G / HS;
  const int n_groups = reidx ? a.n_rows : (a.n_rows + RR - 1) / RR;
  // tiles of one row: its pages, or (reindex) its candidate entries / 128
  const int max_tiles =
      reidx ? ((sel.n_cand << sel.cb_shift) + kBlock - 1) / kBlock : a.max_blocks;
  int upg = (sms + n_groups - 1) / n_groups;
  upg = max(1, min(upg, max_tiles));
  const int chunk = (max_tiles + upg - 1) / upg;
  upg = (max_tiles + chunk - 1) / chunk;
  const long long n_units = (long long)n_groups * upg;
  const int grid = (int)(n_units < sms ? n_units : sms);
  launch_begin(CSA_K_INDEX_SCORE, s);
  const cudaError_t e = launch_kernel(index_score_tc_kernel<G, HS>, dim3(grid), dim3(IT_THREADS),
                                      (size_t)C::SMEM, s, 0, false, a, scores, cols, n_groups,
                                      chunk, upg, zero_ctr, keys_map, sel);
  launch_end(CSA_K_INDEX_SCORE, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_scores(const csa_index_args &a, float *scores, int score_cols,
                                uint32_t *zero_ctr, cudaStream_t s, const ScoreSel &sel) {
  if (a.n_rows <= 0) return cudaSuccess;
  // the two-row tiling (keys through TMEM) is the default: measured on the
  // prefill workloads it also beats the four-row one (8,192 rows: 427 against
  // 442 us a call), whose per-pass query build weighs more
  const bool wide = a.mode == CSA_MODE_PREFILL;
  if (a.n_heads > kHeads)  // two 64-head slots per row
    return wide ? launch_tc<4, 2>(a, scores, score_cols, zero_ctr, s, sel)
                : launch_tc<2, 2>(a, scores, score_cols, zero_ctr, s, sel);
  return wide ? launch_tc<4, 1>(a, scores, score_cols, zero_ctr, s, sel)
              : launch_tc<2, 1>(a, scores, score_cols, zero_ctr, s, sel);
}

}  // namespace csa
