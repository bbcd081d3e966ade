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
//   warp 8      bulk-copies each INT8 page (16 KB) and its scales into a ring,
//   warps 4..7  convert INT8 -> BF16 (exact: |v| <= 127 fits BF16's 8-bit
//               significand) into the 128-byte-swizzled K-major layout,
//   warp 9      issues tcgen05.mma (A = keys, B = queries) into a double-
//               buffered TMEM accumulator,
//   warps 0..3  read TMEM and apply ReLU, the head weights and the key scale.
// Queries rotated by RoPE in FP32 are split into BF16 hi + lo parts so that the
// BF16 tensor-core product keeps FP32-level accuracy (K = 64 + 64 + 64).
#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int IT_THREADS = 320;  // 10 warps

template <int G>
struct IdxTc {
  static constexpr int N = G * kHeads;            // MMA N
  static constexpr int NS = G == 2 ? 4 : 3;       // staging ring depth
  static constexpr int B_CHUNK = N * 128;         // bytes of one 64-wide K chunk of B
  static constexpr int A_CHUNK = kBlock * 128;    // 16 KB
  static constexpr int A_BUF = 2 * A_CHUNK;       // 128 keys x 128 dims bf16
  static constexpr int PAGE = kBlock * kIdxDim;   // 16 KB of int8 keys
  static constexpr int OFF_B = 0;
  static constexpr int OFF_A = OFF_B + 3 * B_CHUNK;
  static constexpr int OFF_ST = OFF_A + 2 * A_BUF;
  static constexpr int OFF_STSC = OFF_ST + NS * PAGE;
  static constexpr int OFF_SC = OFF_STSC + NS * kBlock * 4;
  static constexpr int OFF_W = OFF_SC + 2 * kBlock * 4;
  static constexpr int OFF_MISC = OFF_W + G * kHeads * 4;
  static constexpr int SMEM = OFF_MISC + 512 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 2 * N;
};

struct IdxMisc {
  uint64_t st_full[4];
  uint64_t st_empty[4];
  uint64_t a_full[2];
  uint64_t mma_done[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int st_ok[4];
  int a_ok[2];
  volatile int abort;
  int row_t[4];
  int row_V[4];
  int row_on[4];
};

__device__ __forceinline__ void set_abort(IdxMisc *m, uint32_t *status) {
  m->abort = 1;
  flag(status, CSA_DEV_TIMEOUT);
}

// 8 int8 -> 8 bf16, exactly: (v ^ 0x80) placed in the mantissa of 2^23 gives
// 2^23 + 128 + v as an FP32 value.
__device__ __forceinline__ uint4 i8x8_to_bf16x8(uint2 raw) {
  const uint32_t w[2] = {raw.x ^ 0x80808080u, raw.y ^ 0x80808080u};
  uint32_t out[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float f[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      f[k] = __uint_as_float(__byte_perm(w[h], 0x4B000000u, 0x7440u | k)) - 8388736.0f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(f[0], f[1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(f[2], f[3]);
    out[2 * h] = *reinterpret_cast<uint32_t *>(&lo);
    out[2 * h + 1] = *reinterpret_cast<uint32_t *>(&hi);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int G>
__global__ void __launch_bounds__(IT_THREADS, 1)
    index_score_tc_kernel(csa_index_args a, float *__restrict__ scores, int cols, int n_groups,
                          int chunk_tiles, int units_per_group, uint32_t *zero_ctr) {
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
  IdxMisc *M = reinterpret_cast<IdxMisc *>(sm + C::OFF_MISC);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (zero_ctr && blockIdx.x == 0)
    for (int i = tid; i < a.n_rows; i += IT_THREADS) zero_ctr[i] = 0u;
  const bool rope = a.rope_cos != nullptr;
  const int n_kchunks = rope ? 3 : 2;
  const int n_cap = a.max_blocks * kBlock;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      tc::mbar_init(&M->st_full[s], 1);
      tc::mbar_init(&M->st_empty[s], 128);
    }
    for (int j = 0; j < 2; ++j) {
      tc::mbar_init(&M->a_full[j], 128);
      tc::mbar_init(&M->mma_done[j], 1);
      tc::mbar_init(&M->tmem_empty[j], 128);
    }
    M->abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 9) tc::tmem_alloc(&M->tmem_base, C::TMEM_COLS);
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
      const int t = g * G + i;
      rb[i] = t < a.n_rows ? a.row_req[t] : -1;
      if (rb[i] >= a.n_req) {
        if (chunk == 0 && tid == 0) flag(a.status_dev, CSA_DEV_BAD_POS);
        rb[i] = -1;
      }
    }
    for (int pi = 0; pi < G; ++pi) {
      const int b = rb[pi];
      bool first = b >= 0;
      for (int j = 0; j < pi; ++j) first = first && rb[j] != b;
      if (!first) continue;

      // ---------------- pass setup (all threads)
      __syncthreads();
      if (M->abort) break;
      int vmax = 0;
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int t = g * G + i;
        int V = 0;
        const bool on = rb[i] == b;
        if (on) V = min(visible_count(a.row_pos[t], a.ratio, a.n_cmp[b]), n_cap);
        vmax = max(vmax, V);
        if (tid == 0) {
          M->row_t[i] = t;
          M->row_V[i] = V;
          M->row_on[i] = on;
        }
      }
      const int tiles_total = (vmax + kBlock - 1) / kBlock;
      const int tb = chunk * chunk_tiles;
      const int te = min(tiles_total, tb + chunk_tiles);
      if (tb >= te) continue;  // uniform across the CTA
      // queries (B operand): every 16-byte piece in flight at once (cp.async),
      // then the rotated half is split in place into BF16 hi (chunk 1) and lo
      // (chunk 2) by the thread that copied it
      for (int e = tid; e < 16 * C::N; e += IT_THREADS) {
        const int n = e / 16, part = (e / 8) % 2, jj = e % 8;
        const int i = n / kHeads, h = n % kHeads;
        const int t = g * G + i;
        uint8_t *d = Bs + part * C::B_CHUNK + n * 128 + ((jj ^ (n & 7)) << 4);
        if (rb[i] == b)
          tc::cp_async16(d, static_cast<const uint16_t *>(a.q_idx) +
                                ((long long)t * kHeads + h) * kIdxDim + part * 64 + jj * 8);
        else
          *reinterpret_cast<uint4 *>(d) = make_uint4(0, 0, 0, 0);
        if (part == 1)
          *reinterpret_cast<uint4 *>(d + C::B_CHUNK) = make_uint4(0, 0, 0, 0);
      }
      tc::cp_async_wait_all();
      if (rope) {
        for (int e = tid; e < 16 * C::N; e += IT_THREADS) {
          const int n = e / 16, part = (e / 8) % 2, jj = e % 8;
          const int i = n / kHeads, h = n % kHeads;
          const int t = g * G + i;
          if (part != 1 || rb[i] != b) continue;
          const int p = a.row_pos[t];
          if (p < 0) continue;
          if (p >= a.rope_cap) {
            if (h == 0 && jj == 0) flag(a.status_dev, CSA_DEV_POS_GE_CAP);
            continue;
          }
          uint8_t *d = Bs + C::B_CHUNK + n * 128 + ((jj ^ (n & 7)) << 4);
          const uint4 x = *reinterpret_cast<const uint4 *>(d);
          const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float x0 = __uint_as_float(xw[q] << 16);
            const float x1 = __uint_as_float(xw[q] & 0xFFFF0000u);
            const int pair = jj * 4 + q;
            const float c = a.rope_cos[(long long)p * kRopeHalf + pair];
            const float s = a.rope_sin[(long long)p * kRopeHalf + pair];
            const float y0 = x0 * c - x1 * s;
            const float y1 = x0 * s + x1 * c;
            const __nv_bfloat162 hb = __floats2bfloat162_rn(y0, y1);
            hw[q] = *reinterpret_cast<const uint32_t *>(&hb);
            lw[q] = pack_bf16(y0 - __low2float(hb), y1 - __high2float(hb));
          }
          *reinterpret_cast<uint4 *>(d) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(d + C::B_CHUNK) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      for (int e = tid; e < G * kHeads; e += IT_THREADS) {
        const int i = e / kHeads, t = g * G + i;
        Ws[e] = rb[i] == b ? a.weights[(long long)t * kHeads + (e % kHeads)] : 0.f;
      }
      tc::fence_async_shared();
      __syncthreads();

      const int nt = te - tb;
      if (warp == 8) {
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
            M->st_ok[s] = ok;
            if (ok) {
              tc::mbar_arrive_expect_tx(&M->st_full[s], C::PAGE + kBlock * 4);
              tc::bulk_g2s(St + s * C::PAGE, a.idx_pool + (long long)phys * C::PAGE, C::PAGE,
                           &M->st_full[s]);
              tc::bulk_g2s(StSc + s * kBlock, a.idx_scale_pool + (long long)phys * kBlock,
                           kBlock * 4, &M->st_full[s]);
            } else {
              flag(a.status_dev, CSA_DEV_BAD_BLOCK);
              tc::mbar_arrive(&M->st_full[s]);
            }
          }
        }
      } else if (warp >= 4 && warp < 8) {
        // ---------------- converters: int8 page -> bf16 swizzled A tile
        const int ct = tid - 128;
        for (int k = 0; k < nt; ++k) {
          const uint32_t itk = it + k;
          const int s = itk % C::NS, j = itk % 2;
          if (!tc::mbar_wait(&M->st_full[s], (itk / C::NS) & 1) ||
              !tc::mbar_wait(&M->tmem_empty[j], ((itk / 2) & 1) ^ 1)) {
            set_abort(M, a.status_dev);
            break;
          }
          const int ok = M->st_ok[s];
          if (ok) {
            const uint8_t *src = St + s * C::PAGE;
            uint8_t *dst = As + j * C::A_BUF;
#pragma unroll 4
            for (int q = 0; q < 16; ++q) {
              const int unit = q * 128 + ct;
              const int r = unit / 16, jc = unit % 16;
              const int kc = jc / 8, jj = jc % 8;
              const uint2 raw = *reinterpret_cast<const uint2 *>(src + r * 128 + jc * 8);
              *reinterpret_cast<uint4 *>(dst + kc * C::A_CHUNK + r * 128 +
                                         ((jj ^ (r & 7)) << 4)) = i8x8_to_bf16x8(raw);
            }
            Sc[j * kBlock + ct] = StSc[s * kBlock + ct];
          }
          if (ct == 0) M->a_ok[j] = ok;
          tc::fence_async_shared();
          tc::mbar_arrive(&M->a_full[j]);
          tc::mbar_arrive(&M->st_empty[s]);
        }
      } else if (warp == 9) {
        // ---------------- MMA issuer
        if (lane == 0) {
          constexpr uint32_t idesc = tc::idesc_bf16_f32(128, C::N);
          const uint32_t a_base = tc::smem_u32(As), b_base = tc::smem_u32(Bs);
          for (int k = 0; k < nt; ++k) {
            const uint32_t itk = it + k;
            const int j = itk % 2;
            if (!tc::mbar_wait(&M->a_full[j], (itk / 2) & 1)) {
              set_abort(M, a.status_dev);
              break;
            }
            tc::tc_fence_after();
            const uint32_t d = tmem + j * C::N;
            for (int kc = 0; kc < n_kchunks; ++kc) {
              const uint32_t a_off = a_base + j * C::A_BUF + (kc == 0 ? 0 : C::A_CHUNK);
              const uint32_t b_off = b_base + kc * C::B_CHUNK;
#pragma unroll
              for (int s16 = 0; s16 < 4; ++s16)
                tc::mma_bf16(d, tc::desc_sw128(a_off + s16 * 32), tc::desc_sw128(b_off + s16 * 32),
                             idesc, (kc | s16) != 0);
            }
            tc::mma_commit(&M->mma_done[j]);
          }
        }
      } else {
        // ---------------- epilogue: warps 0..3 own TMEM lanes 32*warp .. +31
        const int r = tid;  // key within the tile
        for (int k = 0; k < nt; ++k) {
          const uint32_t itk = it + k;
          const int j = itk % 2;
          if (!tc::mbar_wait(&M->mma_done[j], (itk / 2) & 1)) {
            set_abort(M, a.status_dev);
            break;
          }
          tc::tc_fence_after();
          const int ok = M->a_ok[j];
          const float scale = Sc[j * kBlock + r];
          const int c = (tb + k) * kBlock + r;
#pragma unroll
          for (int i = 0; i < G; ++i) {
            if (!M->row_on[i]) continue;
            float acc = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float v[32];
              tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + j * C::N + i * kHeads +
                                half * 32,
                            v);
              const float *w = Ws + i * kHeads + half * 32;
              if (a.relu) {
#pragma unroll
                for (int h = 0; h < 32; ++h) acc = fmaf(w[h], fmaxf(v[h], 0.f), acc);
              } else {
#pragma unroll
                for (int h = 0; h < 32; ++h) acc = fmaf(w[h], v[h], acc);
              }
            }
            if (c < M->row_V[i])
              scores[(long long)M->row_t[i] * cols + c] = ok ? scale * acc : -INFINITY;
          }
          tc::tc_fence_before();
          tc::mbar_arrive(&M->tmem_empty[j]);
        }
      }
      it += nt;
    }
  }

  // drain: wait (bounded) for copies still in flight, then free TMEM
  if (warp == 8 && lane == 0 && M->abort) {
    for (int k = 0; k < C::NS && k < (int)it; ++k) {
      const uint32_t itk = it - 1 - k;
      tc::mbar_wait(&M->st_full[itk % C::NS], (itk / C::NS) & 1, 100000000ull);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 9) tc::tmem_dealloc(tmem, C::TMEM_COLS);
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

template <int G>
cudaError_t launch_tc(const csa_index_args &a, float *scores, int cols, uint32_t *zero_ctr,
                      cudaStream_t s) {
  using C = IdxTc<G>;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const int sms = sm_count();
  const int n_groups = (a.n_rows + G - 1) / G;
  const int max_tiles = a.max_blocks;
  int upg = (sms + n_groups - 1) / n_groups;
  upg = max(1, min(upg, max_tiles));
  const int chunk = (max_tiles + upg - 1) / upg;
  upg = (max_tiles + chunk - 1) / chunk;
  const long long n_units = (long long)n_groups * upg;
  const int grid = (int)(n_units < sms ? n_units : sms);
  launch_begin(CSA_K_INDEX_SCORE, s);
  index_score_tc_kernel<G><<<grid, IT_THREADS, C::SMEM, s>>>(a, scores, cols, n_groups, chunk,
                                                             upg, zero_ctr);
  launch_end(CSA_K_INDEX_SCORE, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_scores(const csa_index_args &a, float *scores, int score_cols,
                                uint32_t *zero_ctr, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  const bool wide = a.mode == CSA_MODE_PREFILL || (a.mode == CSA_MODE_AUTO && a.n_rows > 64);
  return wide ? launch_tc<4>(a, scores, score_cols, zero_ctr, s)
              : launch_tc<2>(a, scores, score_cols, zero_ctr, s);
}

}  // namespace csa
