// Deterministic top-k over the lightning-indexer scores: the k entries with
// the highest score (equal scores: the smaller position first), emitted as
// logical positions in ascending order with trailing -1 padding ("DeepSeek
// V4.1 Flash", "Compressor state ownership": Top-K eligibility, uniqueness,
// logical-position ordering and trailing -1; "Hyper-Parallel ... DeepSeek V4
// CP", "10.3 Causal mask" for the visible range).
//
// Scores become order-preserving 32-bit keys, held in registers (each thread
// owns a contiguous run of positions).  A three-digit radix select (11, 11
// and 10 key bits) finds the k-th largest key T and how many keys equal to T
// are taken; equal keys are taken in ascending position.  Rows up to 16384
// entries are selected by one CTA.  Longer rows are split into S slices, the
// CTAs of a cooperative launch: each slice adds its digit histogram into the
// row's histogram in global memory and the slices meet at a bounded barrier
// per digit.  At the last digit every slice also publishes the suffix sums of
// its own histogram, so that each slice can work out, without a further
// barrier, how many entries the slices before it emit; it then writes its
// winners in ascending position order at that offset.
#include <algorithm>

#include "csa_internal.cuh"
#include "tc.cuh"

namespace csa {
namespace {

// Order-preserving 32-bit key of a float score: larger score -> larger key.
// +0 and -0 share a key; NaN maps to the smallest key.
__device__ __forceinline__ uint32_t order_key(float s) {
  if (s != s) return 0u;
  if (s == 0.f) s = 0.f;
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; `warp_sums` holds 32 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const int base = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[nw - 1];
  return base + x - v;
}

// ---------------------------------------------------------------- radix select

constexpr int TK_SHORT_KPT = 16;  // one CTA per row: 16 entries per thread ...
constexpr int TK_SHORT_KPT2 = 32; // ... or 32 (512 threads: rows up to 16384 entries)
constexpr int TK_LONG_THREADS = 512;
constexpr int TK_LONG_KPT = 16;   // entries per thread of a long-row slice
constexpr int TK_PRIV = 4;        // first-digit histograms of a long-row slice, 4 warps each
constexpr int TK_LONG_PER_SM = 2; // long-row slices per SM (the grid is resident at once)
constexpr int TK_B1 = 2048, TK_B2 = 2048, TK_B3 = 1024;  // 11 + 11 + 10 key bits
constexpr int TK_CTL_HDR = 32;  // barrier counter, alone in its 128-byte line
static_assert(TK_CTL_HDR + TK_B1 + TK_B2 + TK_B3 == kTopkCtlWords, "row control block");
constexpr int TK_REC_WORDS = 1056;  // per slice: suffix counts [0, 1024] and the count above
constexpr int TK_REC_GT = 1025;     // the 22-bit prefix, at word 1025

// Dynamic shared memory of a long-row CTA: TK_PRIV first-digit histograms,
// each shared by a quarter of the warps (the first digit is the most crowded:
// spread the warps' counters), and the CTA's histogram -- 40 KB, so that two
// slices share an SM.
template <int NT>
constexpr int topk_smem_bytes() {
  return (TK_PRIV + 1) * TK_B1 * 4;
}

// Barrier of the S CTAs that share a row: the counter only grows, barrier j
// waits for j*S arrivals.  Waits at most `limit_ns` (0: 1 s; negative: not
// at all -- a CTA that is not the last to arrive gives up at once); returns
// false (and flags CSA_DEV_TIMEOUT) when it gives up.
__device__ bool row_barrier(uint32_t *ctr, uint32_t target, uint32_t *status, int *s_ok,
                            long long limit_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t arrived = atomicAdd(ctr, 1u) + 1u;
    const uint64_t lim = limit_ns == 0 ? 1000000000ull : (uint64_t)max(limit_ns, 0ll);
    int ok = 1;
    if (arrived < target) {
      const uint64_t t0 = tc::global_ns();
      while (*reinterpret_cast<volatile uint32_t *>(ctr) < target) {
        if (limit_ns < 0 || tc::global_ns() - t0 > lim) {
          ok = 0;
          flag(status, CSA_DEV_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Warp 0: the digit d at which the count of keys with digit >= d (scanning
// from the top) first reaches `remaining`, and the count strictly above d.
// Lane l sums nb/32 consecutive bins from the top (read in a lane-rotated
// order, so that eight lanes of a quarter-warp hit distinct bank groups),
// a warp scan finds the crossing lane, and a second scan over that lane's
// bins (two per lane) finds the digit.
__device__ __forceinline__ void warp_find_digit(const uint32_t *hist, int nb, int remaining,
                                                int *s_digit, int *s_above) {
  const int lane = threadIdx.x & 31;
  const int per = nb >> 5;  // 64 or 32 bins per lane
  const int lo = nb - (lane + 1) * per;
  const uint4 *v = reinterpret_cast<const uint4 *>(hist + lo);
  const int nv4 = per >> 2;
  int local = 0;
  for (int j = 0; j < nv4; ++j) {
    const uint4 x = v[(j + lane) & (nv4 - 1)];
    local += (int)(x.x + x.y + x.z + x.w);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, incl - local < remaining && incl >= remaining);
  if (!hit) {
    if (lane == 0) {
      *s_digit = 0;
      *s_above = 0;
    }
    return;
  }
  const int L = __ffs(hit) - 1;
  const int before = __shfl_sync(0xffffffffu, incl - local, L);
  // lane m takes bins top - 2m and top - 2m - 1 of lane L's range
  const int top = nb - 1 - L * per;
  const int h0 = 2 * lane < per ? (int)hist[top - 2 * lane] : 0;
  const int h1 = 2 * lane + 1 < per ? (int)hist[top - 2 * lane - 1] : 0;
  int incl2 = h0 + h1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) incl2 += y;
  }
  const int b4 = before + incl2 - (h0 + h1);  // count above this lane's pair
  const unsigned hit2 = __ballot_sync(0xffffffffu, b4 < remaining && b4 + h0 + h1 >= remaining);
  if (lane == __ffs(hit2) - 1) {
    if (b4 + h0 >= remaining) {
      *s_digit = top - 2 * lane;
      *s_above = b4;
    } else {
      *s_digit = top - 2 * lane - 1;
      *s_above = b4 + h0;
    }
  }
}

// Score back from its order key (-0 comes back as +0).
__device__ __forceinline__ float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One CTA of NT threads per (slice, row).  MULTI: S > 1 slices per row meeting
// at barriers through the row's control block `ctl` (zeroed by the scoring
// kernel) and the per-slice records `rec`.
// Eight consecutive floats in one 32-byte load (read-only path; `p` 32-byte
// aligned): half the requests of two 16-byte loads for a thread's run.
__device__ __forceinline__ void ldg8(const float *p, float (&v)[8]) {
  asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
                 "=f"(v[7])
               : "l"(p));
}

template <int NT, int KPT, bool MULTI>
__global__ void __launch_bounds__(NT) topk_radix_kernel(csa_index_args a,
                                                        const float *__restrict__ scores, int cols,
                                                        int row0, int S, int slice, uint32_t *ctl,
                                                        uint32_t *rec, TopkSel sel) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  // long rows: TK_PRIV first-digit histograms (warp w counts into w % TK_PRIV;
  // the first digit is the most crowded) and the CTA's histogram;
  // short rows (one CTA per row, at most 16384 entries): the CTA's histogram
  // alone, then the staging of the winners -- a smaller CTA, so that more rows
  // are resident at once
  uint32_t *priv = MULTI ? tk_smem : tk_smem + TK_B1;  // [TK_PRIV][TK_B1] or staging [2 k]
  uint32_t *hist = MULTI ? tk_smem + TK_PRIV * TK_B1 : tk_smem;  // [TK_B1]
  __shared__ int warp_sums[32];
  __shared__ int s_digit, s_above, s_ok;
  __shared__ int s_gt_before, s_eq_before;
  // the first digit's histograms are cleared while the previous kernel
  // finishes (shared memory only)
  {
    uint4 *p4 = reinterpret_cast<uint4 *>(MULTI ? priv : hist);
    for (int i = threadIdx.x; i < (MULTI ? TK_PRIV : 1) * TK_B1 / 4; i += NT)
      p4[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int t = row0 + blockIdx.y, s = blockIdx.x, tid = threadIdx.x, warp = tid >> 5;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;  // uniform over the row's CTAs
  const int n_cap = a.max_blocks * kBlock;
  int V = min(visible_count(a.row_pos[t], a.ratio, a.n_cmp[b]), n_cap);
  if (sel.v_row)
    V = sel.v_row[t];
  else if (sel.v_div > 1)
    V = (V + sel.v_div - 1) / sel.v_div;
  V = max(0, min(V, sel.n_cap));
  const int k = a.topk;
  int32_t *out = a.topk_idx + (long long)t * k;
  float *out_s = a.topk_score ? a.topk_score + (long long)t * k : nullptr;
  const float *sc = scores + (long long)t * cols;
  // entry i of the row -> the position it stands for
  const int32_t *cand = sel.cand ? sel.cand + (long long)t * sel.cand_stride : nullptr;
  const int cb_mask = (1 << sel.cb_shift) - 1;
  auto position = [&](int i) {
    return cand ? (cand[i >> sel.cb_shift] << sel.cb_shift) | (i & cb_mask) : i;
  };
  if (V <= k) {
    if (s == 0)
      for (int i = tid; i < k; i += NT) {
        out[i] = i < V ? position(i) : -1;
        if (out_s) out_s[i] = i < V ? sc[i] : -INFINITY;
      }
    return;
  }
  const int c_lo = s * slice, c_hi = min(V, c_lo + slice);
  const int c0 = c_lo + tid * KPT;
  const int nv = max(0, min(KPT, c_hi - c0));

  // ---- keys of this thread's run of positions (through L1: the scores come
  // from the scoring kernel that ran before this one; each thread's run covers
  // whole 128-byte lines, fetched once for its consecutive vector loads)
  uint32_t key[KPT];
  if (nv == KPT && (reinterpret_cast<uintptr_t>(sc + c0) & 31u) == 0) {
#pragma unroll
    for (int i = 0; i < KPT; i += 8) {
      float v[8];
      ldg8(sc + c0 + i, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) key[i + q] = order_key(v[q]);
    }
  } else if (nv == KPT && (reinterpret_cast<uintptr_t>(sc + c0) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < KPT; i += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(sc + c0 + i));
      key[i] = order_key(v.x);
      key[i + 1] = order_key(v.y);
      key[i + 2] = order_key(v.z);
      key[i + 3] = order_key(v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; ++i) key[i] = i < nv ? order_key(__ldg(sc + c0 + i)) : 0u;
  }

  uint32_t *row_ctl = MULTI ? ctl + (long long)t * kTopkCtlWords : nullptr;
  int remaining = k;
  uint32_t prefix = 0, pmask = 0;
  int gt22 = 0;
#pragma unroll 1
  for (int j = 0; j < 3; ++j) {  // digit j: nb bins at `shift`
    const int nb = j == 2 ? TK_B3 : TK_B1;
    const int shift = j == 0 ? 21 : (j == 1 ? 10 : 0);
    if (j > 0)
      for (int i = tid; i < nb; i += NT) hist[i] = 0u;
    if (MULTI && j == 2) {
      // keys above the 22-bit prefix, for the offsets of later slices
      int c = 0;
#pragma unroll
      for (int i = 0; i < KPT; ++i) c += (i < nv && (key[i] >> 10) > (prefix >> 10)) ? 1 : 0;
      int tot;
      block_exclusive_scan(c, warp_sums, &tot);
      gt22 = tot;
    }
    __syncthreads();
    if (MULTI && j == 0) {
      uint32_t *mine = priv + (warp % TK_PRIV) * TK_B1;
#pragma unroll
      for (int i = 0; i < KPT; ++i)
        if (i < nv) atomicAdd(&mine[key[i] >> 21], 1u);
      __syncthreads();
      for (int i = tid; i < TK_B1; i += NT) {
        uint32_t sum = 0;
#pragma unroll
        for (int w = 0; w < TK_PRIV; ++w) sum += priv[w * TK_B1 + i];
        hist[i] = sum;
      }
    } else {
#pragma unroll
      for (int i = 0; i < KPT; ++i)
        if (i < nv && (key[i] & pmask) == prefix) atomicAdd(&hist[(key[i] >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (MULTI) {
      uint32_t *g = row_ctl + TK_CTL_HDR + (j == 0 ? 0 : (j == 1 ? TK_B1 : TK_B1 + TK_B2));
      for (int i = tid; i < nb; i += NT) {
        const uint32_t v = hist[i];
        if (v) atomicAdd(&g[i], v);
      }
      if (j == 2) {
        // suffix sums of this slice's own last-digit histogram
        static_assert(TK_B3 == 2 * NT || !MULTI, "two last-digit bins per thread");
        uint32_t *r = rec + ((long long)t * S + s) * TK_REC_WORDS;
        const int hi = TK_B3 - 1 - 2 * tid;
        const int h0 = (int)hist[hi], h1 = (int)hist[hi - 1];
        int tot;
        const int before = block_exclusive_scan(h0 + h1, warp_sums, &tot);
        r[hi] = (uint32_t)(before + h0);
        r[hi - 1] = (uint32_t)(before + h0 + h1);
        if (tid == 0) {
          r[TK_B3] = 0u;
          r[TK_REC_GT] = (uint32_t)gt22;
        }
      }
      if (!row_barrier(row_ctl, (uint32_t)((j + 1) * S), a.status_dev, &s_ok, a.wait_limit_ns))
        return;
      for (int i = tid; i < nb; i += NT) hist[i] = __ldcg(&g[i]);
      __syncthreads();
    }
    if (tid < 32) warp_find_digit(hist, nb, remaining, &s_digit, &s_above);
    __syncthreads();
    prefix |= (uint32_t)s_digit << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    remaining -= s_above;
  }
  const uint32_t T = prefix;  // the k-th largest key; `remaining` keys equal to T are taken
  const int d3 = (int)(T & (TK_B3 - 1));

  // ---- entries of the slices before this one
  int gt_before = 0, eq_before = 0;
  if (MULTI) {
    if (tid == 0) {
      s_gt_before = 0;
      s_eq_before = 0;
    }
    __syncthreads();
    for (int j = tid; j < s; j += NT) {
      const uint32_t *r = rec + ((long long)t * S + j) * TK_REC_WORDS;
      const int above = (int)__ldcg(r + d3 + 1);
      const int ge = (int)__ldcg(r + d3);
      atomicAdd(&s_gt_before, (int)__ldcg(r + TK_REC_GT) + above);
      atomicAdd(&s_eq_before, ge - above);
    }
    __syncthreads();
    gt_before = s_gt_before;
    eq_before = s_eq_before;
  }
  const int quota = max(0, remaining - eq_before);  // equal keys this slice may still take
  const int offset = gt_before + min(remaining, eq_before);

  // ---- ordered compaction: greater keys, then equal keys by ascending position
  int n_gt = 0, n_eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    n_gt += (i < nv && key[i] > T) ? 1 : 0;
    n_eq += (i < nv && key[i] == T) ? 1 : 0;
  }
  // one scan of both counts (each total stays below 2^16)
  int tot;
  const int before = block_exclusive_scan((n_eq << 16) | n_gt, warp_sums, &tot);
  const int eq_rank = before >> 16, gt_rank = before & 0xFFFF;
  const int take_eq = max(0, min(n_eq, quota - eq_rank));
  // the slice's winners are staged in shared memory (the first-digit
  // histograms are free by now) and leave in coalesced stores
  const int n_sel = tot & 0xFFFF;
  const int n_take = min(n_sel + min(quota, tot >> 16), k - offset);
  int32_t *st_idx = reinterpret_cast<int32_t *>(priv);
  uint32_t *st_key = priv + k;
  int pos = gt_rank + min(eq_rank, quota);
  int eq_seen = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (i < nv) {
      bool take = key[i] > T;
      if (key[i] == T) take = eq_seen++ < take_eq;
      if (take) {
        if (pos < n_take) {
          st_idx[pos] = c0 + i;
          st_key[pos] = key[i];
        }
        ++pos;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < n_take; i += NT) {
    out[offset + i] = position(st_idx[i]);
    if (out_s) out_s[offset + i] = key_score(st_key[i]);
  }
}

int device_sms() {
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

constexpr int TK_SHORT_MAX = 512 * TK_SHORT_KPT2;
constexpr int TK_SLICE_MAX = TK_LONG_THREADS * TK_LONG_KPT;

// Opt a kernel into more than 48 KB of dynamic shared memory, once per device.
template <typename K>
cudaError_t allow_smem(K kern, int bytes, bool *done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <int NT, int KPT>
cudaError_t launch_short(const csa_index_args &a, const float *scores, int cols, cudaStream_t s,
                         const TopkSel &sel) {
  static bool done[64] = {};
  const auto kern = topk_radix_kernel<NT, KPT, false>;
  // the CTA's histogram and the staging of at most k winners (keys and indices)
  const int smem = (TK_B1 + 2 * a.topk) * 4;
  cudaError_t e = allow_smem(kern, (TK_B1 + 2 * 2048) * 4, done);
  if (e != cudaSuccess) return e;
  constexpr int kMaxGridY = 65535;
  for (int row0 = 0; row0 < a.n_rows && e == cudaSuccess; row0 += kMaxGridY)
    e = launch_kernel(kern, dim3(1, std::min(kMaxGridY, a.n_rows - row0)), dim3(NT),
                      (size_t)smem, s, 0, false, a, scores, cols, row0, 1, NT * KPT,
                      static_cast<uint32_t *>(nullptr), static_cast<uint32_t *>(nullptr), sel);
  return e != cudaSuccess ? e : cudaGetLastError();
}

struct LongLayout {
  size_t ctl, rec, total;
};

LongLayout long_layout(int n_rows, int S) {
  LongLayout L;
  L.ctl = 0;
  L.rec = align_up((size_t)n_rows * kTopkCtlWords * 4, 256);
  L.total = L.rec + align_up((size_t)n_rows * S * TK_REC_WORDS * 4, 256);
  return L;
}

}  // namespace

bool topk_is_long(int n_cap) { return n_cap > TK_SHORT_MAX; }

// Slices per row for the long-row path: about TK_LONG_PER_SM CTAs per SM over
// the rows, each slice a multiple of 32 entries and at most 512 x 16 entries.
void topk_long_geometry(int n_rows, int n_cap, int *S, int *slice) {
  const int s_min = (n_cap + TK_SLICE_MAX - 1) / TK_SLICE_MAX;
  int s = n_rows > 0 ? TK_LONG_PER_SM * device_sms() / n_rows : 1;
  if (s < s_min) s = s_min;
  int sl = (n_cap + s - 1) / s;
  sl = (sl + 31) / 32 * 32;
  if (sl > TK_SLICE_MAX) sl = TK_SLICE_MAX;
  *S = (n_cap + sl - 1) / sl;
  *slice = sl;
}

size_t topk_ws_bytes(int n_rows, int n_cap) {
  if (!topk_is_long(n_cap)) return 0;
  int S, slice;
  topk_long_geometry(n_rows, n_cap, &S, &slice);
  return long_layout(n_rows, S).total;
}

uint32_t *topk_counters(void *ws, int n_rows, int n_cap) {
  if (!topk_is_long(n_cap)) return nullptr;
  return reinterpret_cast<uint32_t *>(ws);
}

cudaError_t launch_index_topk(const csa_index_args &a, const float *scores, int score_cols,
                              void *topk_ws, cudaStream_t s, const TopkSel &sel_in) {
  if (a.n_rows <= 0) return cudaSuccess;
  TopkSel sel = sel_in;
  if (sel.n_cap <= 0) sel.n_cap = a.max_blocks * kBlock;
  const int n_cap = sel.n_cap;
  if (!topk_is_long(n_cap)) {
    // the smallest CTA whose threads hold a whole row, 16 (or 32) entries each
    launch_begin(CSA_K_INDEX_TOPK, s);
    const cudaError_t e =
        n_cap <= 128 * TK_SHORT_KPT   ? launch_short<128, TK_SHORT_KPT>(a, scores, score_cols, s, sel)
        : n_cap <= 256 * TK_SHORT_KPT ? launch_short<256, TK_SHORT_KPT>(a, scores, score_cols, s, sel)
        : n_cap <= 512 * TK_SHORT_KPT ? launch_short<512, TK_SHORT_KPT>(a, scores, score_cols, s, sel)
                                      : launch_short<512, TK_SHORT_KPT2>(a, scores, score_cols, s, sel);
    launch_end(CSA_K_INDEX_TOPK, s);
    return e;
  }
  int S, slice;
  topk_long_geometry(a.n_rows, n_cap, &S, &slice);
  const LongLayout L = long_layout(a.n_rows, S);
  uint8_t *base = static_cast<uint8_t *>(topk_ws);
  uint32_t *ctl = reinterpret_cast<uint32_t *>(base + L.ctl);
  uint32_t *rec = reinterpret_cast<uint32_t *>(base + L.rec);
  // the CTAs of a row wait on one another: a launch holds only as many rows
  // as can be resident at once
  const auto kern = topk_radix_kernel<TK_LONG_THREADS, TK_LONG_KPT, true>;
  constexpr int smem = topk_smem_bytes<TK_LONG_THREADS>();
  static bool done[64] = {};
  cudaError_t e = allow_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TK_LONG_THREADS, smem);
  if (e != cudaSuccess) return e;
  const long long resident = (long long)per_sm * device_sms();
  if (resident < S) return cudaErrorCooperativeLaunchTooLarge;
  const int rows_per_launch = (int)std::min<long long>(a.n_rows, resident / S);
  csa_index_args aa = a;
  const float *sp = scores;
  int cols = score_cols;
  launch_begin(CSA_K_INDEX_TOPK, s);
  for (int row0 = 0; row0 < a.n_rows && e == cudaSuccess; row0 += rows_per_launch) {
    const int nr = std::min(rows_per_launch, a.n_rows - row0);
    e = launch_kernel(kern, dim3(S, nr), dim3(TK_LONG_THREADS), (size_t)smem, s, 0, true, aa, sp,
                      cols, row0, S, slice, ctl, rec, sel);
  }
  launch_end(CSA_K_INDEX_TOPK, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
