// Deterministic top-k over the lightning-indexer scores: the k entries with
// the highest score (equal scores: the smaller position first), emitted as
// logical positions in ascending order with trailing -1 padding ("DeepSeek
// V4.1 Flash", "Compressor state ownership": Top-K eligibility, uniqueness,
// logical-position ordering and trailing -1; "Hyper-Parallel ... DeepSeek V4
// CP", "10.3 Causal mask" for the visible range).
//
// Scores become order-preserving 32-bit keys.  Rows up to 8192 entries are
// selected by one CTA in shared memory (4-digit radix select, then an
// ordered compaction).  Longer rows are split over S CTAs of a cooperative
// launch: each slice histograms the top 11 key bits, the CTAs of a row meet
// at a bounded barrier, every slice marks its certain winners in a bitmap
// and spills the entries of the threshold bin, and the row's first CTA
// resolves those exactly and compacts the bitmap into ascending positions.
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

// Warp 0 finds, scanning digits from the top, the digit d whose cumulative
// count first reaches `remaining`; returns d and the count above it.
__device__ __forceinline__ void warp_find_digit(const uint32_t *hist, int n_digits, int remaining,
                                                int *digit, int *above) {
  const int lane = threadIdx.x & 31;
  int cum = 0, sel = -1, before = 0;
  for (int base = n_digits - 1; base >= 0 && sel < 0; base -= 32) {
    const int cnt = (int)hist[base - lane];
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, cum + incl >= remaining);
    if (hit) {
      const int l = __ffs(hit) - 1;
      sel = base - l;
      before = cum + __shfl_sync(0xffffffffu, incl - cnt, l);
    } else {
      cum += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  *digit = sel < 0 ? 0 : sel;
  *above = before;
}

// ---------------------------------------------------------------- short rows

constexpr int SR_THREADS = 256;
constexpr int SR_MAX = 8192;

__global__ void __launch_bounds__(SR_THREADS) topk_short_kernel(csa_index_args a,
                                                                const float *__restrict__ scores,
                                                                int cols) {
  __shared__ uint32_t keys[SR_MAX];
  __shared__ uint32_t hist[256];
  __shared__ int warp_sums[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem;
  const int t = blockIdx.x;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;
  const int V = min(min(visible_count(a.row_pos[t], a.ratio, a.n_cmp[b]), a.max_blocks * kBlock),
                    SR_MAX);
  const int k = a.topk;
  int32_t *out = a.topk_idx + (long long)t * k;
  float *out_s = a.topk_score ? a.topk_score + (long long)t * k : nullptr;
  const float *sc = scores + (long long)t * cols;
  if (V <= k) {
    for (int i = threadIdx.x; i < k; i += SR_THREADS) {
      out[i] = i < V ? i : -1;
      if (out_s) out_s[i] = i < V ? sc[i] : -INFINITY;
    }
    return;
  }
  for (int c = threadIdx.x; c < V; c += SR_THREADS) keys[c] = order_key(sc[c]);
  // radix select of the k-th largest key, 4 digits of 8 bits
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += SR_THREADS) hist[i] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < V; c += SR_THREADS) {
      const uint32_t key = keys[c];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int d, above;
      warp_find_digit(hist, 256, remaining, &d, &above);
      if (threadIdx.x == 0) {
        s_prefix = prefix | ((uint32_t)d << shift);
        s_rem = remaining - above;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_rem;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;  // the k-th largest key; `remaining` equal keys are taken
  int eq_base = 0, sel_base = 0;
  for (int c0 = 0; c0 < V; c0 += SR_THREADS) {
    const int c = c0 + threadIdx.x;
    const uint32_t key = c < V ? keys[c] : 0u;
    const int gt = (c < V && key > T) ? 1 : 0;
    const int eq = (c < V && key == T) ? 1 : 0;
    int eq_total, sel_total;
    const int eq_rank = eq_base + block_exclusive_scan(eq, warp_sums, &eq_total);
    const int sel = gt | (eq && eq_rank < remaining);
    const int pos = sel_base + block_exclusive_scan(sel, warp_sums, &sel_total);
    if (sel && pos < k) {
      out[pos] = c;
      if (out_s) out_s[pos] = sc[c];
    }
    eq_base += eq_total;
    sel_base += sel_total;
  }
  for (int i = sel_base + threadIdx.x; i < k; i += SR_THREADS) {
    out[i] = -1;
    if (out_s) out_s[i] = -INFINITY;
  }
}

// ---------------------------------------------------------------- long rows

constexpr int LR_THREADS = 512;
constexpr int LR_BINS = 2048;  // top 11 key bits
constexpr int LR_TIE_SMEM = 4096;

struct LongWs {
  uint32_t *hist_part;  // [rows][S][2048]
  uint32_t *tie_count;  // [rows][S]
  uint64_t *ties;       // [rows][S][slice]  (key << 32 | ~position)
  uint32_t *bitmap;     // [rows][n_cap / 32]
  uint32_t *counters;   // [rows], zeroed by the scoring kernel
};

// Barrier of the S CTAs that share a row.  Waits at most ~1 s; returns false
// (and flags CSA_DEV_TIMEOUT) when it gives up.
__device__ bool row_barrier(uint32_t *ctr, uint32_t target, uint32_t *status, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t t0 = tc::global_ns();
    int ok = 1;
    while (*reinterpret_cast<volatile uint32_t *>(ctr) < target) {
      if (tc::global_ns() - t0 > 1000000000ull) {
        ok = 0;
        flag(status, CSA_DEV_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Radix select of the `need` largest 64-bit composites among the ties (the
// composites are unique since positions differ); returns the smallest taken.
template <typename Visit>
__device__ uint64_t select_ties(int need, uint32_t *hist, int *s_digit, int *s_rem, Visit visit) {
  uint64_t prefix = 0, mask = 0;
  int remaining = need;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += LR_THREADS) hist[i] = 0;
    __syncthreads();
    visit([&](uint64_t v) {
      if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (threadIdx.x < 32) {
      int d, above;
      warp_find_digit(hist, 256, remaining, &d, &above);
      if (threadIdx.x == 0) {
        *s_digit = d;
        *s_rem = remaining - above;
      }
    }
    __syncthreads();
    prefix |= (uint64_t)(*s_digit) << shift;
    remaining = *s_rem;
    mask |= (uint64_t)255 << shift;
    __syncthreads();
  }
  return prefix;
}

__global__ void __launch_bounds__(LR_THREADS) topk_long_kernel(csa_index_args a,
                                                              const float *__restrict__ scores,
                                                              int cols, LongWs ws, int S,
                                                              int slice) {
  __shared__ uint32_t hist[LR_BINS];
  __shared__ int warp_sums[32];
  __shared__ int s_ok, s_ntie, s_digit, s_rem;
  __shared__ uint64_t tie_s[LR_TIE_SMEM];
  const int t = blockIdx.y, s = blockIdx.x, tid = threadIdx.x;
  const int b = a.row_req[t];
  if (b < 0 || b >= a.n_req) return;  // uniform over the row's CTAs
  const int n_cap = a.max_blocks * kBlock;
  const int V = min(visible_count(a.row_pos[t], a.ratio, a.n_cmp[b]), n_cap);
  const int k = a.topk;
  int32_t *out = a.topk_idx + (long long)t * k;
  float *out_s = a.topk_score ? a.topk_score + (long long)t * k : nullptr;
  const float *sc = scores + (long long)t * cols;
  if (V <= k) {
    if (s == 0)
      for (int i = tid; i < k; i += LR_THREADS) {
        out[i] = i < V ? i : -1;
        if (out_s) out_s[i] = i < V ? sc[i] : -INFINITY;
      }
    return;
  }
  const int c_lo = s * slice, c_hi = min(V, c_lo + slice);
  uint32_t *ctr = ws.counters + t;

  // ---- phase 1: histogram of this slice's top 11 key bits
  for (int i = tid; i < LR_BINS; i += LR_THREADS) hist[i] = 0;
  __syncthreads();
  for (int c = c_lo + tid; c < c_hi; c += LR_THREADS)
    atomicAdd(&hist[order_key(sc[c]) >> 21], 1u);
  __syncthreads();
  uint32_t *hp = ws.hist_part + ((long long)t * S + s) * LR_BINS;
  for (int i = tid; i < LR_BINS; i += LR_THREADS) hp[i] = hist[i];
  if (!row_barrier(ctr, (uint32_t)S, a.status_dev, &s_ok)) return;

  // ---- phase 2: threshold bin b* of the row (same result in every CTA)
  for (int i = tid; i < LR_BINS; i += LR_THREADS) {
    uint32_t sum = 0;
    for (int j = 0; j < S; ++j) sum += ws.hist_part[((long long)t * S + j) * LR_BINS + i];
    hist[i] = sum;
  }
  __syncthreads();
  if (tid < 32) {
    int d, above;
    warp_find_digit(hist, LR_BINS, k, &d, &above);
    if (tid == 0) {
      s_digit = d;
      s_rem = k - above;  // entries of bin b* to take
      s_ntie = 0;
    }
  }
  __syncthreads();
  const uint32_t bstar = (uint32_t)s_digit;
  const int need = s_rem;
  // mark certain winners (bin > b*), spill the threshold bin
  uint64_t *tie_g = ws.ties + ((long long)t * S + s) * slice;
  uint32_t *bm = ws.bitmap + (long long)t * (n_cap / 32);
  for (int w0 = c_lo; w0 < c_hi; w0 += 32 * LR_THREADS) {
    const int c0 = w0 + tid * 32;
    if (c0 < c_hi) {
      uint32_t word = 0;
#pragma unroll 4
      for (int i = 0; i < 32; ++i) {
        const int c = c0 + i;
        if (c < c_hi) {
          const uint32_t key = order_key(sc[c]);
          const uint32_t bin = key >> 21;
          if (bin > bstar) {
            word |= 1u << i;
          } else if (bin == bstar) {
            const int slot = atomicAdd(&s_ntie, 1);
            tie_g[slot] = ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)c);
          }
        }
      }
      bm[c0 >> 5] = word;
    }
  }
  __syncthreads();
  if (tid == 0) ws.tie_count[(long long)t * S + s] = (uint32_t)s_ntie;
  if (!row_barrier(ctr, (uint32_t)(2 * S), a.status_dev, &s_ok)) return;
  if (s != 0) return;

  // ---- phase 3 (first CTA of the row): exact choice inside the threshold bin
  int n_tie = 0;
  for (int j = 0; j < S; ++j) n_tie += (int)ws.tie_count[(long long)t * S + j];
  auto each_tie_global = [&](auto &&f) {
    for (int j = 0; j < S; ++j) {
      const int nj = (int)ws.tie_count[(long long)t * S + j];
      const uint64_t *src = ws.ties + ((long long)t * S + j) * slice;
      for (int i = tid; i < nj; i += LR_THREADS) f(src[i]);
    }
  };
  uint64_t cut;
  if (n_tie <= LR_TIE_SMEM) {
    int off = 0;
    for (int j = 0; j < S; ++j) {
      const int nj = (int)ws.tie_count[(long long)t * S + j];
      const uint64_t *src = ws.ties + ((long long)t * S + j) * slice;
      for (int i = tid; i < nj; i += LR_THREADS) tie_s[off + i] = src[i];
      off += nj;
    }
    __syncthreads();
    auto each_tie_smem = [&](auto &&f) {
      for (int i = tid; i < n_tie; i += LR_THREADS) f(tie_s[i]);
    };
    cut = select_ties(need, hist, &s_digit, &s_rem, each_tie_smem);
    each_tie_smem([&](uint64_t v) {
      if (v >= cut) {
        const uint32_t c = ~(uint32_t)(v & 0xFFFFFFFFu);
        atomicOr(&bm[c >> 5], 1u << (c & 31));
      }
    });
  } else {
    cut = select_ties(need, hist, &s_digit, &s_rem, each_tie_global);
    each_tie_global([&](uint64_t v) {
      if (v >= cut) {
        const uint32_t c = ~(uint32_t)(v & 0xFFFFFFFFu);
        atomicOr(&bm[c >> 5], 1u << (c & 31));
      }
    });
  }
  __threadfence_block();
  __syncthreads();

  // ---- ordered compaction of the bitmap: positions ascending
  const int n_words = (V + 31) / 32;
  const int per = (n_words + LR_THREADS - 1) / LR_THREADS;
  const int w_lo = min(n_words, tid * per), w_hi = min(n_words, w_lo + per);
  const uint32_t tail_mask = (V & 31) ? ((1u << (V & 31)) - 1u) : 0xFFFFFFFFu;
  int cnt = 0;
  for (int w = w_lo; w < w_hi; ++w) {
    uint32_t word = bm[w];
    if (w == n_words - 1) word &= tail_mask;
    cnt += __popc(word);
  }
  int total;
  int pos = block_exclusive_scan(cnt, warp_sums, &total);
  for (int w = w_lo; w < w_hi; ++w) {
    uint32_t word = bm[w];
    if (w == n_words - 1) word &= tail_mask;
    while (word) {
      const int i = __ffs(word) - 1;
      word &= word - 1;
      const int c = w * 32 + i;
      if (pos < k) {
        out[pos] = c;
        if (out_s) out_s[pos] = sc[c];
      }
      ++pos;
    }
  }
  for (int i = total + tid; i < k; i += LR_THREADS) {
    out[i] = -1;
    if (out_s) out_s[i] = -INFINITY;
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

struct LongLayout {
  size_t hist, tie_count, ties, bitmap, counters, total;
};

LongLayout long_layout(int n_rows, int n_cap, int S, int slice) {
  LongLayout L;
  size_t off = 0;
  L.hist = off;
  off += align_up((size_t)n_rows * S * LR_BINS * 4, 256);
  L.tie_count = off;
  off += align_up((size_t)n_rows * S * 4, 256);
  L.ties = off;
  off += align_up((size_t)n_rows * S * slice * 8, 256);
  L.bitmap = off;
  off += align_up((size_t)n_rows * (n_cap / 32) * 4, 256);
  L.counters = off;
  off += align_up((size_t)n_rows * 4, 256);
  L.total = off;
  return L;
}

}  // namespace

bool topk_is_long(int n_cap) { return n_cap > SR_MAX; }

// Slices per row for the long-row path: about one CTA per SM in total, each
// slice a multiple of 32 entries (one bitmap word per thread step).
void topk_long_geometry(int n_rows, int n_cap, int *S, int *slice) {
  int s = n_rows > 0 ? (148 + n_rows - 1) / n_rows : 1;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  int sl = (n_cap + s - 1) / s;
  sl = (sl + 31) / 32 * 32;
  *S = (n_cap + sl - 1) / sl;
  *slice = sl;
}

size_t topk_ws_bytes(int n_rows, int n_cap) {
  if (!topk_is_long(n_cap)) return 0;
  int S, slice;
  topk_long_geometry(n_rows, n_cap, &S, &slice);
  return long_layout(n_rows, n_cap, S, slice).total;
}

uint32_t *topk_counters(void *ws, int n_rows, int n_cap) {
  if (!topk_is_long(n_cap)) return nullptr;
  int S, slice;
  topk_long_geometry(n_rows, n_cap, &S, &slice);
  return reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                      long_layout(n_rows, n_cap, S, slice).counters);
}

cudaError_t launch_index_topk(const csa_index_args &a, const float *scores, int score_cols,
                              void *topk_ws, cudaStream_t s) {
  if (a.n_rows <= 0) return cudaSuccess;
  const int n_cap = a.max_blocks * kBlock;
  if (!topk_is_long(n_cap)) {
    launch_begin(CSA_K_INDEX_TOPK, s);
    topk_short_kernel<<<a.n_rows, SR_THREADS, 0, s>>>(a, scores, score_cols);
    launch_end(CSA_K_INDEX_TOPK, s);
    return cudaGetLastError();
  }
  int S, slice;
  topk_long_geometry(a.n_rows, n_cap, &S, &slice);
  const LongLayout L = long_layout(a.n_rows, n_cap, S, slice);
  uint8_t *base = static_cast<uint8_t *>(topk_ws);
  LongWs ws;
  ws.hist_part = reinterpret_cast<uint32_t *>(base + L.hist);
  ws.tie_count = reinterpret_cast<uint32_t *>(base + L.tie_count);
  ws.ties = reinterpret_cast<uint64_t *>(base + L.ties);
  ws.bitmap = reinterpret_cast<uint32_t *>(base + L.bitmap);
  ws.counters = reinterpret_cast<uint32_t *>(base + L.counters);
  const dim3 grid(S, a.n_rows);
  if (S > 1) {
    // the CTAs of a row wait on one another: they must all be resident at once
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_long_kernel, LR_THREADS, 0) !=
            cudaSuccess ||
        (long long)S * a.n_rows > (long long)per_sm * device_sms())
      return cudaErrorCooperativeLaunchTooLarge;
  }
  csa_index_args aa = a;
  const float *sp = scores;
  int cols = score_cols;
  void *args[] = {&aa, &sp, &cols, &ws, &S, &slice};
  launch_begin(CSA_K_INDEX_TOPK, s);
  cudaError_t e = S > 1 ? cudaLaunchCooperativeKernel((const void *)topk_long_kernel, grid,
                                                      dim3(LR_THREADS), args, 0, s)
                        : cudaLaunchKernel((const void *)topk_long_kernel, grid,
                                           dim3(LR_THREADS), args, 0, s);
  launch_end(CSA_K_INDEX_TOPK, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa
