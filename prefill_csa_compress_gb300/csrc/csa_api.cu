// extern "C" entry points: host-side argument checks, workspace layout and
// kernel dispatch.  No entry point synchronises or allocates device memory.
#include <atomic>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <vector>

#include "csa_internal.cuh"

namespace csa {

// ---------------------------------------------------------------- launch accounting

static std::atomic<uint64_t> g_launches{0};

struct ProfState {
  std::mutex mu;
  int kernel_id = -1;
  int max_launches = 0;
  int recorded = 0;
  std::vector<cudaEvent_t> ev;     // 2 per launch
  cudaStream_t side = nullptr;     // where the timing events are recorded
  cudaEvent_t fork = nullptr;      // hands the launching stream's position to `side`
  cudaEvent_t join = nullptr;
};
static ProfState g_prof;

// Inside stream capture an event record becomes a graph node only with the
// external flag; such nodes re-record the event at every replay.
void record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

// Records `e` on the side stream once everything issued so far on `s` is
// done.  Nothing is added to `s` itself, so the next kernel on `s` still
// launches as a programmatic dependent of the one before it.
static void record_beside(cudaEvent_t e, cudaStream_t s) {
  cudaEventRecord(g_prof.fork, s);
  cudaStreamWaitEvent(g_prof.side, g_prof.fork, 0);
  record_event(e, g_prof.side);
}

void launch_begin(int kernel_id, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof.kernel_id != kernel_id) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.recorded < g_prof.max_launches) record_beside(g_prof.ev[2 * g_prof.recorded], s);
}

void launch_end(int kernel_id, cudaStream_t s) {
  if (g_prof.kernel_id != kernel_id) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.recorded < g_prof.max_launches) {
    record_beside(g_prof.ev[2 * g_prof.recorded + 1], s);
    ++g_prof.recorded;
  }
}

// The arguments as this library's struct: a caller built against the header
// without the hierarchical-indexer fields gets neither mode.
csa_index_args full_index_args(const csa_index_args *a) {
  csa_index_args f;
  memset(&f, 0, sizeof(f));
  memcpy(&f, a, a->struct_size < sizeof(f) ? a->struct_size : sizeof(f));
  f.struct_size = sizeof(f);
  return f;
}

bool index_pointers_ok(const csa_index_args *a) {
  const bool fp4 = a->key_fmt == CSA_FMT_FP4_E8M0 || a->key_fmt == CSA_FMT_MXFP8;
  if (!a->q_idx || !a->weights || !a->row_req || !a->row_pos || !a->n_cmp || !a->idx_pool ||
      !a->cmp_block_table || !a->topk_idx)
    return false;
  if (fp4 ? !a->key_scale_pool : !a->idx_scale_pool) return false;
  if (a->n_req <= 0 || a->n_blocks <= 0) return false;
  if ((a->rope_cos == nullptr) != (a->rope_sin == nullptr)) return false;
  if (a->rope_cos && a->rope_cap <= 0) return false;
  const void *scales = fp4 ? static_cast<const void *>(a->key_scale_pool)
                           : static_cast<const void *>(a->idx_scale_pool);
  const uintptr_t m = reinterpret_cast<uintptr_t>(a->idx_pool) |
                      reinterpret_cast<uintptr_t>(a->q_idx) | reinterpret_cast<uintptr_t>(scales);
  return (m & 15u) == 0;
}

csa_status_t index_normalize_strides(csa_index_args *a) {
  if (a->key_fmt == CSA_FMT_FP4_E8M0) {  // packed keys: dense only
    if (a->key_page_stride || a->key_row_stride || a->scale_page_stride)
      return CSA_ERR_UNSUPPORTED;
    a->key_row_stride = kIdxDim / 2;
    a->key_page_stride = kBlock * a->key_row_stride;
    a->scale_page_stride = kBlock * 4;
    return CSA_OK;
  }
  if (a->key_fmt == CSA_FMT_MXFP8 && a->scale_page_stride) return CSA_ERR_UNSUPPORTED;
  if (!normalize_strides(&a->key_page_stride, &a->key_row_stride, kIdxDim))
    return CSA_ERR_INVALID_ARG;
  if (a->scale_page_stride == 0) a->scale_page_stride = kBlock * 4;
  if (a->scale_page_stride % 16 != 0 || a->scale_page_stride < kBlock * 4)
    return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

bool index_struct_ok(const csa_index_args *a) {
  return a && a->struct_size >= offsetof(csa_index_args, cand_block);
}

}  // namespace csa

using namespace csa;

namespace {

constexpr size_t kAlign = 256;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

// shape checks (enough to size the workspace)
csa_status_t check_attn_shape(const csa_attn_args *a) {
  if (!a) return CSA_ERR_INVALID_ARG;
  if (a->n_rows < 0 || a->n_req < 0 || a->topk < 0 || a->topk > CSA_MAX_TOPK)
    return CSA_ERR_INVALID_ARG;
  if (a->n_heads < 1 || a->n_heads > kMaxHeads || a->head_dim != kHeadDim || a->window != kWindow)
    return CSA_ERR_UNSUPPORTED;
  if (a->ratio < 1) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

// pointer and size checks before a launch
csa_status_t check_attn_args(const csa_attn_args *a) {
  if (!a->q || !a->row_req || !a->row_pos || !a->kv_pool || !a->kv_block_table || !a->kv_len ||
      !a->cmp_pool || !a->cmp_block_table || !a->n_cmp || !a->out)
    return CSA_ERR_INVALID_ARG;
  if ((a->rope_cos == nullptr) != (a->rope_sin == nullptr)) return CSA_ERR_INVALID_ARG;
  if (a->rope_cos && a->rope_cap <= 0) return CSA_ERR_INVALID_ARG;
  if (a->kv_max_blocks <= 0 || a->cmp_max_blocks <= 0 || a->kv_n_blocks <= 0 ||
      a->cmp_n_blocks <= 0 || a->n_req <= 0)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(a->q) || !aligned16(a->kv_pool) || !aligned16(a->cmp_pool) || !aligned16(a->out))
    return CSA_ERR_INVALID_ARG;
  if (a->kv_fmt == CSA_FMT_MXFP8 && !a->kv_scale_pool) return CSA_ERR_INVALID_ARG;
  if (a->cmp_fmt == CSA_FMT_FP4_E4M3 &&
      (!a->cmp_scale_pool || (reinterpret_cast<uintptr_t>(a->cmp_scale_pool) & 1u)))
    return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

csa_status_t run_attn(csa_attn_args *user, cudaStream_t s, bool decode) {
  // the arguments as this library's struct: a caller built against the header
  // without the cache-format fields reads both pools as BF16
  if (!user || user->struct_size < offsetof(csa_attn_args, kv_fmt)) return CSA_ERR_INVALID_ARG;
  csa_attn_args A;
  memset(&A, 0, sizeof(A));
  memcpy(&A, user, user->struct_size < sizeof(A) ? user->struct_size : sizeof(A));
  A.struct_size = sizeof(A);
  csa_attn_args *a = &A;
  csa_status_t st = check_attn_shape(a);
  if (st != CSA_OK) return st;
  if ((a->kv_fmt != CSA_FMT_BF16 && a->kv_fmt != CSA_FMT_MXFP8) ||
      (a->cmp_fmt != CSA_FMT_BF16 && a->cmp_fmt != CSA_FMT_FP4_E4M3))
    return CSA_ERR_UNSUPPORTED;
  // pool strides: explicit for BF16 pools, dense for the low-bit formats
  if ((a->kv_fmt != CSA_FMT_BF16 && (a->kv_page_stride || a->kv_row_stride)) ||
      (a->cmp_fmt != CSA_FMT_BF16 && (a->cmp_page_stride || a->cmp_row_stride)))
    return CSA_ERR_UNSUPPORTED;
  if (!normalize_strides(&a->kv_page_stride, &a->kv_row_stride,
                         a->kv_fmt == CSA_FMT_BF16 ? 2 * kHeadDim : kHeadDim) ||
      !normalize_strides(&a->cmp_page_stride, &a->cmp_row_stride,
                         a->cmp_fmt == CSA_FMT_BF16 ? 2 * kHeadDim : kHeadDim / 2))
    return CSA_ERR_INVALID_ARG;
  // the decode call merges its split partials through the workspace; the
  // prefill call's low-bit pools go through a BF16 arena in it
  const size_t need = decode ? attn_decode_workspace(*a) : attn_arena_bytes(*a);
  if (!a->workspace) {
    user->workspace_bytes = need;
    return CSA_OK;
  }
  if (a->workspace_bytes < need) return CSA_ERR_INVALID_ARG;
  if (a->n_rows == 0) return CSA_OK;
  st = check_attn_args(a);
  if (st != CSA_OK) return st;
  if (decode) return from_cuda(launch_attn_decode(*a, s));
  if (!attn_prefill_supported(*a)) return CSA_ERR_UNSUPPORTED;
  if (need == 0) return from_cuda(launch_attn_prefill(*a, s));
  csa_attn_args bf;
  const cudaError_t e = launch_dequant_arena(*a, a->workspace, &bf, s);
  return from_cuda(e != cudaSuccess ? e : launch_attn_prefill(bf, s));
}

}  // namespace

extern "C" {

CSA_API const char *csa_version(void) { return "csa 0.1.0 sm_103a"; }

CSA_API const char *csa_status_string(csa_status_t s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

CSA_API uint64_t csa_launch_count(void) { return g_launches.load(); }

// ---------------------------------------------------------------- compress

// Host checks of one compressor call.  Sets *size_query when the call only
// reports its workspace size (already stored in a->workspace_bytes).
static csa_status_t check_compress(csa_compress_args *a, bool *size_query) {
  *size_query = false;
  if (!a || a->struct_size < offsetof(csa_compress_args, state_cache)) return CSA_ERR_INVALID_ARG;
  if (a->n_rows < 0 || a->n_req < 0) return CSA_ERR_INVALID_ARG;
  if (a->ratio != 1 && a->ratio != 2 && a->ratio != 4 && a->ratio != 128)
    return CSA_ERR_UNSUPPORTED;
  if (a->d != 128 && a->d != 512) return CSA_ERR_UNSUPPORTED;
  if (a->overlap != 0 && a->overlap != 1) return CSA_ERR_INVALID_ARG;
  if (a->overlap && a->ratio > 64) return CSA_ERR_UNSUPPORTED;
  if (a->dx <= 0 || a->dx % 64 != 0 || a->dx > 1024) return CSA_ERR_UNSUPPORTED;
  if (a->out_mode < CSA_OUT_BF16 || a->out_mode > CSA_OUT_MXFP8) return CSA_ERR_INVALID_ARG;
  const size_t need = align_up((size_t)a->n_rows * a->d * sizeof(float), kAlign);
  if (!a->workspace) {
    a->workspace_bytes = need;
    *size_query = true;
    return CSA_OK;
  }
  if (a->workspace_bytes < need) return CSA_ERR_INVALID_ARG;
  if (a->n_rows == 0) return CSA_OK;
  if (!a->x || !a->kv || !a->w_gate || !a->ape || !a->positions || !a->row_req ||
      !a->block_table)
    return CSA_ERR_INVALID_ARG;
  if (a->n_req <= 0 || a->max_blocks <= 0 || a->n_blocks <= 0) return CSA_ERR_INVALID_ARG;
  if (a->out_mode == CSA_OUT_BF16 && !a->cmp_pool) return CSA_ERR_INVALID_ARG;
  if (a->out_mode == CSA_OUT_INT8 && (!a->idx_pool || !a->idx_scale_pool))
    return CSA_ERR_INVALID_ARG;
  if ((a->out_mode == CSA_OUT_FP4_E4M3 || a->out_mode == CSA_OUT_FP4_E8M0 ||
       a->out_mode == CSA_OUT_MXFP8) &&
      (!a->cmp_pool || !a->scale_pool))
    return CSA_ERR_INVALID_ARG;
  if (a->rotate && (!a->rope_cos || !a->rope_sin || a->rope_cap <= 0)) return CSA_ERR_INVALID_ARG;
  if (!aligned16(a->x) || !aligned16(a->kv) || !aligned16(a->w_gate)) return CSA_ERR_INVALID_ARG;
  if (a->state_cache &&
      (!a->state_block_table || a->n_state_blocks <= 0 ||
       a->state_capacity < (a->overlap ? 2 : 1) * a->ratio || a->state_capacity > 256))
    return CSA_ERR_INVALID_ARG;
  // output pool strides: explicit for BF16 and INT8 publication, dense for
  // the low-bit formats
  if (a->out_mode == CSA_OUT_BF16 || a->out_mode == CSA_OUT_INT8) {
    if (!normalize_strides(&a->pool_page_stride, &a->pool_row_stride,
                           a->out_mode == CSA_OUT_BF16 ? 2 * a->d : a->d))
      return CSA_ERR_INVALID_ARG;
    if (a->scale_page_stride == 0) a->scale_page_stride = kBlock * 4;
    if (a->scale_page_stride % 4 != 0 || a->scale_page_stride < kBlock * 4)
      return CSA_ERR_INVALID_ARG;
  } else if (a->pool_page_stride || a->pool_row_stride || a->scale_page_stride) {
    return CSA_ERR_UNSUPPORTED;
  }
  return CSA_OK;
}

// The arguments as this library's struct: a caller built against the header
// without the state-ring fields (a smaller struct_size) gets no ring.
static csa_compress_args full_args(const csa_compress_args *a) {
  csa_compress_args f;
  memset(&f, 0, sizeof(f));
  memcpy(&f, a, a->struct_size < sizeof(f) ? a->struct_size : sizeof(f));
  f.struct_size = sizeof(f);
  return f;
}

CSA_API csa_status_t csa_compress(csa_compress_args *a, csa_stream_t stream) {
  if (!a || a->struct_size < offsetof(csa_compress_args, state_cache)) return CSA_ERR_INVALID_ARG;
  csa_compress_args f = full_args(a);
  bool query = false;
  const csa_status_t st = check_compress(&f, &query);
  if (query) a->workspace_bytes = f.workspace_bytes;
  if (st != CSA_OK || query || f.n_rows == 0) return st;
  return from_cuda(
      launch_compress(f, static_cast<float *>(f.workspace), static_cast<cudaStream_t>(stream)));
}

CSA_API csa_status_t csa_compress_pair(csa_compress_args *first, csa_compress_args *second,
                                       csa_stream_t stream) {
  for (const csa_compress_args *x : {first, second})
    if (!x || x->struct_size < offsetof(csa_compress_args, state_cache)) return CSA_ERR_INVALID_ARG;
  csa_compress_args f1 = full_args(first), f2 = full_args(second);
  bool q1 = false, q2 = false;
  csa_status_t st = check_compress(&f1, &q1);
  if (q1) first->workspace_bytes = f1.workspace_bytes;
  if (st != CSA_OK) return st;
  st = check_compress(&f2, &q2);
  if (q2) second->workspace_bytes = f2.workspace_bytes;
  if (st != CSA_OK || q1 || q2) return st;
  return from_cuda(launch_compress_pair(f1, static_cast<float *>(f1.workspace), f2,
                                        static_cast<float *>(f2.workspace),
                                        static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- index + top-k

namespace {

int log2_exact(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return (1 << s) == x ? s : -1;
}

// Workspace of csa_index_topk: [scores][top-k control][level one: block
// maxima][level one: block top-k control][reindex: per-row entry counts].
struct IndexLayout {
  int row_cap;   // entries of one score row
  int blk_cols;  // level one: blocks of one row
  size_t scores, topk, blk, topk2, v_row, total;
};

IndexLayout index_layout(const csa_index_args &a, bool own_scores) {
  IndexLayout L{};
  const int n_cap = a.max_blocks * kBlock;
  const bool lvl1 = a.cand_out != nullptr, reidx = a.cand_in != nullptr;
  L.row_cap = reidx ? a.n_cand * a.cand_block : n_cap;
  L.blk_cols = lvl1 ? n_cap / a.cand_block : 0;
  size_t off = 0;
  L.scores = off;
  off += own_scores ? 0 : align_up((size_t)a.n_rows * L.row_cap * sizeof(float), kAlign);
  L.topk = off;
  off += align_up(topk_ws_bytes(a.n_rows, L.row_cap), kAlign);
  L.blk = off;
  if (lvl1) off += align_up((size_t)a.n_rows * L.blk_cols * sizeof(float), kAlign);
  L.topk2 = off;
  if (lvl1) off += align_up(topk_ws_bytes(a.n_rows, L.blk_cols), kAlign);
  L.v_row = off;
  if (reidx) off += align_up((size_t)a.n_rows * sizeof(int32_t), kAlign);
  L.total = off;
  return L;
}

}  // namespace

CSA_API csa_status_t csa_index_topk(csa_index_args *user, csa_stream_t stream) {
  if (!index_struct_ok(user)) return CSA_ERR_INVALID_ARG;
  csa_index_args A = full_index_args(user);
  const csa_index_args *a = &A;
  if (a->n_rows < 0 || a->n_req < 0) return CSA_ERR_INVALID_ARG;
  {
    const csa_status_t st = index_normalize_strides(&A);
    if (st != CSA_OK) return st;
  }
  if (a->n_heads < 1 || a->n_heads > kMaxHeads || a->head_dim != kIdxDim)
    return CSA_ERR_UNSUPPORTED;
  if (a->topk < 1 || a->topk > CSA_MAX_TOPK || a->ratio < 1) return CSA_ERR_INVALID_ARG;
  if (a->max_blocks <= 0) return CSA_ERR_INVALID_ARG;
  // the hierarchical modes take one 64-head slot per row
  if (a->n_heads > kHeads && (a->cand_out || a->cand_in)) return CSA_ERR_UNSUPPORTED;
  if (a->key_fmt != 0 && a->key_fmt != CSA_FMT_INT8 && a->key_fmt != CSA_FMT_FP4_E8M0 &&
      a->key_fmt != CSA_FMT_MXFP8)
    return CSA_ERR_UNSUPPORTED;
  const bool lvl1 = a->cand_out != nullptr, reidx = a->cand_in != nullptr;
  int cb_shift = 3;
  if (lvl1 || reidx) {
    if (lvl1 && reidx) return CSA_ERR_INVALID_ARG;
    if (a->cand_block != 8 && a->cand_block != 16 && a->cand_block != 32)
      return CSA_ERR_UNSUPPORTED;
    if (a->n_cand < 1 || a->n_cand > CSA_MAX_TOPK) return CSA_ERR_INVALID_ARG;
    cb_shift = log2_exact(a->cand_block);
  }
  const bool own_scores = a->scores != nullptr;
  const IndexLayout L = index_layout(*a, own_scores);
  if (own_scores && a->score_cols < L.row_cap) return CSA_ERR_INVALID_ARG;
  if (!a->workspace) {
    user->workspace_bytes = L.total;
    return CSA_OK;
  }
  if (a->workspace_bytes < L.total) return CSA_ERR_INVALID_ARG;
  if (a->n_rows == 0) return CSA_OK;
  if (!index_pointers_ok(a)) return CSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(a->workspace);
  float *scores = own_scores ? a->scores : reinterpret_cast<float *>(ws + L.scores);
  const int cols = own_scores ? a->score_cols : L.row_cap;
  void *topk_ws = ws + L.topk;
  ScoreSel ss;
  TopkSel ts;
  ts.n_cap = L.row_cap;
  if (reidx) {
    ss.cand_in = a->cand_in;
    ss.n_cand = a->n_cand;
    ss.cb_shift = cb_shift;
    ss.v_row = reinterpret_cast<int32_t *>(ws + L.v_row);
    ts.v_row = ss.v_row;
    ts.cand = a->cand_in;
    ts.cand_stride = a->n_cand;
    ts.cb_shift = cb_shift;
  }
  if (lvl1) {
    ss.cb_shift = cb_shift;
    ss.blk = reinterpret_cast<float *>(ws + L.blk);
    ss.blk_cols = L.blk_cols;
    ss.zero2 = topk_counters(ws + L.topk2, a->n_rows, L.blk_cols);
  }
  cudaError_t e =
      launch_index_scores(*a, scores, cols, topk_counters(topk_ws, a->n_rows, L.row_cap), s, ss);
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  e = launch_index_topk(*a, scores, cols, topk_ws, s, ts);
  if (e != cudaSuccess || !lvl1) return from_cuda(e);
  // level one: the best n_cand blocks by block maximum
  csa_index_args B = *a;
  B.topk = a->n_cand;
  B.topk_idx = a->cand_out;
  B.topk_score = nullptr;
  TopkSel tb;
  tb.v_div = a->cand_block;
  tb.n_cap = L.blk_cols;
  return from_cuda(launch_index_topk(B, ss.blk, L.blk_cols, ws + L.topk2, s, tb));
}

// ---------------------------------------------------------------- attention

CSA_API csa_status_t csa_sparse_attn_decode(csa_attn_args *a, csa_stream_t stream) {
  return run_attn(a, static_cast<cudaStream_t>(stream), true);
}

CSA_API csa_status_t csa_sparse_attn_prefill(csa_attn_args *a, csa_stream_t stream) {
  return run_attn(a, static_cast<cudaStream_t>(stream), false);
}

// ---------------------------------------------------------------- timing hooks

static void prof_release() {
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  if (g_prof.fork) cudaEventDestroy(g_prof.fork);
  if (g_prof.join) cudaEventDestroy(g_prof.join);
  if (g_prof.side) cudaStreamDestroy(g_prof.side);
  g_prof.fork = g_prof.join = nullptr;
  g_prof.side = nullptr;
  g_prof.kernel_id = -1;
  g_prof.recorded = 0;
  g_prof.max_launches = 0;
}

CSA_API csa_status_t csa_prof_enable(int32_t kernel_id, int32_t max_launches) {
  if (kernel_id < 0 || kernel_id >= CSA_K_COUNT || max_launches <= 0) return CSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  prof_release();
  bool ok = cudaStreamCreateWithFlags(&g_prof.side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&g_prof.fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&g_prof.join, cudaEventDisableTiming) == cudaSuccess;
  g_prof.ev.assign(2 * (size_t)max_launches, nullptr);
  for (auto &e : g_prof.ev) ok = ok && cudaEventCreate(&e) == cudaSuccess;
  if (!ok) {
    prof_release();
    return CSA_ERR_CUDA;
  }
  g_prof.max_launches = max_launches;
  g_prof.recorded = 0;
  g_prof.kernel_id = kernel_id;
  return CSA_OK;
}

CSA_API csa_status_t csa_prof_join(csa_stream_t stream) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.side) return CSA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // inside a capture, join only a side stream that this capture forked
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone, ss = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess ||
      cudaStreamIsCapturing(g_prof.side, &ss) != cudaSuccess)
    return CSA_ERR_CUDA;
  if ((cs == cudaStreamCaptureStatusActive) != (ss == cudaStreamCaptureStatusActive)) return CSA_OK;
  if (cudaEventRecord(g_prof.join, g_prof.side) != cudaSuccess ||
      cudaStreamWaitEvent(s, g_prof.join, 0) != cudaSuccess)
    return CSA_ERR_CUDA;
  return CSA_OK;
}

CSA_API csa_status_t csa_prof_read(int32_t kernel_id, float *total_ms, int32_t *n_launches) {
  if (!total_ms || !n_launches) return CSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  *total_ms = 0.f;
  *n_launches = 0;
  if (g_prof.kernel_id != kernel_id) return CSA_OK;
  float sum = 0.f;
  for (int i = 0; i < g_prof.recorded; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return CSA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return CSA_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *n_launches = g_prof.recorded;
  return CSA_OK;
}

CSA_API csa_status_t csa_prof_disable(void) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  prof_release();
  return CSA_OK;
}

}  // extern "C"
