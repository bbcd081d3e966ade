// csa_index_topk_noalloc: the indexer top-k for callers that cannot allocate
// device memory (see include/csa.h).  Its score scratch is a file-scope device
// array shared by every call on a device.
#include "csa_internal.cuh"

namespace {

constexpr size_t kMaxScores = CSA_NOALLOC_MAX_SCORES;

// Score scratch for calls that bring no workspace: kMaxScores FP32 entries
// (4 MiB), resident on every GPU that loads the library until the process
// exits.  Host code must not pass this symbol to a kernel: its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scores[kMaxScores];

// Device address of the scratch array in the current device's context.  The
// lookup runs on every call (a host-side table lookup once the module is
// loaded), so a context that was reset or replaced never gets a stale
// address.  Returns nullptr on failure.
float *scratch_for_current_device() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scores) != cudaSuccess || !p) return nullptr;
  return static_cast<float *>(p);
}

}  // namespace

using namespace csa;

extern "C" CSA_API csa_status_t csa_index_topk_noalloc(csa_index_args *user,
                                                        csa_stream_t stream) {
  if (!index_struct_ok(user)) return CSA_ERR_INVALID_ARG;
  csa_index_args A = full_index_args(user);
  const csa_index_args *a = &A;
  if (a->cand_out || a->cand_in) return CSA_ERR_UNSUPPORTED;
  {
    const csa_status_t st = index_normalize_strides(&A);
    if (st != CSA_OK) return st;
  }
  if (a->n_rows < 0 || a->n_req < 0) return CSA_ERR_INVALID_ARG;
  if (a->n_heads < 1 || a->n_heads > kMaxHeads || a->head_dim != kIdxDim)
    return CSA_ERR_UNSUPPORTED;
  if (a->topk < 1 || a->topk > CSA_MAX_TOPK || a->ratio < 1 || a->max_blocks <= 0)
    return CSA_ERR_INVALID_ARG;
  const long long n_cap = (long long)a->max_blocks * kBlock;
  // only the single-CTA top-k runs without further scratch (rows of at most
  // 8192 entries here); the scores must fit the static array
  if (n_cap > 8192 || topk_is_long((int)n_cap)) return CSA_ERR_UNSUPPORTED;
  const bool own_scores = a->scores != nullptr;
  if (own_scores && a->score_cols < n_cap) return CSA_ERR_INVALID_ARG;
  if (!own_scores && (long long)a->n_rows * n_cap > (long long)kMaxScores)
    return CSA_ERR_UNSUPPORTED;
  if (a->n_rows == 0) return CSA_OK;
  if (a->key_fmt != 0 && a->key_fmt != CSA_FMT_INT8 && a->key_fmt != CSA_FMT_FP4_E8M0 &&
      a->key_fmt != CSA_FMT_MXFP8)
    return CSA_ERR_UNSUPPORTED;
  if (!index_pointers_ok(a)) return CSA_ERR_INVALID_ARG;
  float *scores = a->scores;
  int cols = a->score_cols;
  if (!own_scores) {
    scores = scratch_for_current_device();
    if (!scores) return CSA_ERR_CUDA;
    cols = (int)n_cap;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // entries past a row's visible count are never read, so the scratch needs no
  // clearing between calls
  if (launch_index_scores(*a, scores, cols, nullptr, s) != cudaSuccess) return CSA_ERR_CUDA;
  return launch_index_topk(*a, scores, cols, nullptr, s) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
