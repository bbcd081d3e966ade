// Low-bit caches for the prefill attention ("DeepSeek V4.1 Flash", production
// cache ABI: FP4 compressed KV with E4M3 scales per 16 channels, MXFP8 window
// KV with E8M0 scales per 32): every mapped page of the requests' block
// tables is dequantised once into a BF16 arena in the caller's workspace,
// indexed by (request, logical page), with a block table of its own.  A
// prefill tile of 128 query rows reads each compressed row up to 128 times and
// a chunk reads it from every tile, so converting once per call costs less than
// converting in every tile's gather.  Dequantisation is exact (every value of
// these formats is a BF16 value).
#include "csa_internal.cuh"
#include "lowbit.cuh"
#include "tc.cuh"

namespace csa {
namespace {

constexpr int DQ_THREADS = 256;

// One CTA per (request, logical page): the page's 128 rows, 16 threads per
// row, each thread 32 channels (one slab) of 8 rows.  fmt: CSA_FMT_FP4_E4M3
// (codes: 256 bytes per row, scales: 32) or CSA_FMT_MXFP8 (512 + 16).
__global__ void __launch_bounds__(DQ_THREADS)
    dequant_pages_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales,
                         const int32_t *__restrict__ table, int max_blocks, int n_blocks,
                         int fmt, __nv_bfloat16 *__restrict__ arena, int32_t *__restrict__ arena_table,
                         uint32_t *status) {
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  const int page = blockIdx.x;  // b * max_blocks + j
  const int phys = table[page];
  if (threadIdx.x == 0) arena_table[page] = phys >= 0 && phys < n_blocks ? page : -1;
  if (phys < 0 || phys >= n_blocks) return;  // the attention flags a read of it
  const bool fp4 = fmt == CSA_FMT_FP4_E4M3;
  const int row_bytes = fp4 ? kHeadDim / 2 : kHeadDim;
  const int groups = fp4 ? kHeadDim / 16 : kHeadDim / 32;
  const int slab = threadIdx.x & 15;
  for (int r = threadIdx.x >> 4; r < kBlock; r += DQ_THREADS / 16) {
    const long long src_row = (long long)phys * kBlock + r;
    const uint8_t *c = codes + src_row * row_bytes;
    const uint8_t *sc = scales + src_row * groups;
    uint4 *dst = reinterpret_cast<uint4 *>(arena + ((long long)page * kBlock + r) * kHeadDim +
                                           slab * 32);
    if (fp4) {
      const uint4 w = *reinterpret_cast<const uint4 *>(c + slab * 16);
      const uint32_t s2 = *reinterpret_cast<const uint16_t *>(sc + slab * 2);
      dst[0] = lowbit::e2m1x8_e4m3_to_bf16x8(w.x, s2 & 0xFFu);
      dst[1] = lowbit::e2m1x8_e4m3_to_bf16x8(w.y, s2 & 0xFFu);
      dst[2] = lowbit::e2m1x8_e4m3_to_bf16x8(w.z, s2 >> 8);
      dst[3] = lowbit::e2m1x8_e4m3_to_bf16x8(w.w, s2 >> 8);
    } else {
      const uint4 w0 = *reinterpret_cast<const uint4 *>(c + slab * 32);
      const uint4 w1 = *reinterpret_cast<const uint4 *>(c + slab * 32 + 16);
      const float e8 = lowbit::pow2f((int)sc[slab] - 127);
      dst[0] = lowbit::e4m3x8_e8m0_to_bf16x8(make_uint2(w0.x, w0.y), e8);
      dst[1] = lowbit::e4m3x8_e8m0_to_bf16x8(make_uint2(w0.z, w0.w), e8);
      dst[2] = lowbit::e4m3x8_e8m0_to_bf16x8(make_uint2(w1.x, w1.y), e8);
      dst[3] = lowbit::e4m3x8_e8m0_to_bf16x8(make_uint2(w1.z, w1.w), e8);
    }
  }
}

size_t arena_bytes(int n_req, int max_blocks) {
  return align_up((size_t)n_req * max_blocks * kBlock * kHeadDim * 2, 256) +
         align_up((size_t)n_req * max_blocks * 4, 256);
}

}  // namespace

size_t attn_arena_bytes(const csa_attn_args &a) {
  size_t n = 0;
  if (a.cmp_fmt == CSA_FMT_FP4_E4M3) n += arena_bytes(a.n_req, a.cmp_max_blocks);
  if (a.kv_fmt == CSA_FMT_MXFP8) n += arena_bytes(a.n_req, a.kv_max_blocks);
  return n;
}

cudaError_t launch_dequant_arena(const csa_attn_args &a, void *ws, csa_attn_args *bf,
                                 cudaStream_t s) {
  *bf = a;
  uint8_t *p = static_cast<uint8_t *>(ws);
  for (int k = 0; k < 2; ++k) {
    const bool cmp = k == 0;
    if (cmp ? a.cmp_fmt != CSA_FMT_FP4_E4M3 : a.kv_fmt != CSA_FMT_MXFP8) continue;
    const int mb = cmp ? a.cmp_max_blocks : a.kv_max_blocks;
    const size_t pages = (size_t)a.n_req * mb;
    __nv_bfloat16 *arena = reinterpret_cast<__nv_bfloat16 *>(p);
    int32_t *table = reinterpret_cast<int32_t *>(p + align_up(pages * kBlock * kHeadDim * 2, 256));
    p += arena_bytes(a.n_req, mb);
    launch_begin(CSA_K_DEQUANT, s);
    const cudaError_t e = launch_kernel(
        dequant_pages_kernel, dim3((unsigned)pages), dim3(DQ_THREADS), 0, s, 0, false,
        static_cast<const uint8_t *>(cmp ? a.cmp_pool : a.kv_pool),
        cmp ? a.cmp_scale_pool : a.kv_scale_pool, cmp ? a.cmp_block_table : a.kv_block_table, mb,
        cmp ? a.cmp_n_blocks : a.kv_n_blocks, cmp ? a.cmp_fmt : a.kv_fmt, arena, table,
        a.status_dev);
    launch_end(CSA_K_DEQUANT, s);
    if (e != cudaSuccess) return e;
    if (cmp) {
      bf->cmp_pool = arena;
      bf->cmp_row_stride = 2 * kHeadDim;
      bf->cmp_page_stride = (long long)kBlock * 2 * kHeadDim;
      bf->cmp_block_table = table;
      bf->cmp_n_blocks = (int)pages;
      bf->cmp_fmt = CSA_FMT_BF16;
      bf->cmp_scale_pool = nullptr;
    } else {
      bf->kv_pool = arena;
      bf->kv_row_stride = 2 * kHeadDim;
      bf->kv_page_stride = (long long)kBlock * 2 * kHeadDim;
      bf->kv_block_table = table;
      bf->kv_n_blocks = (int)pages;
      bf->kv_fmt = CSA_FMT_BF16;
      bf->kv_scale_pool = nullptr;
    }
  }
  return cudaGetLastError();
}

}  // namespace csa
