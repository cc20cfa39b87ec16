// tcgen05 scorer, host side: shape support, tensor maps, layout and launch.
// The kernel (and its design notes) is in umma_kernel.cuh; its instantiations
// are compiled in umma_bf16.cu and umma_fp8.cu.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "qsa_internal.h"
#include "sm100_ptx.cuh"
#include "umma_kernel.cuh"

namespace qsa {
namespace umma {

__device__ unsigned int g_fault_word = 0;

namespace {


PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int pick_n(int rows_per_group, int heads) {
  const int need = rows_per_group * heads;
  for (int n : {16, 32, 64, 128, 192, 256})
    if (need <= n) return n;
  return 0;
}

// Rows a group stacks into the MMA's N (rows x heads <= 256).  A request
// with more rows than fit takes groups of 192 / H rows: N = 192 is one batch
// of four units per epilogue warp, three warps a TMEM lane quadrant, where
// N = 256 gives the quadrant's warps 6, 5 and 5 units (prefill scoring 480 ->
// 411 us).
void group_shape(const qsa_paged_desc& d, int* G_rows, int* N) {
  const bool many = (int64_t)d.rows_per_req * d.num_heads > 256;
  int g = (many ? 192 : 256) / d.num_heads;
  if (g < 1) g = 1;
  if (g > d.rows_per_req) g = d.rows_per_req;
  *G_rows = g;
  *N = pick_n(g, d.num_heads);
}

}  // namespace
}  // namespace umma

// Device address of g_fault_word on the current device (looked up once per device).
cudaError_t fault_word_address(unsigned int** out) {
  static std::mutex mu;
  static unsigned int* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && addr[dev]) {
    *out = addr[dev];
    return cudaSuccess;
  }
  void* a = nullptr;
  e = cudaGetSymbolAddress(&a, umma::g_fault_word);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) addr[dev] = static_cast<unsigned int*>(a);
  *out = static_cast<unsigned int*>(a);
  return cudaSuccess;
}

using namespace umma;

bool umma_supports(const qsa_paged_desc& d, const char** why) {
  const int pc = d.page_cols;
  if (pc % 8 != 0 || !(kBM % pc == 0 || pc % kBM == 0)) {
    *why = "page_cols must be a multiple of 8 that divides 128 or is a multiple of 128";
    return false;
  }
  if (d.kv_dtype == QSA_KV_FP8_E4M3 && d.scale_page_stride % 16 != 0) {
    *why = "fp8 scale_page_stride must be a multiple of 16 bytes for the bulk copies";
    return false;
  }
  if (d.out_cols > (int64_t)0x7FFFFF00LL) {
    *why = "out_cols too large for the tile index";
    return false;
  }
  int Gr, N;
  group_shape(d, &Gr, &N);
  if (N == 0) {
    *why = "rows x heads of a group exceed 256";
    return false;
  }
  const int64_t groups = (int64_t)d.num_requests * ((d.rows_per_req + Gr - 1) / Gr);
  if (groups > (1 << 20) || make_layout(N, (int)groups, d.kv_dtype == QSA_KV_FP8_E4M3).stages < 2) {
    *why = "too many row groups for the on-chip schedule";
    return false;
  }
  switch (d.num_heads) {
    case 1: case 2: case 4: case 8: case 16: case 32: case 64: break;
    default:
      *why = "the tcgen05 epilogue is built for 1, 2, 4, ..., 64 heads";
      return false;
  }
  const int64_t qrows = (int64_t)d.num_requests * d.rows_per_req * d.num_heads;
  if (qrows > 0x7FFFFFFFLL) {
    *why = "too many q rows for the tensor map";
    return false;
  }
  return true;
}

bool umma_lean_supports(const qsa_paged_desc& d, bool q8, const char** why) {
  if (!umma_supports(d, why)) return false;
  if (d.kv_dtype == QSA_KV_FP8_E4M3 && !q8) {
    *why = "the lean form has no fp8 -> bf16 converter (fp8 keys need fp8 q)";
    return false;
  }
  if ((int64_t)d.num_requests * d.rows_per_req > kFastSchedRows) {
    *why = "the lean form serves at most 256 rows";
    return false;
  }
  int Gr, N;
  group_shape(d, &Gr, &N);
  const int64_t groups = (int64_t)d.num_requests * ((d.rows_per_req + Gr - 1) / Gr);
  if (N > kLeanMaxN) {
    *why = "the lean form serves groups of at most 64 rows x heads";
    return false;
  }
  const int kind = d.kv_dtype == QSA_KV_FP8_E4M3 ? kKindFp8Q : kKindBf16;
  if (make_layout(N, (int)groups, kind, false, true).stages < 3) {
    *why = "the lean form's shared memory holds fewer than three key stages";
    return false;
  }
  return true;
}

int64_t umma_num_groups(const qsa_paged_desc& d) {
  int Gr, N;
  group_shape(d, &Gr, &N);
  return (int64_t)d.num_requests * ((d.rows_per_req + Gr - 1) / Gr);
}

cudaError_t launch_umma(const ScoreParams& p, cudaStream_t stream, const char** msg, const FuseArgs* fuse,
                        bool lean) {
  if (p.num_rows == 0 || p.out_cols == 0) return cudaSuccess;
  qsa_paged_desc d{};
  d.num_requests = p.num_requests;
  d.rows_per_req = p.rows_per_req;
  d.num_heads = p.num_heads;
  d.head_dim = 128;
  d.page_cols = p.page_cols;
  d.kv_dtype = p.fp8 ? QSA_KV_FP8_E4M3 : QSA_KV_BF16;
  d.out_cols = p.out_cols;
  d.key_page_stride = p.key_page_stride;
  d.scale_page_stride = p.scale_page_stride;
  if (!umma_supports(d, msg)) return cudaErrorInvalidValue;
  if (lean && (fuse != nullptr || !umma_lean_supports(d, p.q8 != 0, msg))) {
    if (fuse != nullptr) *msg = "the lean form has no fused selection";
    return cudaErrorInvalidValue;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) {
    *msg = "cuTensorMapEncodeTiled is unavailable from the driver";
    return cudaErrorInvalidValue;
  }
  int Gr, N;
  group_shape(d, &Gr, &N);
  unsigned int* fault = nullptr;
  cudaError_t e0 = fault_word_address(&fault);
  if (e0 != cudaSuccess) return e0;
  UmmaParams up;
  up.fault = fault;
  up.scales = p.scales;
  up.scale_stride = p.scale_page_stride;
  up.weights = p.weights;
  up.q = p.q;
  up.block_table = p.block_table;
  up.visible = p.visible;
  up.next_n_lens = p.next_n_lens;
  up.out = p.out;
  up.out_cols = p.out_cols;
  up.capacity = p.capacity;
  up.num_rows = p.num_rows;
  up.rows_per_req = p.rows_per_req;
  up.num_heads = p.num_heads;
  up.page_cols = p.page_cols;
  up.max_pages = p.max_pages;
  up.num_pages = p.num_pages;
  up.group_rows = Gr;
  up.groups_per_req = (p.rows_per_req + Gr - 1) / Gr;
  up.num_groups = p.num_requests * up.groups_per_req;
  up.tiles_cap = (int32_t)((p.out_cols + kBM - 1) / kBM);
  up.box_rows = p.page_cols < kBM ? p.page_cols : kBM;
  up.bpt_shift = 0;
  while (p.page_cols < kBM && (p.page_cols << up.bpt_shift) < kBM) ++up.bpt_shift;
  up.pc_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == p.page_cols) up.pc_shift = sh;
  up.stream_out = (int64_t)p.num_rows * p.out_cols * 4 > (64LL << 20) ? 1 : 0;
  up.keep_keys = up.groups_per_req > 1 ? 1 : 0;

  CUtensorMap kv_map, q_map;
  CUresult r;
  if (p.fp8) {
    // fp8: one 128-byte row (all of D) per key; a box is a page's (or a
    // 128-key slice of a page's) rows
    cuuint64_t dims[3] = {128, (cuuint64_t)p.page_cols, (cuuint64_t)p.num_pages};
    cuuint64_t strides[2] = {128, (cuuint64_t)p.key_page_stride};
    cuuint32_t box[3] = {128, (cuuint32_t)up.box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    r = enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(p.kv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // bf16: a key row is two 64-element (128-byte) K-halves.  Dimensions,
    // innermost first: element of the half, key within its group of 8, half,
    // group of 8 within the page, page.  One box of a page's rows then lands
    // as, per group of 8 keys, K-half 0 (a 1 KB swizzle atom) then K-half 1 -
    // a whole page in one copy.
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)(p.page_cols / 8), (cuuint64_t)p.num_pages};
    cuuint64_t strides[4] = {256, 128, 8 * 256, (cuuint64_t)p.key_page_stride};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)(up.box_rows / 8), 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    r = enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<uint8_t*>(p.kv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    *msg = "key-cache tensor map rejected by the driver";
    return cudaErrorInvalidValue;
  }
  {
    // bf16 q: 64-element (128-byte) K-halves; fp8 q: one 128-byte row of D codes
    cuuint64_t dims[2] = {128, (cuuint64_t)p.num_rows * (cuuint64_t)p.num_heads};
    cuuint64_t strides[1] = {(cuuint64_t)(p.q8 ? 128 : 256)};
    cuuint32_t box[2] = {(cuuint32_t)(p.q8 ? 128 : 64), (cuuint32_t)N};
    cuuint32_t es[2] = {1, 1};
    r = enc(&q_map, p.q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<uint16_t*>(p.q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "q tensor map rejected by the driver";
      return cudaErrorInvalidValue;
    }
  }
  DeviceInfo info;
  cudaError_t e = device_info(&info);
  if (e != cudaSuccess) return e;
  const int64_t upper = (int64_t)up.num_groups * up.tiles_cap;
  const int grid = (int)(upper < info.num_sms ? (upper < 1 ? 1 : upper) : info.num_sms);
  const int kind = !p.fp8 ? kKindBf16 : (p.q8 ? kKindFp8Q : kKindFp8Keys);
  const Layout L = make_layout(N, up.num_groups, kind, fuse != nullptr, lean);
  up.topk_out = nullptr;
  up.fuse_sync = nullptr;
  up.topk_k = up.topk_cap = up.topk_cpw = up.topk_pcap = 0;
  if (fuse) {
    if (up.num_groups > kFuseMaxGroups) {
      *msg = "too many row groups for the fused selection";
      return cudaErrorInvalidValue;
    }
    // the selection runs on 512 threads (256 with the converter warps) in the
    // stage area, idle once the CTA's tiles are scored: per-warp candidate
    // lists, the histogram and as much of a row as fits cached
    const int nt = kind == kKindFp8Keys ? 256 : 512;
    const int cpw = sel::kCpwMax;
    const int64_t room = ((int64_t)L.bar_off - kSelSharedBytes) / 4 - (int64_t)(nt / 32) * cpw - sel::kBins;
    const int64_t cap = (room < sel::kCacheMax ? room : sel::kCacheMax) & ~int64_t(3);
    if (cap < 4) {
      *msg = "no shared memory left for the fused selection";
      return cudaErrorInvalidValue;
    }
    up.topk_out = fuse->topk_out;
    up.fuse_sync = fuse->sync;
    up.topk_k = fuse->k;
    up.topk_cap = (int32_t)cap;
    up.topk_cpw = cpw;
    // the sampled-pivot path's candidates after its histograms: a column and a key each
    const int64_t pc = (((int64_t)L.bar_off - kSelSharedBytes) / 4 - sel::kRegHistWords) / 2;
    const int64_t pmax = (int64_t)nt * kFuseKeys;
    up.topk_pcap = (int32_t)((pc < pmax ? pc : pmax) & ~int64_t(3));
    if (kind == kKindFp8Q) return launch_q8_topk(p.num_heads, kv_map, q_map, up, L, grid, stream);
    return p.fp8 ? launch_fp8_topk(p.num_heads, kv_map, q_map, up, L, grid, stream)
                 : launch_bf16_topk(p.num_heads, kv_map, q_map, up, L, grid, stream);
  }
  if (lean) return launch_lean(p.num_heads, kind, kv_map, q_map, up, L, grid, stream);
  if (kind == kKindFp8Q) return launch_q8(p.num_heads, kv_map, q_map, up, L, grid, stream);
  return p.fp8 ? launch_fp8(p.num_heads, kv_map, q_map, up, L, grid, stream)
               : launch_bf16(p.num_heads, kv_map, q_map, up, L, grid, stream);
}

cudaError_t read_fault_word(uint32_t* flags, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof v);
  if (e != cudaSuccess) return e;
  *flags = v;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_fault_word, &z, sizeof z);
  }
  return e;
}

}  // namespace qsa
