// Per-row top-k kernel: one CTA, or one thread-block cluster, per row; the
// selection itself (and its description) is in topk_select.cuh.
#include <cooperative_groups.h>

#include <mutex>

#include "device_common.cuh"
#include "qsa_internal.h"
#include "sm100_ptx.cuh"
#include "topk_select.cuh"

namespace qsa {
namespace {

using namespace sel;

constexpr int kT = 512;  // threads per CTA
constexpr int kW = kT / 32;
// The narrow form: 256 threads and at most kNarrowSmem of shared memory, so
// that four CTAs (four rows) share an SM, for launches of many rows longer
// than the register path's 8192 columns.  A row's phases (sample, pass,
// candidate select) are latency-bound, so more rows in flight an SM pay
// more than more threads a row.
constexpr int kTn = 256;
constexpr int64_t kNarrowSmem = 55 * 1024;
// The register form: 1024 threads holding 8 keys each, one CTA an SM, for
// launches of at most two rows an SM whose rows are at most kTr * kRegKeysR
// columns (by the capacity, or by the caller's bound: the decode rows).  A
// row is one latency-bound chain on one SM (loads, digit histograms, scans,
// stores); twice the threads halve each thread's part of it (single-row
// decode top-k 5.78 -> 5.27 us against 512 threads of 16 keys).  Its
// registers are bounded as for two CTAs an SM (32 a thread, with a few
// spills that cost it nothing measurable), so that it leaves half the
// register file to a lean scoring CTA (256 threads of 128), while its shared
// memory (below) keeps a second top-k CTA off the SM: the scoring launch that follows a
// top-k then becomes resident on every SM while the top-k runs, instead of
// starting its CTAs on the top-k's SMs only after it ends, with their 2.7 us
// set-up exposed (decode step 16.6 -> 16.0 us).
constexpr int kTr = 1024;
constexpr int kRegKeysR = 8;
// Its shared memory: the three histograms need 20 KB, but the launch takes
// 116 KiB, so that two of its CTAs never share an SM (2 x (116 + 1 reserved)
// KiB > 228 KiB) while a lean scoring CTA of the decode shapes (106 KB) still
// fits beside one.  After a scoring form whose CTAs take whole SMs and leave
// one by one (fp8 keys with bf16 q), a 20 KB launch put two rows on the first
// SMs freed: a step of 16 rows of 8192 columns with 64 heads took 21.9 us,
// against 19.4 us at 116 KiB (decode step unchanged, 16.3 us; tiny MTP
// steps of 8 rows 8.85 -> 9.02 us).
constexpr size_t kRegFormSmem = 116 * 1024;
constexpr size_t kSmPerSm = 228 * 1024;  // shared memory of an SM
static_assert(2 * (kRegFormSmem + 1024) > kSmPerSm, "two register-form CTAs must not fit one SM");
static_assert(kRegFormSmem >= 4 * (size_t)kRegHistWords, "the register path's histograms fit");
constexpr int64_t kSmemMax = 226 * 1024;  // dynamic shared memory per CTA (static part aside)
constexpr int kRegKeys = 16;              // keys per thread of the register path (rows <= 8192)

struct TopkArgs {
  const float* logits;
  int64_t row_stride;
  const int32_t* visible;
  const int32_t* next_n_lens;  // live rows per request (dead rows select nothing), or null
  int64_t capacity;            // visible counts are clamped to [0, capacity]
  int32_t rows_per_req;
  int32_t* out;
  unsigned int* fault;
  int32_t k;
  int32_t cap;   // cached columns per CTA (multiple of 4, <= kCacheMax)
  int32_t cpw;   // candidate list entries per warp (multiple of 4)
  int32_t bulk;  // segments start 16-byte aligned: bulk copies fill the cache
  int32_t pcap;  // candidates of the sampled-pivot path (0: off)
};

template <bool CLUSTER, int NT>
__global__ void __launch_bounds__(NT, NT == kTn ? 4 : 2) topk_kernel(const TopkArgs a) {
  extern __shared__ uint4 dyn_topk[];
  __shared__ Shared sh;
  int CL = 1, rank = 0;  // cluster size and this CTA's rank in it
  if (CLUSTER) {
    cg::cluster_group cl = cg::this_cluster();
    CL = (int)cl.num_blocks();
    rank = (int)cl.block_rank();
  }
  const int64_t row = blockIdx.x / CL;
  // The row's visible count is read while the previous kernel may still run:
  // a kernel lets this one start early only after its own dependency wait, and
  // the scoring kernels that precede it never write the counts (the contract
  // of qsa_select_topk states it).  The logits are read after the wait.
  const int n = (int)row_visible(a.visible, a.next_n_lens, row, a.rows_per_req, a.capacity);
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const RowTask task{a.logits + row * a.row_stride, n, a.out + row * (int64_t)a.k};
  const Config cf{a.k, a.cap, a.cpw, a.bulk, a.fault, a.pcap};
  select_row<NT, CLUSTER, false, NT == kTr ? kRegKeysR : kRegKeys>(task, cf, reinterpret_cast<uint32_t*>(dyn_topk), sh,
                                                                   CL, rank);
}

}  // namespace

namespace {

// Shared-memory plan of one launch: the segment cache, per-warp candidate
// lists and the histograms.  One CTA a row aims at two CTAs per SM (lists of
// at least 64 entries a warp); when a whole row does not fit that budget it
// is cached whole at one CTA per SM, unless the rows outnumber the SMs
// (`waves`): then two CTAs an SM cache part of their rows (the rest is read
// back from L2) and the launch takes half the waves.  A cluster launch keeps
// one CTA per SM (its solo rows then never share an SM) and kCpwMax-entry
// lists.
struct TopkPlan {
  int64_t cap, cpw;
  size_t smem;
};

TopkPlan plan_for(int C, int64_t row_stride, bool waves = false) {
  int64_t per_cta = ((row_stride + C - 1) / C + 3) & ~int64_t(3);
  if (C > 1) {  // a solo row is cached whole
    const int64_t solo = ((row_stride < kSoloMax ? row_stride : kSoloMax) + 3) & ~int64_t(3);
    if (per_cta < solo) per_cta = solo;
  }
  int64_t cap = per_cta < kCacheMax ? per_cta : kCacheMax;
  const int64_t fixed = 4LL * (kBins + (C > 1 ? kAccWords : 0));
  int64_t cpw = kCpwMax;
  if (C == 1) {
    const int64_t two_per_sm = 110LL * 1024;
    if (waves && 4 * cap + fixed + 4LL * kW * 64 > two_per_sm) {
      cpw = 256;
      cap = ((two_per_sm - fixed - 4LL * kW * cpw) / 4) & ~int64_t(3);
      return TopkPlan{cap, cpw, (size_t)(4 * (cap + kW * cpw) + fixed)};
    }
    if (4 * cap + fixed + 4LL * kW * 64 <= two_per_sm) {
      cpw = ((two_per_sm - 4 * cap - fixed) / (4LL * kW)) & ~int64_t(3);
      if (cpw > kCpwMax) cpw = kCpwMax;
    }
  }
  const int64_t room = (kSmemMax - fixed - 4LL * kW * cpw) / 4;
  if (cap > room) cap = room & ~int64_t(3);
  size_t bytes = (size_t)(4 * (cap + kW * cpw) + fixed);
  const size_t reg = 4 * (size_t)(kRegHistWords + (C > 1 ? kAccWords : 0));  // keys in registers
  return TopkPlan{cap, cpw, bytes > reg ? bytes : reg};
}

// Clusters of c CTAs with `smem` bytes each that the device holds at once
// (queried once per device, cluster size and shared-memory size).
cudaError_t max_active_clusters(int c, size_t smem, int* out) {
  struct Entry {
    int dev, c;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].c == c && cache[i].smem == smem) {
      *out = cache[i].n;
      return cudaSuccess;
    }
  e = cudaFuncSetAttribute(topk_kernel<true, kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c, 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, topk_kernel<true, kT>, &cfg);
  if (e != cudaSuccess) return e;
  cache[used % 32] = Entry{dev, c, smem, n};
  if (used < 32) ++used;
  *out = n;
  return cudaSuccess;
}

// The register form (kTr threads, kRegKeysR keys each): the launch uses
// only the register path's three histograms, with no cache, candidate lists
// or pivot candidates.  A row longer than kTr * kRegKeysR columns (a caller's
// bound below its count) still selects exactly: the pivot is off (no
// candidates), so it takes candidate compaction, whose lists of 0 entries
// overflow at once, and which then reads its segment from global memory in
// every pass, its one histogram at the start of the allocation.
cudaError_t launch_register_form(const float* logits, int64_t num_rows, int64_t row_stride, const int32_t* visible,
                                 const int32_t* next_n_lens, int32_t rows_per_req, int64_t cap_cols, int32_t k,
                                 int32_t* out, unsigned int* fault, cudaStream_t stream) {
  TopkArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.visible = visible;
  a.next_n_lens = next_n_lens;
  a.capacity = cap_cols;
  a.rows_per_req = rows_per_req;
  a.out = out;
  a.fault = fault;
  a.k = k;
  a.cap = 0;
  a.cpw = 0;
  a.pcap = 0;
  a.bulk = 0;
  const size_t smem = kRegFormSmem;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<false, kTr>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_rows, 1, 1);
  cfg.blockDim = dim3(kTr, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_kernel<false, kTr>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride, const int32_t* visible,
                        const int32_t* next_n_lens, int32_t rows_per_req, int64_t capacity, int64_t max_visible,
                        int32_t k, int32_t* out, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  if (num_rows > 0x7FFFFFFFLL / kMaxCluster || row_stride > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  unsigned int* fault = nullptr;
  cudaError_t e = fault_word_address(&fault);
  if (e != cudaSuccess) return e;
  DeviceInfo dinfo;
  e = device_info(&dinfo);
  if (e != cudaSuccess) return e;
  // Rows of at most kTr * kRegKeysR columns (by the capacity, or by the
  // caller's bound), few enough that each has an SM to itself or shares it
  // with one other: the register form.
  const int64_t cap_cols = capacity < row_stride ? capacity : row_stride;  // visible counts are clamped to it
  const int64_t expect = max_visible > 0 && max_visible < cap_cols ? max_visible : cap_cols;
  if (expect <= (int64_t)kTr * kRegKeysR && num_rows <= 2 * (int64_t)dinfo.num_sms)
    return launch_register_form(logits, num_rows, row_stride, visible, next_n_lens, rows_per_req, cap_cols, k, out,
                                fault, stream);
  // Rows that may be longer than kSoloMax columns, and few enough that the
  // device holds all their clusters at once: split over the largest cluster.
  int C = 1;
  if (row_stride > kSoloMax)
    for (int c = kMaxCluster; c >= 2; c /= 2) {
      int fit = 0;
      e = max_active_clusters(c, plan_for(c, row_stride).smem, &fit);
      if (e != cudaSuccess) return e;
      if (num_rows <= fit) {
        C = c;
        break;
      }
    }
  // many rows, longer than the register path: the narrow form (its plan: the
  // histograms, 256-entry candidate lists, the rest a partial row cache)
  const bool narrow = C == 1 && row_stride > (int64_t)kT * kRegKeys && num_rows > 2 * (int64_t)dinfo.num_sms;
  const int nt = narrow ? kTn : kT;
  TopkPlan pl = plan_for(C, row_stride, num_rows > dinfo.num_sms);
  if (narrow) {
    const int64_t fixed = 4LL * kBins, cpw = 256;
    int64_t cap = ((kNarrowSmem - fixed - 4LL * (kTn / 32) * cpw) / 4) & ~int64_t(3);
    const int64_t per_row = (row_stride + 3) & ~int64_t(3);
    if (cap > per_row) cap = per_row;
    size_t bytes = (size_t)(4 * (cap + (kTn / 32) * cpw) + fixed);
    const size_t reg = 4 * (size_t)kRegHistWords;
    pl = TopkPlan{cap, cpw, bytes > reg ? bytes : reg};
  }
  TopkArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.visible = visible;
  a.next_n_lens = next_n_lens;
  a.capacity = capacity < row_stride ? capacity : row_stride;
  a.rows_per_req = rows_per_req;
  a.out = out;
  a.fault = fault;
  a.k = k;
  a.cap = (int32_t)pl.cap;
  a.cpw = (int32_t)pl.cpw;
  // the sampled-pivot path's candidates after its histograms: a column and a key each
  const int64_t pc = ((int64_t)pl.smem / 4 - kRegHistWords) / 2;
  a.pcap = (int32_t)((pc < (int64_t)nt * kRegKeys ? pc : (int64_t)nt * kRegKeys) & ~int64_t(3));
  // segment starts are multiples of 4 columns: 16-byte aligned when rows are
  a.bulk = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (row_stride & 3) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_rows * C), 1, 1);
  cfg.blockDim = dim3(nt, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 2 : 1;
  if (C > 1) {
    e = cudaFuncSetAttribute(topk_kernel<true, kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<true, kT>, a);
  } else if (narrow) {
    e = cudaFuncSetAttribute(topk_kernel<false, kTn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<false, kTn>, a);
  } else {
    e = cudaFuncSetAttribute(topk_kernel<false, kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<false, kT>, a);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
