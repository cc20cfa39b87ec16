// Page stream: the rate at which this GPU delivers a list of whole pages from
// HBM into shared memory, with no arithmetic on them - the achievable side of
// the paged scorers' roofline (their key bytes arrive the same way: one copy
// per page, pages in block-table order, scattered over the pool; tensor and
// plain bulk copies of these sizes stream at the same rate).
//
// One CTA per SM takes a contiguous share of the list.  Thread 0 streams the
// share through a ring of stages with plain bulk copies (cp.async.bulk, one
// per page), several pages a stage (at least 16 KB, as a scorer key tile
// holds); warp 1 consumes each stage - it XORs the stage's 32-bit words into
// a running value, so the bytes are really read - and releases it.  The
// CTAs' values are XORed into *checksum: the XOR of every 32-bit word of
// every listed page copy (a page listed twice cancels), which a test
// recomputes on the host bit for bit.  Every wait gives up after about a
// second and sets bit 2 of the device fault word.
//
// The launch mechanics are the lean scorer's: programmatic dependent launch
// (a launch's CTAs become resident, and set up their ring, while the kernel
// before them in the stream runs; they read the page list and copy only after
// it completes) and a 96 KB ring, so that two CTAs fit an SM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "qsa_internal.h"
#include "sm100_ptx.cuh"

namespace qsa {
namespace pstream {

constexpr int kMaxStages = 8;
constexpr int kStageSmem = 98304;      // ring bytes: two CTAs fit an SM, as the lean scorer's do
constexpr int kMinStageBytes = 16384;  // pages a stage: at least this many bytes of them
constexpr long long kSpin = 2000000000LL;

__global__ void __launch_bounds__(64, 1)
    page_stream_kernel(const uint8_t* base, int64_t page_stride, int32_t page_bytes, const int32_t* pages,
                       int64_t num_listed, int64_t pool_pages, int32_t stages, int32_t per_stage,
                       uint32_t* checksum, unsigned int* fault) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages];
  __shared__ volatile int abort_flag;
  const int64_t per = (num_listed + gridDim.x - 1) / gridDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * per;
  const int64_t i1 = i0 + per < num_listed ? i0 + per : num_listed;
  const int64_t nst = i1 > i0 ? (i1 - i0 + per_stage - 1) / per_stage : 0;  // stage fills of this CTA
  const int64_t stage_bytes = (int64_t)per_stage * page_bytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dep_wait();    // the page list and the pages are read after the kernel before
  ptx::grid_dep_launch();  // the next launch's CTAs may become resident now
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (abort_flag) return false;
      if (clock64() - t0 > kSpin) {
        abort_flag = 1;
        atomicOr(fault, 4u);
        return false;
      }
    }
    return true;
  };
  if (threadIdx.x == 0) {
    const uint64_t policy = ptx::policy_evict_first();
    // stages with copies issued, and the phase of each one's last fill, for
    // the drain after an abort
    uint32_t issued = 0, last_ph = 0;
    for (int64_t j = 0; j < nst; ++j) {
      const int s = (int)(j % stages);
      const uint32_t ph = (uint32_t)((j / stages) & 1);
      if (!wait(&empty[s], ph ^ 1u)) break;
      const int64_t a = i0 + j * per_stage, b = a + per_stage < i1 ? a + per_stage : i1;
      ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)((b - a) * page_bytes));
      for (int64_t i = a; i < b; ++i) {
        int64_t pg = pages[i];
        pg = pg < 0 ? 0 : (pg >= pool_pages ? pool_pages - 1 : pg);  // clamp: no fault
        ptx::bulk_load(ring + s * stage_bytes + (i - a) * page_bytes, base + pg * page_stride, (uint32_t)page_bytes,
                       &full[s], policy);
      }
      issued |= 1u << s;
      last_ph = (last_ph & ~(1u << s)) | (ph << s);
    }
    if (abort_flag)  // every issued copy lands before the CTA exits
      for (int s = 0; s < stages; ++s)
        if (issued & (1u << s)) {
          const long long t0 = clock64();
          while (!ptx::mbar_try_wait(&full[s], (last_ph >> s) & 1u) && clock64() - t0 < kSpin) {
          }
        }
  } else if (threadIdx.x >= 32) {
    const int lane = threadIdx.x & 31;
    uint32_t x = 0;
    for (int64_t j = 0; j < nst; ++j) {
      const int s = (int)(j % stages);
      const uint32_t ph = (uint32_t)((j / stages) & 1);
      if (!__all_sync(0xffffffffu, wait(&full[s], ph))) break;
      const int64_t a = i0 + j * per_stage, b = a + per_stage < i1 ? a + per_stage : i1;
      const uint4* w = reinterpret_cast<const uint4*>(ring + s * stage_bytes);
      const int64_t n16 = (b - a) * page_bytes / 16;
      for (int64_t k = lane; k < n16; k += 32) {
        const uint4 v = w[k];
        x ^= v.x ^ v.y ^ v.z ^ v.w;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0 && x != 0) atomicXor(checksum, x);
  }
}

}  // namespace pstream

cudaError_t launch_page_stream(const uint8_t* base, int64_t page_stride, int32_t page_bytes, const int32_t* pages,
                               int64_t num_listed, int64_t pool_pages, uint32_t* checksum, cudaStream_t stream) {
  unsigned int* fault = nullptr;
  cudaError_t e = fault_word_address(&fault);
  if (e != cudaSuccess) return e;
  // pages a stage: at least 16 KB of them (as a scorer key tile holds), and
  // as many stages of that as the ring takes, up to 8
  const int per_stage = page_bytes >= pstream::kMinStageBytes ? 1 : (pstream::kMinStageBytes + page_bytes - 1) / page_bytes;
  int stages = pstream::kStageSmem / (per_stage * page_bytes);
  stages = stages > pstream::kMaxStages ? pstream::kMaxStages : stages;
  const int smem = stages * per_stage * page_bytes;
  e = cudaFuncSetAttribute(pstream::page_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  DeviceInfo info;
  e = device_info(&info);
  if (e != cudaSuccess) return e;
  const int64_t want = (num_listed + 4 * per_stage - 1) / (4 * per_stage);  // at least 4 stage fills a CTA
  const int grid = (int)(want < info.num_sms ? (want < 1 ? 1 : want) : info.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(64, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pstream::page_stream_kernel, base, page_stride, page_bytes, pages, num_listed,
                            pool_pages, stages, per_stage, checksum, fault);
}

}  // namespace qsa
