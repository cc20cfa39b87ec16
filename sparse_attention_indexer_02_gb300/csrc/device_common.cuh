// Device helpers shared by the scoring and top-k kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

// bf16 pair packed in a 32-bit word -> two fp32 values (exact: bf16 is the top
// half of a binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ReLU that keeps NaN (a poisoned key stays visible), like torch.relu.
__device__ __forceinline__ float relu_keep_nan(float x) { return x < 0.0f ? 0.0f : x; }

// max(x, 0) in one instruction that returns NaN for a NaN input (max.NaN),
// so a poisoned key is not hidden by the ReLU.
__device__ __forceinline__ float relu_nan(float x) {
  float r;
  asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(x));
  return r;
}

// Order-preserving map of fp32 to uint32 for a descending top-k: a larger
// float gives a larger key; -0.0 is folded onto +0.0 first.
__device__ __forceinline__ uint32_t topk_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

// Visible count of row r with the live-row rule of the ragged call: row i of
// request b sees no column when i >= next_n_lens[b] (clamped to the rows of a
// request); next_n_lens null means every row is live.
__device__ __forceinline__ int64_t row_visible(const int32_t* visible, const int32_t* next_n_lens, int64_t r,
                                               int rows_per_req, int64_t capacity) {
  int64_t v = clamp64(visible[r], 0, capacity);
  if (next_n_lens != nullptr) {
    const int64_t b = r / rows_per_req;
    if (r - b * rows_per_req >= clamp64(next_n_lens[b], 0, rows_per_req)) v = 0;
  }
  return v;
}

// 16-byte read-only global load that bypasses L1 allocation (streamed keys).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace qsa
