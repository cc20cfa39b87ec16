// Per-row top-k selection over [0, visible) of a logits row.
//
// vLLM #62589 "Details": the decode top-k reads only [0, visible_blocks[row]);
// SGLang #48649: rows whose visible count fits in k select every column.
// Selection rule: the k columns first in (logit descending, column ascending);
// the set is written in ascending column order, -1 in unused slots.
//
// One CTA per row.  Logits map to order-preserving uint32 keys, cached in
// shared memory in column order when the row fits (else re-read from global
// memory each pass).  The k-th largest key is found digit by digit, most
// significant first (12, 10 and 10 bits), each digit from a shared-memory
// histogram over the keys that still match the prefix.  The first digit (sign,
// exponent and 3 fraction bits) spreads logits of similar magnitude over many
// bins, so plain shared-memory atomics see little contention.  A last ordered
// pass keeps every key above the threshold and the lowest-column keys equal
// to it, each written at its rank.  Every pass handles 4 consecutive columns
// per thread (one 16-byte shared-memory access), so a CTA step covers
// 4 * 512 columns and the ordered pass needs one block prefix sum per step.
#include "device_common.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStep = 4 * kThreads;          // columns per CTA step
constexpr int kMaxCachedKeys = 48 * 1024;    // 192 KB of keys
constexpr int kBins = 4096;

struct TopkArgs {
  const float* logits;
  int64_t num_rows, row_stride;
  const int32_t* visible;
  int32_t k;
  int32_t* out;
  int32_t cache_cap;  // keys the dynamic shared memory caches (multiple of 4)
};

struct TopkShared {
  uint32_t hist[kBins];
  int32_t warp_tot[kWarps];
  int32_t digit, above, equal;
};

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// Exclusive block-wide prefix of a per-thread count, and the block total.
__device__ __forceinline__ int block_excl_sum(int v, int32_t* warp_tot, int* total) {
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  const int t = lane < kWarps ? warp_tot[lane] : 0;
  int wincl = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
    if (lane >= o) wincl += u;
  }
  const int warp_excl = __shfl_sync(0xFFFFFFFFu, wincl - t, warp);
  *total = __shfl_sync(0xFFFFFFFFu, wincl, 31);
  __syncthreads();  // warp_tot is reused by the next call
  return warp_excl + incl - v;
}

// All threads: the digit whose bin holds the `remaining`-th largest
// candidate.  Thread t owns bins/kThreads consecutive bins in descending
// order; a block prefix sum of their totals locates the bin.  Writes
// sh.digit / sh.above / sh.equal; the caller synchronises before reading.
__device__ __forceinline__ void find_digit(TopkShared& sh, int bins, int remaining) {
  const int per = bins / kThreads;
  const int top = bins - 1 - (int)threadIdx.x * per;
  int tot = 0;
  for (int j = 0; j < per; ++j) tot += (int)sh.hist[top - j];
  int block_tot;
  int run = block_excl_sum(tot, sh.warp_tot, &block_tot);
  if (run < remaining && run + tot >= remaining) {
    for (int j = 0; j < per; ++j) {
      const int c = (int)sh.hist[top - j];
      if (run + c >= remaining) {
        sh.digit = top - j;
        sh.above = run;
        sh.equal = c;
        break;
      }
      run += c;
    }
  }
}

// Keys of columns c .. c+3 (c a multiple of 4): from the shared-memory cache,
// or from global memory (16-byte load when aligned).  Columns >= n give 0.
struct RowKeys {
  const float* x;
  const uint32_t* cache;  // null: read global memory
  int n;
  bool vec;

  __device__ __forceinline__ uint4 get4(int c) const {
    if (cache != nullptr && c + 4 <= n) return *reinterpret_cast<const uint4*>(cache + c);
    uint4 r;
    if (cache == nullptr && vec && c + 4 <= n) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(x + c));
      r.x = topk_key(f.x);
      r.y = topk_key(f.y);
      r.z = topk_key(f.z);
      r.w = topk_key(f.w);
      return r;
    }
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = c + u < n ? (cache != nullptr ? cache[c + u] : topk_key(__ldg(x + c + u))) : 0u;
    r.x = v[0];
    r.y = v[1];
    r.z = v[2];
    r.w = v[3];
    return r;
  }
};

__device__ __forceinline__ uint32_t lane_of(const uint4& v, int u) {
  return u == 0 ? v.x : (u == 1 ? v.y : (u == 2 ? v.z : v.w));
}

__global__ void __launch_bounds__(kThreads, 2) topk_kernel(const TopkArgs a) {
  extern __shared__ uint4 dyn4[];
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(dyn4);
  __shared__ TopkShared sh;
  const int64_t row = blockIdx.x;
  const int k = a.k;
  int32_t* o = a.out + row * (int64_t)k;
  const int n = (int)clamp64(a.visible[row], 0, a.row_stride);
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) o[i] = i < n ? i : -1;
    return;
  }
  const float* x = a.logits + row * a.row_stride;
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  RowKeys rk{x, nullptr, n, vec};
  if (n <= a.cache_cap) {
    // cache the row's keys: 16-byte loads, two steps in flight per thread
    for (int base = 0; base < n; base += 2 * kStep) {
      const int c0 = base + 4 * threadIdx.x, c1 = c0 + kStep;
      const uint4 k0 = rk.get4(c0);
      const uint4 k1 = rk.get4(c1);
      if (c0 < n) *reinterpret_cast<uint4*>(keys_s + c0) = k0;
      if (c1 < n) *reinterpret_cast<uint4*>(keys_s + c1) = k1;
    }
    rk.cache = keys_s;
  }

  uint32_t prefix = 0, mask = 0;
  int remaining = k, equal_total = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int bins = pass == 0 ? 4096 : 1024;
    for (int i = threadIdx.x; i < bins; i += kThreads) sh.hist[i] = 0;
    __syncthreads();  // also orders the cache fill before the first read
#pragma unroll 1
    for (int base = 0; base < n; base += kStep) {
      const int c = base + 4 * threadIdx.x;
      const uint4 kk = rk.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t key = lane_of(kk, u);
        if (c + u < n && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & (uint32_t)(bins - 1)], 1u);
      }
    }
    __syncthreads();
    find_digit(sh, bins, remaining);
    __syncthreads();
    remaining -= sh.above;
    equal_total = sh.equal;
    prefix |= (uint32_t)sh.digit << shift;
    mask |= (uint32_t)(bins - 1) << shift;
    __syncthreads();  // sh.* is rewritten by the next pass
  }

  // prefix is the k-th largest key; `remaining` of the equal_total keys equal to
  // it are kept (lowest columns first), every larger key is kept.
  const uint32_t thr = prefix;
  const bool take_all_equal = remaining >= equal_total;
  int written = 0, equal_seen = 0;
#pragma unroll 1
  for (int base = 0; base < n; base += kStep) {
    const int c = base + 4 * threadIdx.x;
    const uint4 kk = rk.get4(c);
    int neq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) neq += (c + u < n && lane_of(kk, u) == thr);
    int eqs = equal_seen;
    if (!take_all_equal) {
      int tot;
      eqs += block_excl_sum(neq, sh.warp_tot, &tot);
      equal_seen += tot;
    }
    bool sel[4];
    int nsel = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t key = lane_of(kk, u);
      const bool ok = c + u < n;
      const bool eq = ok && key == thr;
      sel[u] = ok && (key > thr || (eq && (take_all_equal || eqs < remaining)));
      eqs += eq;
      nsel += sel[u];
    }
    int tot;
    int pos = written + block_excl_sum(nsel, sh.warp_tot, &tot);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sel[u]) {
        if (pos < k) o[pos] = c + u;
        ++pos;
      }
    written += tot;
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                        const int32_t* visible, int32_t k, int32_t* out, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  if (num_rows > 0x7FFFFFFFLL || row_stride > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  TopkArgs a{logits, num_rows, row_stride, visible, k, out, 0};
  int64_t cap = row_stride < kMaxCachedKeys ? row_stride : kMaxCachedKeys;
  cap = (cap + 3) & ~int64_t(3);
  a.cache_cap = (int32_t)cap;
  const size_t smem = sizeof(uint32_t) * (size_t)cap;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<(unsigned)num_rows, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qsa
