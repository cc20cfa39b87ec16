// Per-row top-k selection over [0, visible) of a logits row.
//
// vLLM #62589 "Details": the decode top-k reads only [0, visible_blocks[row]);
// SGLang #48649: rows whose visible count fits in k select every column.
// Selection rule: the k columns first in (logit descending, column ascending);
// the set is written in ascending column order, -1 in unused slots.
//
// One CTA per row.  Logits map to order-preserving uint32 keys; the k-th
// largest key is found digit by digit (four 8-bit radix passes, each a
// shared-memory histogram over the candidates that still match the prefix),
// then one ordered pass over the row keeps every key above the threshold and
// the lowest-column keys equal to it, writing each kept column at its rank
// (block-wide ballot scans).  The row is cached in shared memory when it fits.
#include "device_common.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCachedKeys = 48 * 1024;  // 192 KB of shared memory

struct TopkArgs {
  const float* logits;
  int64_t num_rows, row_stride;
  const int32_t* visible;
  int32_t k;
  int32_t* out;
  int32_t cache_cap;  // keys the dynamic shared memory holds
};

struct TopkShared {
  uint32_t hist[256];
  int32_t warp_tot[kWarps];
  int32_t digit;
  int32_t above;  // candidates with a larger digit than `digit`
  int32_t equal;  // candidates with exactly `digit`
};

// Exclusive block-wide rank of `flag` in thread order, and the block total.
__device__ __forceinline__ int block_rank(bool flag, int32_t* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  int t = lane < kWarps ? warp_tot[lane] : 0;
  int incl = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  const int warp_excl = __shfl_sync(0xFFFFFFFFu, incl - t, warp);
  *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  __syncthreads();  // warp_tot is reused by the next call
  return warp_excl + in_warp;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys_s[];
  __shared__ TopkShared sh;
  const int64_t row = blockIdx.x;
  const int k = a.k;
  int32_t* o = a.out + row * (int64_t)k;
  const int64_t n = clamp64(a.visible[row], 0, a.row_stride);
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) o[i] = i < n ? i : -1;
    return;
  }
  const float* x = a.logits + row * a.row_stride;
  const bool cached = n <= a.cache_cap;
  if (cached)
    for (int64_t i = threadIdx.x; i < n; i += kThreads) keys_s[i] = topk_key(x[i]);
  auto key_at = [&](int64_t i) -> uint32_t { return cached ? keys_s[i] : topk_key(__ldg(x + i)); };

  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // how many of the still-matching candidates to keep
  int equal_total = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t kk = key_at(i);
      if ((kk & mask) == prefix) atomicAdd(&sh.hist[(kk >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending); find the digit where
      // the count of larger candidates first reaches `remaining`.
      const int lane = threadIdx.x;
      uint32_t c[8];
      uint32_t tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sh.hist[255 - (8 * lane + j)];
        tot += c[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      uint32_t run = incl - tot;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run < (uint32_t)remaining && run + c[j] >= (uint32_t)remaining) {
          sh.digit = 255 - (8 * lane + j);
          sh.above = (int)run;
          sh.equal = (int)c[j];
        }
        run += c[j];
      }
    }
    __syncthreads();
    const uint32_t digit = (uint32_t)sh.digit;
    remaining -= sh.above;
    equal_total = sh.equal;
    prefix |= digit << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  // prefix is the k-th largest key; `remaining` of the equal_total keys equal to
  // it are kept (lowest columns first), every larger key is kept.
  const uint32_t thr = prefix;
  const bool take_all_equal = remaining >= equal_total;
  int written = 0, equal_seen = 0;
  for (int64_t base = 0; base < n; base += kThreads) {
    const int64_t i = base + threadIdx.x;
    const uint32_t kk = i < n ? key_at(i) : 0u;
    const bool gt = i < n && kk > thr;
    const bool eq = i < n && kk == thr;
    bool sel;
    if (take_all_equal) {
      sel = gt || eq;
    } else {
      int eq_tot;
      const int eq_rank = block_rank(eq, sh.warp_tot, &eq_tot);
      sel = gt || (eq && equal_seen + eq_rank < remaining);
      equal_seen += eq_tot;
    }
    int sel_tot;
    const int rank = block_rank(sel, sh.warp_tot, &sel_tot);
    if (sel && written + rank < k) o[written + rank] = (int32_t)i;
    written += sel_tot;
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                        const int32_t* visible, int32_t k, int32_t* out, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  TopkArgs a{logits, num_rows, row_stride, visible, k, out, 0};
  int64_t cap = row_stride < kMaxCachedKeys ? row_stride : kMaxCachedKeys;
  a.cache_cap = (int32_t)cap;
  const size_t smem = sizeof(uint32_t) * (size_t)cap;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (num_rows > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  topk_kernel<<<(unsigned)num_rows, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qsa
