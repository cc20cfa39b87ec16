// Per-row top-k selection over [0, visible) of a logits row.
//
// vLLM #62589 "Details": the decode top-k reads only [0, visible_blocks[row]);
// SGLang #48649: rows whose visible count fits in k select every column.
// Selection rule: the k columns first in (logit descending, column ascending);
// the set is written in ascending column order, -1 in unused slots.
//
// Rows are handled by one CTA each (many rows), or - when there are few rows
// for the GPU - by a thread-block cluster of 2, 4 or 8 CTAs each owning a
// contiguous segment of the row (topk_cluster_kernel, below).
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
#include <cooperative_groups.h>

#include "device_common.cuh"
#include "qsa_internal.h"

namespace cg = cooperative_groups;

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

// ---------------------------------------------------------------------------
// Cluster variant: a row split over the C CTAs of a cluster.  Each CTA caches
// and histograms its own segment; per digit the C histograms are
// reduce-scattered through distributed shared memory (CTA q sums bin range q
// over all CTAs), the range totals are exchanged, and the CTA whose range holds
// the threshold finds the digit and broadcasts it.  For the output each CTA
// publishes its counts of keys above / equal to the threshold; a CTA's
// selected columns start after those of the segments before it (equal keys:
// lowest columns first across the whole row).
// ---------------------------------------------------------------------------

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCStep = 4 * kCThreads;
constexpr int kMaxCluster = 8;

struct ClusterShared {
  uint32_t hist[kBins];        // this CTA's histogram of its segment
  uint32_t sum[kBins / 2];     // summed counts of this CTA's bin range (<= kBins / 2 bins)
  int32_t warp_tot[kCWarps];
  int32_t range_tot[kMaxCluster];  // written by every CTA of the cluster
  int32_t res[3];                  // digit, above, equal - written by the owning CTA
  int32_t cnt_gt[kMaxCluster], cnt_eq[kMaxCluster];
};

__device__ __forceinline__ int cblock_excl_sum(int v, int32_t* warp_tot, int* total) {
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  const int t = lane < kCWarps ? warp_tot[lane] : 0;
  int wincl = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
    if (lane >= o) wincl += u;
  }
  const int warp_excl = __shfl_sync(0xFFFFFFFFu, wincl - t, warp);
  *total = __shfl_sync(0xFFFFFFFFu, wincl, 31);
  __syncthreads();
  return warp_excl + incl - v;
}

__global__ void __launch_bounds__(kCThreads) topk_cluster_kernel(const TopkArgs a) {
  extern __shared__ uint4 dyn4c[];
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(dyn4c);
  __shared__ ClusterShared sh;
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int part = (int)cl.block_rank();
  const int64_t row = blockIdx.x / C;
  const int k = a.k;
  int32_t* o = a.out + row * (int64_t)k;
  const int n = (int)clamp64(a.visible[row], 0, a.row_stride);
  if (n <= k) {  // the same for every CTA of the cluster: no cluster barrier is pending
    if (part == 0)
      for (int i = threadIdx.x; i < k; i += kCThreads) o[i] = i < n ? i : -1;
    return;
  }
  // segment [s0, s1) of the row, boundaries on multiples of 4 columns
  const int s0 = part == 0 ? 0 : min(n, (int)(((int64_t)n * part / C + 3) & ~int64_t(3)));
  const int s1 = part == C - 1 ? n : min(n, (int)(((int64_t)n * (part + 1) / C + 3) & ~int64_t(3)));
  const int len = s1 - s0;
  const float* x = a.logits + row * a.row_stride + s0;
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  RowKeys rk{x, nullptr, len, vec};
  for (int base = 0; base < len; base += 2 * kCStep) {
    const int c0 = base + 4 * threadIdx.x, c1 = c0 + kCStep;
    const uint4 k0 = rk.get4(c0);
    const uint4 k1 = rk.get4(c1);
    if (c0 < len) *reinterpret_cast<uint4*>(keys_s + c0) = k0;
    if (c1 < len) *reinterpret_cast<uint4*>(keys_s + c1) = k1;
  }
  rk.cache = keys_s;

  uint32_t prefix = 0, mask = 0;
  int remaining = k, equal_total = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int bins = pass == 0 ? 4096 : 1024;
    for (int i = threadIdx.x; i < bins; i += kCThreads) sh.hist[i] = 0;
    __syncthreads();
#pragma unroll 1
    for (int base = 0; base < len; base += kCStep) {
      const int c = base + 4 * threadIdx.x;
      const uint4 kk = rk.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t key = lane_of(kk, u);
        if (c + u < len && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & (uint32_t)(bins - 1)], 1u);
      }
    }
    cl.sync();  // every segment's histogram is complete
    // reduce-scatter: this CTA sums bin range [r0, r0 + rb) over the cluster
    const int rb = bins / C, r0 = part * rb;
    int mine = 0;
    for (int i = threadIdx.x; i < rb; i += kCThreads) {
      uint32_t t = 0;
      for (int q = 0; q < C; ++q) t += cl.map_shared_rank(sh.hist, q)[r0 + i];
      sh.sum[i] = t;
      mine += (int)t;
    }
    int range_total;
    cblock_excl_sum(mine, sh.warp_tot, &range_total);
    if (threadIdx.x < C) cl.map_shared_rank(sh.range_tot, (int)threadIdx.x)[part] = range_total;
    cl.sync();  // range totals everywhere; histograms no longer read remotely
    int above_ranges = 0;
    for (int q = part + 1; q < C; ++q) above_ranges += sh.range_tot[q];
    const bool owner = above_ranges < remaining && above_ranges + sh.range_tot[part] >= remaining;
    if (owner) {  // uniform within the CTA
      const int want = remaining - above_ranges;
      const int per = (rb + kCThreads - 1) / kCThreads;
      const int top = rb - 1 - (int)threadIdx.x * per;
      int tot = 0;
      for (int j = 0; j < per; ++j)
        if (top - j >= 0) tot += (int)sh.sum[top - j];
      int block_tot;
      int run = cblock_excl_sum(tot, sh.warp_tot, &block_tot);
      if (run < want && run + tot >= want) {
        for (int j = 0; j < per && top - j >= 0; ++j) {
          const int c = (int)sh.sum[top - j];
          if (run + c >= want) {
            const int res[3] = {r0 + top - j, above_ranges + run, c};
            for (int q = 0; q < C; ++q) {
              int32_t* dst = cl.map_shared_rank(sh.res, q);
              dst[0] = res[0];
              dst[1] = res[1];
              dst[2] = res[2];
            }
            break;
          }
          run += c;
        }
      }
    }
    cl.sync();  // the digit is everywhere
    remaining -= sh.res[1];
    equal_total = sh.res[2];
    prefix |= (uint32_t)sh.res[0] << shift;
    mask |= (uint32_t)(bins - 1) << shift;
    __syncthreads();
  }

  // per-segment counts above / equal to the threshold, exchanged in the cluster
  const uint32_t thr = prefix;
  int ngt = 0, neq = 0;
  for (int base = 0; base < len; base += kCStep) {
    const int c = base + 4 * threadIdx.x;
    const uint4 kk = rk.get4(c);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t key = lane_of(kk, u);
      ngt += (c + u < len && key > thr);
      neq += (c + u < len && key == thr);
    }
  }
  int seg_gt, seg_eq;
  cblock_excl_sum(ngt, sh.warp_tot, &seg_gt);
  cblock_excl_sum(neq, sh.warp_tot, &seg_eq);
  if (threadIdx.x < C) {
    cl.map_shared_rank(sh.cnt_gt, (int)threadIdx.x)[part] = seg_gt;
    cl.map_shared_rank(sh.cnt_eq, (int)threadIdx.x)[part] = seg_eq;
  }
  cl.sync();
  // equal keys are kept lowest-column first across the row
  int written = 0, equal_seen = 0;
  for (int q = 0; q < part; ++q) {
    const int take_eq = min(max(remaining - equal_seen, 0), sh.cnt_eq[q]);
    written += sh.cnt_gt[q] + take_eq;
    equal_seen += sh.cnt_eq[q];
  }
  const bool take_all_equal = remaining >= equal_total;
#pragma unroll 1
  for (int base = 0; base < len; base += kCStep) {
    const int c = base + 4 * threadIdx.x;
    const uint4 kk = rk.get4(c);
    int nq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) nq += (c + u < len && lane_of(kk, u) == thr);
    int eqs = equal_seen;
    if (!take_all_equal) {
      int tot;
      eqs += cblock_excl_sum(nq, sh.warp_tot, &tot);
      equal_seen += tot;
    }
    bool sel[4];
    int nsel = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t key = lane_of(kk, u);
      const bool okc = c + u < len;
      const bool eq = okc && key == thr;
      sel[u] = okc && (key > thr || (eq && (take_all_equal || eqs < remaining)));
      eqs += eq;
      nsel += sel[u];
    }
    int tot;
    int pos = written + cblock_excl_sum(nsel, sh.warp_tot, &tot);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sel[u]) {
        if (pos < k) o[pos] = s0 + c + u;
        ++pos;
      }
    written += tot;
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                        const int32_t* visible, int32_t k, int32_t* out, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  if (num_rows > 0x7FFFFFFFLL / kMaxCluster || row_stride > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  TopkArgs a{logits, num_rows, row_stride, visible, k, out, 0};
  DeviceInfo info;
  cudaError_t e = device_info(&info);
  if (e != cudaSuccess) return e;
  // few rows: split each row over a cluster so more SMs work on it
  int C = 1;
  for (int c = kMaxCluster; c >= 2; c /= 2)
    if (num_rows * c <= 2LL * info.num_sms && (row_stride + c - 1) / c + 8 <= kMaxCachedKeys) {
      C = c;
      break;
    }
  if (C > 1) {
    const int64_t seg = (row_stride + C - 1) / C + 8;
    const size_t smem = sizeof(uint32_t) * (size_t)((seg + 3) & ~int64_t(3));
    e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_rows * C), 1, 1);
    cfg.blockDim = dim3(kCThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  int64_t cap = row_stride < kMaxCachedKeys ? row_stride : kMaxCachedKeys;
  cap = (cap + 3) & ~int64_t(3);
  a.cache_cap = (int32_t)cap;
  const size_t smem = sizeof(uint32_t) * (size_t)cap;
  e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<(unsigned)num_rows, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qsa
