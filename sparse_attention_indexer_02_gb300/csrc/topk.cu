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
#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kMaxCachedKeys = 48 * 1024;    // cluster kernel: 192 KB of keys per CTA at most
constexpr int kBins = 4096;
constexpr long long kTopkSpinCycles = 2000000000LL;  // ~1 s at 2 GHz

struct TopkArgs {
  const float* logits;
  int64_t num_rows, row_stride;
  const int32_t* visible;
  int32_t k;
  int32_t* out;
  int32_t cache_cap;  // keys the dynamic shared memory caches (multiple of 4)
};

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

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

// ---------------------------------------------------------------------------
// One CTA per row.
//
// The row's first `cap` columns are copied into shared memory as raw floats by
// bulk copies (16 KB chunks, one mbarrier each) that the first pass consumes
// as they land; columns past `cap` (rows longer than the cache) are read from
// global memory in every pass.  Logits map to order-preserving uint32 keys on
// the fly.  The k-th largest key is found digit by digit, most significant
// first (11, 11 and 10 bits), each digit from a shared-memory histogram of the
// keys that still match the prefix.  Then each warp takes a contiguous segment
// of the row: it counts its keys above and equal to the threshold, one
// exchange of the 16 warps' counts gives every warp its first output slot and
// the number of tied keys before it, and the warp writes its selected columns
// in order with ballots - no block-wide step per column block.
// ---------------------------------------------------------------------------

constexpr int kRT = 512;                   // threads of a row CTA
constexpr int kRW = kRT / 32;
constexpr int kRBins = 2048;               // largest digit: 11 bits
constexpr int kChunk = 4096;               // floats per bulk copy (16 KB)
constexpr int kRowCacheMax = 11 * kChunk;  // 176 KB of cached floats at most
constexpr int kSeg = 128;                  // columns a warp covers per step

struct RowArgs {
  const float* logits;
  int64_t row_stride;
  const int32_t* visible;
  int32_t* out;
  unsigned int* fault;
  int32_t k;
  int32_t cap;   // cached columns (multiple of 4, <= kRowCacheMax)
  int32_t bulk;  // rows start 16-byte aligned: bulk copies fill the cache
};

struct RowShared {
  uint32_t hist[kRBins];
  uint64_t bar[kRowCacheMax / kChunk];
  int32_t warp_tot[kRW];
  int32_t wgt[kRW], weq[kRW];
  int32_t digit, above, equal;
  int32_t timed_out;
};

__device__ __forceinline__ uint4 keys4(const float4 f) {
  return make_uint4(topk_key(f.x), topk_key(f.y), topk_key(f.z), topk_key(f.w));
}

// Keys of columns c .. c+3 (c a multiple of 4); lanes past n hold 0 and are
// masked by the callers.  Cached columns come from shared memory.
struct RowSource {
  const float* x;
  const float* cache;
  int n, nc4;  // columns in the row; fully cached 4-column groups end at nc4
  bool vec;    // 16-byte global loads are aligned

  __device__ __forceinline__ uint4 get4(int c) const {
    if (c + 4 <= nc4) return keys4(*reinterpret_cast<const float4*>(cache + c));
    if (vec && c + 4 <= n) return keys4(__ldg(reinterpret_cast<const float4*>(x + c)));
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = c + u < n ? topk_key(__ldg(x + c + u)) : 0u;
    return make_uint4(v[0], v[1], v[2], v[3]);
  }
};

// Exclusive prefix over the CTA's threads of v, and the total.
__device__ __forceinline__ int row_excl_sum(int v, int32_t* warp_tot, int* total) {
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  const int t = lane < kRW ? warp_tot[lane] : 0;
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

// The digit whose bin holds the `remaining`-th largest candidate (bins in
// descending order over the threads); sets sh.digit / above / equal.
__device__ __forceinline__ void row_find_digit(RowShared& sh, int bins, int remaining) {
  const int per = bins / kRT;
  const int top = bins - 1 - (int)threadIdx.x * per;
  int tot = 0;
  for (int j = 0; j < per; ++j) tot += (int)sh.hist[top - j];
  int block_tot;
  int run = row_excl_sum(tot, sh.warp_tot, &block_tot);
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

__global__ void __launch_bounds__(kRT, 2) topk_row_kernel(const RowArgs a) {
  extern __shared__ uint4 dyn_row[];
  float* cache = reinterpret_cast<float*>(dyn_row);
  __shared__ RowShared sh;
  ptx::grid_dep_wait();  // the logits come from the previous kernel in the stream
  ptx::grid_dep_launch();
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int k = a.k;
  int32_t* o = a.out + row * (int64_t)k;
  const int n = (int)clamp64(a.visible[row], 0, a.row_stride);
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kRT) o[i] = i < n ? i : -1;
    return;
  }
  const float* x = a.logits + row * a.row_stride;
  const int nc = min(n, a.cap);
  const int nc4 = nc & ~3;
  const int nchunks = a.bulk ? (nc4 + kChunk - 1) / kChunk : 0;
  for (int i = threadIdx.x; i < kRBins; i += kRT) sh.hist[i] = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nchunks; ++i) ptx::mbar_init(&sh.bar[i], 1);
    sh.timed_out = 0;
    ptx::fence_mbar_init();
  }
  if (!a.bulk) {  // plain 16-byte (or 4-byte) loads fill the cache
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    for (int c = 4 * threadIdx.x; c < nc4; c += 4 * kRT) {
      if (vec) {
        *reinterpret_cast<float4*>(cache + c) = __ldg(reinterpret_cast<const float4*>(x + c));
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) cache[c + u] = __ldg(x + c + u);
      }
    }
  }
  __syncthreads();  // barriers initialised, histogram zeroed, plain-filled cache visible
  if (threadIdx.x == 0) {
    const uint64_t policy = ptx::policy_evict_first();  // the logits are read by this CTA only
    for (int i = 0; i < nchunks; ++i) {
      const uint32_t bytes = 4u * (uint32_t)min(kChunk, nc4 - i * kChunk);
      ptx::mbar_arrive_expect_tx(&sh.bar[i], bytes);
      ptx::bulk_load(cache + (int64_t)i * kChunk, x + (int64_t)i * kChunk, bytes, &sh.bar[i], policy);
    }
  }
  const RowSource src{x, cache, n, nc4, ((reinterpret_cast<uintptr_t>(x) & 15u) == 0)};

  // pass 1: histogram of the top 11 bits, chunk by chunk as the copies land
  {
    int ready = -1;
    for (int c = 4 * threadIdx.x; c < n; c += 4 * kRT) {
      if (c < nc4) {
        const int ch = c / kChunk;
        while (ready < ch && ready + 1 < nchunks) {
          ++ready;
          if (!ptx::mbar_try_wait(&sh.bar[ready], 0)) {
            const long long t0 = clock64();
            bool ok = false;
            while (!(ok = ptx::mbar_try_wait(&sh.bar[ready], 0)) && clock64() - t0 < kTopkSpinCycles) {
            }
            if (!ok) {
              sh.timed_out = 1;
              atomicOr(a.fault, 2u);
            }
          }
        }
      }
      const uint4 kk = src.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + u < n) atomicAdd(&sh.hist[lane_of(kk, u) >> 21], 1u);
    }
  }
  __syncthreads();
  int remaining = k;
  row_find_digit(sh, 2048, remaining);
  __syncthreads();
  const uint32_t d0 = (uint32_t)sh.digit;
  remaining -= sh.above;
  __syncthreads();
  for (int i = threadIdx.x; i < kRBins; i += kRT) sh.hist[i] = 0;
  __syncthreads();
  // pass 2: next 11 bits of the keys whose top 11 bits are d0
  for (int c = 4 * threadIdx.x; c < n; c += 4 * kRT) {
    const uint4 kk = src.get4(c);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t key = lane_of(kk, u);
      if (c + u < n && (key >> 21) == d0) atomicAdd(&sh.hist[(key >> 10) & 2047u], 1u);
    }
  }
  __syncthreads();
  row_find_digit(sh, 2048, remaining);
  __syncthreads();
  const uint32_t p22 = (d0 << 11) | (uint32_t)sh.digit;
  remaining -= sh.above;
  __syncthreads();
  for (int i = threadIdx.x; i < 1024; i += kRT) sh.hist[i] = 0;
  __syncthreads();
  // pass 3: low 10 bits of the keys whose top 22 bits are p22
  for (int c = 4 * threadIdx.x; c < n; c += 4 * kRT) {
    const uint4 kk = src.get4(c);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t key = lane_of(kk, u);
      if (c + u < n && (key >> 10) == p22) atomicAdd(&sh.hist[key & 1023u], 1u);
    }
  }
  __syncthreads();
  row_find_digit(sh, 1024, remaining);
  __syncthreads();
  // the k-th largest key; `remaining` of the `equal_total` keys equal to it are
  // kept (lowest columns first), every larger key is kept
  const uint32_t thr = (p22 << 10) | (uint32_t)sh.digit;
  remaining -= sh.above;
  const int equal_total = sh.equal;
  const bool take_all_equal = remaining >= equal_total;

  // per-warp counts over contiguous segments of kSeg-column steps
  const int seg = (n + kRW * kSeg - 1) / (kRW * kSeg) * kSeg;
  const int w0 = warp * seg, w1 = min(n, w0 + seg);
  {
    int gt = 0, eq = 0;
    for (int c = w0 + 4 * lane; c < w1; c += kSeg) {
      const uint4 kk = src.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t key = lane_of(kk, u);
        gt += (c + u < w1 && key > thr);
        eq += (c + u < w1 && key == thr);
      }
    }
    gt = __reduce_add_sync(0xFFFFFFFFu, gt);
    eq = __reduce_add_sync(0xFFFFFFFFu, eq);
    if (lane == 0) {
      sh.wgt[warp] = gt;
      sh.weq[warp] = eq;
    }
  }
  __syncthreads();
  // this warp's first output slot and the tied keys in the segments before it
  int base, eq_before, mine;
  {
    const int g = lane < kRW ? sh.wgt[lane] : 0;
    const int e = lane < kRW ? sh.weq[lane] : 0;
    int ei = e;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, ei, s);
      if (lane >= s) ei += t;
    }
    const int eb = ei - e;
    const int take = take_all_equal ? e : min(max(remaining - eb, 0), e);
    const int cnt = g + take;
    int ci = cnt;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, ci, s);
      if (lane >= s) ci += t;
    }
    base = __shfl_sync(0xFFFFFFFFu, ci - cnt, warp);
    eq_before = __shfl_sync(0xFFFFFFFFu, eb, warp);
    mine = __shfl_sync(0xFFFFFFFFu, cnt, warp);
  }
  // ordered write of this warp's selected columns
  if (mine > 0) {
    const unsigned lt = (1u << lane) - 1u;
    int run = 0, eq_run = eq_before;
    for (int c0 = w0; c0 < w1 && run < mine; c0 += kSeg) {
      const int c = c0 + 4 * lane;
      const uint4 kk = src.get4(c);
      bool ge[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ge[u] = c + u < w1 && lane_of(kk, u) >= thr;
      if (!__any_sync(0xFFFFFFFFu, ge[0] | ge[1] | ge[2] | ge[3])) continue;
      bool sel[4];
      if (take_all_equal) {
#pragma unroll
        for (int u = 0; u < 4; ++u) sel[u] = ge[u];
      } else {
        bool eqf[4];
        unsigned eb[4];
        int lane_eq_before = 0, step_eq = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          eqf[u] = ge[u] && lane_of(kk, u) == thr;
          eb[u] = __ballot_sync(0xFFFFFFFFu, eqf[u]);
          lane_eq_before += __popc(eb[u] & lt);
          step_eq += __popc(eb[u]);
        }
        int r = eq_run + lane_eq_before;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sel[u] = ge[u] && (!eqf[u] || r < remaining);
          r += eqf[u];
        }
        eq_run += step_eq;
      }
      int pos = base + run;
      int step_sel = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned sb = __ballot_sync(0xFFFFFFFFu, sel[u]);
        pos += __popc(sb & lt);
        step_sel += __popc(sb);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (sel[u]) {
          if (pos < k) o[pos] = c + u;
          ++pos;
        }
      run += step_sel;
    }
  }
  // a copy that timed out may still land: wait for it again (bounded) before exit
  if (sh.timed_out && threadIdx.x == 0)
    for (int i = 0; i < nchunks; ++i) {
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(&sh.bar[i], 0) && clock64() - t0 < kTopkSpinCycles) {
      }
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
// lowest columns first across the whole row).  A row with at most
// kSoloMaxCols visible columns is done by the cluster's first CTA alone (no
// cluster barriers; measured faster at that size), the others exit.
// ---------------------------------------------------------------------------

constexpr int kCThreads = 512;
constexpr int kSoloMaxCols = 12288;  // rows up to this many visible columns skip the cluster exchange
constexpr int kCWarps = kCThreads / 32;
constexpr int kCStep = 4 * kCThreads;
constexpr int kMaxCluster = 8;

struct ClusterShared {
  uint32_t hist[kBins];        // this CTA's histogram of its segment
  uint32_t sum[kBins];         // summed counts of this CTA's bin range (all bins when solo)
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
  // solo: uniform over the cluster (it depends on the row only)
  const bool solo = n <= kSoloMaxCols;
  if (solo && part != 0) return;
  const int CC = solo ? 1 : C;  // CTAs sharing the row
  // segment [s0, s1) of the row, boundaries on multiples of 4 columns
  const int s0 = part == 0 ? 0 : min(n, (int)(((int64_t)n * part / CC + 3) & ~int64_t(3)));
  const int s1 = part == CC - 1 ? n : min(n, (int)(((int64_t)n * (part + 1) / CC + 3) & ~int64_t(3)));
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
    if (!solo) cl.sync();  // every segment's histogram is complete
    else __syncthreads();
    // reduce-scatter: this CTA sums bin range [r0, r0 + rb) over the cluster
    // (its own counts from local shared memory; the other CTAs' counts of a
    // bin are all loaded before any is added)
    const int rb = bins / CC, r0 = part * rb;
    int mine = 0;
    for (int i = threadIdx.x; i < rb; i += kCThreads) {
      uint32_t t = sh.hist[r0 + i];
      if (!solo) {
        uint32_t v[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
          v[q] = q < CC && q != part ? cl.map_shared_rank(sh.hist, q)[r0 + i] : 0u;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) t += v[q];
      }
      sh.sum[i] = t;
      mine += (int)t;
    }
    int range_total;
    cblock_excl_sum(mine, sh.warp_tot, &range_total);
    if (threadIdx.x < CC) cl.map_shared_rank(sh.range_tot, (int)threadIdx.x)[part] = range_total;
    if (!solo) cl.sync();  // range totals everywhere; histograms no longer read remotely
    else __syncthreads();
    int above_ranges = 0;
    for (int q = part + 1; q < CC; ++q) above_ranges += sh.range_tot[q];
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
            for (int q = 0; q < CC; ++q) {
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
    if (!solo) cl.sync();  // the digit is everywhere
    else __syncthreads();
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
  if (threadIdx.x < CC) {
    cl.map_shared_rank(sh.cnt_gt, (int)threadIdx.x)[part] = seg_gt;
    cl.map_shared_rank(sh.cnt_eq, (int)threadIdx.x)[part] = seg_eq;
  }
  if (!solo) cl.sync();
  else __syncthreads();
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
  int C = 1;
  if (C > 1) {
    const int64_t solo = row_stride < kSoloMaxCols ? row_stride : kSoloMaxCols;
    int64_t seg = (row_stride + C - 1) / C + 8;
    if (seg < solo + 8) seg = solo + 8;
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
  unsigned int* fault = nullptr;
  e = fault_word_address(&fault);
  if (e != cudaSuccess) return e;
  RowArgs ra;
  ra.logits = logits;
  ra.row_stride = row_stride;
  ra.visible = visible;
  ra.out = out;
  ra.fault = fault;
  ra.k = k;
  int64_t cap = (row_stride + 3) & ~int64_t(3);
  ra.cap = (int32_t)(cap < kRowCacheMax ? cap : kRowCacheMax);
  ra.bulk = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (row_stride & 3) == 0;
  const size_t smem = sizeof(float) * (size_t)ra.cap;
  e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_rows, 1, 1);
  cfg.blockDim = dim3(kRT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_row_kernel, ra);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
