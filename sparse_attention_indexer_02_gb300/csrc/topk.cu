// Per-row top-k selection over [0, visible) of a logits row.
//
// vLLM #62589 "Details": the decode top-k reads only [0, visible_blocks[row]);
// SGLang #48649: rows whose visible count fits in k select every column.
// Selection rule: the k columns first in (logit descending, column ascending);
// the set is written in ascending column order, -1 in unused slots.
//
// A row is split over C CTAs (C = 1, or a thread-block cluster of 2, 4 or 8
// when there are few rows for the GPU and the row is longer than 16384
// columns), each owning a contiguous segment of the row.  Per CTA:
//  1. The segment is copied into shared memory by 16 KB bulk copies (mbarrier
//     per chunk) and turned in place into order-preserving uint32 keys while
//     the top 11 key bits are counted in a histogram.  Columns past the cache
//     (rows longer than it) are read from global memory in every pass.
//  2. The histograms of the C CTAs are summed over distributed shared memory
//     and every CTA finds the same first digit d0: the bin holding the k-th
//     largest key of the row.
//  3. One ordered pass over the segment counts, per warp, the keys above bin
//     d0, and compacts the keys inside it (the candidates) into the warp's
//     own list while counting their next 11 bits.  The next two digits (11
//     and 10 bits) come from the candidates alone.  (A CTA one of whose warps
//     overflows its list falls back to scanning its whole segment.)
//  4. The k-th largest key is the threshold; all larger keys are selected,
//     and of the keys equal to it the lowest columns.  Per-warp and per-CTA
//     counts give every warp its first output slot, and each warp writes its
//     selected columns in order with ballots.
// The cluster exchanges histograms and counts through distributed shared
// memory with one cluster barrier per digit and one for the counts (each
// digit has its own accumulator, zeroed at the start).
#include <cooperative_groups.h>

#include <mutex>

#include "device_common.cuh"
#include "qsa_internal.h"
#include "sm100_ptx.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kT = 512;                       // threads per CTA
constexpr int kW = kT / 32;                   // warps per CTA
constexpr int kBins = 2048;                   // 11-bit digits (the last one has 10 bits)
constexpr int kChunk = 4096;                  // floats per bulk copy (16 KB)
constexpr int kMaxChunks = 10;
constexpr int kCacheMax = kChunk * kMaxChunks;  // cached columns per CTA (160 KB)
constexpr int kCpwMax = 512;                  // candidate list entries per warp, at most
constexpr int kSoloMax = 16384;               // rows up to this long: one CTA even in a cluster
constexpr int kAccWords = 2 * 2048 + 1024;    // cluster accumulators of the three digits
constexpr int64_t kSmemMax = 226 * 1024;      // dynamic shared memory per CTA (static part aside)
constexpr int kSeg = 128;                     // columns a warp covers per step
constexpr int kMaxCluster = 8;
constexpr long long kTopkSpinCycles = 2000000000LL;  // ~1 s at 2 GHz

struct TopkArgs {
  const float* logits;
  int64_t row_stride;
  const int32_t* visible;
  int32_t* out;
  unsigned int* fault;
  int32_t k;
  int32_t cap;   // cached columns per CTA (multiple of 4, <= kCacheMax)
  int32_t cpw;   // candidate list entries per warp (multiple of 4)
  int32_t bulk;  // segments start 16-byte aligned: bulk copies fill the cache
};

struct TopkShared {
  uint64_t bar[kMaxChunks];
  int32_t warp_tot[kW];
  int32_t wgt[kW], weq[kW];  // per warp: keys above / equal to the threshold
  int32_t digit, above, equal;
  int32_t overflow;          // a warp's candidates did not fit its list
  int32_t cta_gt, cta_eq;    // read by the other CTAs of the cluster
  int32_t timed_out;
};

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ uint32_t lane_of(const uint4& v, int u) {
  return u == 0 ? v.x : (u == 1 ? v.y : (u == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint4 keys4(const float4 f) {
  return make_uint4(topk_key(f.x), topk_key(f.y), topk_key(f.z), topk_key(f.w));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Keys of one CTA's segment: columns [0, nc4) from the shared-memory cache
// (keys once pass 1 has converted them; read through 32-bit shared-window
// addresses), the rest from global memory.
struct Segment {
  const float* x;  // first column of the segment
  const uint32_t* cache;
  uint32_t cache_s;  // shared-window address of cache
  int len, nc4;
  bool vec;  // 16-byte global loads are aligned

  // keys of columns c .. c+3 (c a multiple of 4); lanes past len hold 0
  __device__ __forceinline__ uint4 get4(int c) const {
    if (c + 4 <= nc4) return lds128(cache_s + 4u * (uint32_t)c);
    if (vec && c + 4 <= len) return keys4(__ldg(reinterpret_cast<const float4*>(x + c)));
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = c + u < len ? topk_key(__ldg(x + c + u)) : 0u;
    return make_uint4(v[0], v[1], v[2], v[3]);
  }
  __device__ __forceinline__ uint32_t get1(int c) const { return c < nc4 ? cache[c] : topk_key(__ldg(x + c)); }
};

// Exclusive prefix of v over the CTA's threads, and the total.
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
  const int t = lane < kW ? warp_tot[lane] : 0;
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

// The digit whose bin holds the `remaining`-th largest candidate; thread t
// owns bins/kT consecutive bins in descending order.  Sets sh.digit / above /
// equal; callers synchronise before reading them.
__device__ __forceinline__ void find_digit(TopkShared& sh, const uint32_t* hist, int bins, int remaining) {
  const int per = bins / kT;
  const int top = bins - 1 - (int)threadIdx.x * per;
  int tot = 0;
  for (int j = 0; j < per; ++j) tot += (int)hist[top - j];
  int block_tot;
  int run = block_excl_sum(tot, sh.warp_tot, &block_tot);
  if (run < remaining && run + tot >= remaining) {
    for (int j = 0; j < per; ++j) {
      const int c = (int)hist[top - j];
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

// ---- cluster exchange -------------------------------------------------------
// Bin b of a cluster-wide histogram is owned by CTA b / (bins / C).  Every CTA
// adds its local counts into the owners' accumulators with remote reductions
// (zero bins skipped), one cluster barrier later every CTA reads the summed
// bins from their owners: one barrier per digit and 4 bytes of remote traffic
// per bin and CTA each way.

__device__ __forceinline__ uint32_t cluster_addr(const void* p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(ptx::smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_red_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Sums `bins` local histogram bins over the cluster into tot (local; may be
// the histogram itself: a thread reads its bins before it overwrites them);
// the accumulator `acc` (this digit's own, zero at kernel start) gets the
// pushes.  Thread t handles bins [t * per, t * per + per), per = bins / kT.
__device__ __forceinline__ void cluster_sum(const uint32_t* hist, uint32_t* acc, uint32_t* tot, int bins, int C) {
  const int per = bins / kT;  // 4 or 2
  const int b0 = (int)threadIdx.x * per;
  const int owner = b0 / (bins / C);
  const uint32_t dst = cluster_addr(acc + b0, owner);
  for (int j = 0; j < per; ++j) {
    const uint32_t v = hist[b0 + j];
    if (v) cluster_red_add(dst + 4u * (uint32_t)j, v);
  }
  cg::this_cluster().sync();  // every CTA's counts have landed in the owners' accumulators
  const uint32_t* src = cg::this_cluster().map_shared_rank(acc, owner) + b0;
  if (per == 4) {
    *reinterpret_cast<uint4*>(tot + b0) = *reinterpret_cast<const uint4*>(src);
  } else {
    *reinterpret_cast<uint2*>(tot + b0) = *reinterpret_cast<const uint2*>(src);
  }
  __syncthreads();
}

// Shared-memory layout (dynamic part), 16-byte aligned pieces:
//   cache [cap] | candidate lists [kW][cpw] | hist [kBins]
//   | cluster only: accumulators [kAccWords]
template <bool CLUSTER>
__global__ void __launch_bounds__(kT, 2) topk_kernel(const TopkArgs a) {
  extern __shared__ uint4 dyn_topk[];
  uint32_t* cache = reinterpret_cast<uint32_t*>(dyn_topk);  // floats as copied, keys after pass 1
  int32_t* cand = reinterpret_cast<int32_t*>(cache + a.cap);
  uint32_t* hist = reinterpret_cast<uint32_t*>(cand + kW * a.cpw);
  // cluster: per-digit accumulators of this CTA's bins (2048, 2048, 1024); the
  // summed histogram overwrites the local one, which is pushed by then
  uint32_t* acc = hist + kBins;
  uint32_t* tot = hist;
  __shared__ TopkShared sh;
  ptx::grid_dep_wait();  // the logits come from the previous kernel in the stream
  ptx::grid_dep_launch();

  const int lane = lane_id(), warp = threadIdx.x >> 5;
  int CL = 1, rank = 0;  // cluster size and this CTA's rank in it
  if (CLUSTER) {
    cg::cluster_group cl = cg::this_cluster();
    CL = (int)cl.num_blocks();
    rank = (int)cl.block_rank();
  }
  const int64_t row = blockIdx.x / CL;
  const int k = a.k;
  int32_t* o = a.out + row * (int64_t)k;
  const int n = (int)clamp64(a.visible[row], 0, a.row_stride);
  if (n <= k) {  // the same for every CTA of the cluster: no cluster barrier is pending
    if (rank == 0)
      for (int i = threadIdx.x; i < k; i += kT) o[i] = i < n ? i : -1;
    return;
  }
  // A row of at most kSoloMax columns is done by the cluster's first CTA
  // alone (measured faster than any exchange), the others leave at once;
  // the decision depends on the row only, so it is the same in every CTA.
  const bool multi = CLUSTER && n > kSoloMax;
  if (CLUSTER && !multi && rank != 0) return;
  const int C = multi ? CL : 1;
  const int part = multi ? rank : 0;
  // this CTA's segment [s0, s0 + len) of the row; boundaries on multiples of 4
  const int per_cta = ((n + C - 1) / C + 3) & ~3;
  const int s0 = min(n, part * per_cta);
  const int len = min(n, s0 + per_cta) - s0;
  const float* x = a.logits + row * a.row_stride + s0;
  const int nc4 = min(len, a.cap) & ~3;
  const int nchunks = a.bulk ? (nc4 + kChunk - 1) / kChunk : 0;
  const Segment seg{x, cache, ptx::smem_u32(cache), len, nc4, (reinterpret_cast<uintptr_t>(x) & 15u) == 0};

  for (int i = threadIdx.x; i < kBins; i += kT) hist[i] = 0;
  if (multi)
    for (int i = threadIdx.x; i < kAccWords; i += kT) acc[i] = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nchunks; ++i) ptx::mbar_init(&sh.bar[i], 1);
    sh.timed_out = 0;
    sh.overflow = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < kW) sh.weq[threadIdx.x] = 0;
  if (!a.bulk) {  // plain loads fill the cache
    for (int c = 4 * threadIdx.x; c < nc4; c += 4 * kT) {
      if (seg.vec) {
        *reinterpret_cast<float4*>(cache + c) = __ldg(reinterpret_cast<const float4*>(x + c));
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) reinterpret_cast<float*>(cache)[c + u] = __ldg(x + c + u);
      }
    }
  }
  __syncthreads();  // barriers initialised, histogram zeroed, plain-filled cache visible
  if (multi) cluster_arrive();  // accumulators zeroed (waited for before the first push)
  if (threadIdx.x == 0) {
    const uint64_t policy = ptx::policy_evict_first();  // each logit is read by one CTA
    for (int i = 0; i < nchunks; ++i) {
      const uint32_t bytes = 4u * (uint32_t)min(kChunk, nc4 - i * kChunk);
      ptx::mbar_arrive_expect_tx(&sh.bar[i], bytes);
      ptx::bulk_load(cache + (int64_t)i * kChunk, x + (int64_t)i * kChunk, bytes, &sh.bar[i], policy);
    }
  }

  // ---- pass 1: keys in place, histogram of the top 11 bits
  {
    int ready = -1;
    for (int c = 4 * threadIdx.x; c < len; c += 4 * kT) {
      uint4 kk;
      if (c + 4 <= nc4) {
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
        const uint4 f = lds128(seg.cache_s + 4u * (uint32_t)c);
        kk = keys4(make_float4(__uint_as_float(f.x), __uint_as_float(f.y), __uint_as_float(f.z),
                               __uint_as_float(f.w)));
        sts128(seg.cache_s + 4u * (uint32_t)c, kk);
      } else {
        kk = seg.get4(c);
      }
      if (c + 4 <= len) {  // every group but the segment's last: no per-key test
        atomicAdd(&hist[kk.x >> 21], 1u);
        atomicAdd(&hist[kk.y >> 21], 1u);
        atomicAdd(&hist[kk.z >> 21], 1u);
        atomicAdd(&hist[kk.w >> 21], 1u);
      } else {
#pragma unroll
        for (int u = 0; u < 3; ++u)
          if (c + u < len) atomicAdd(&hist[lane_of(kk, u) >> 21], 1u);
      }
    }
  }
  __syncthreads();
  int remaining = k;
  const uint32_t* H = hist;
  if (multi) {
    cluster_wait();
    cluster_sum(hist, acc, tot, kBins, C);
    H = tot;
  }
  find_digit(sh, H, kBins, remaining);
  __syncthreads();
  const uint32_t d0 = (uint32_t)sh.digit;
  remaining -= sh.above;
  __syncthreads();  // digit read; the local histogram is free again
  for (int i = threadIdx.x; i < kBins; i += kT) hist[i] = 0;
  __syncthreads();

  // ---- pass 2 (ordered, warp-contiguous): keys above bin d0 per warp, and
  // the candidates of bin d0 into the warp's list with a histogram of their
  // next 11 bits
  const int wseg = (len + kW * kSeg - 1) / (kW * kSeg) * kSeg;
  const int w0 = warp * wseg, w1 = min(len, w0 + wseg);
  const unsigned lt = (1u << lane) - 1u;
  int32_t* wl = cand + warp * a.cpw;  // this warp's candidate columns
  int ncw = 0;                        // candidates of this warp (warp-uniform)
  {
    int gt0 = 0;
    for (int c0 = w0; c0 < w1; c0 += kSeg) {  // warp-uniform trip count: collectives inside
      const int c = c0 + 4 * lane;
      const uint4 kk = seg.get4(c);
      const int lim = w1 - c;  // keys of this lane's group inside the warp's range
      bool cnd[4];
      int nc = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t top = lane_of(kk, u) >> 21;
        const bool in = u < lim;
        gt0 += (int)(in & (top > d0));
        cnd[u] = in & (top == d0);
        nc += (int)cnd[u];
      }
      if (__any_sync(0xFFFFFFFFu, nc > 0)) {
        int incl = nc;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
          const int t = __shfl_up_sync(0xFFFFFFFFu, incl, s);
          if (lane >= s) incl += t;
        }
        int pos = ncw + incl - nc;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (cnd[u]) {
            if (pos < a.cpw) wl[pos] = c + u;
            ++pos;
            atomicAdd(&hist[(lane_of(kk, u) >> 10) & 2047u], 1u);
          }
        ncw += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    gt0 = __reduce_add_sync(0xFFFFFFFFu, gt0);
    if (lane == 0) {
      sh.wgt[warp] = gt0;
      if (ncw > a.cpw) sh.overflow = 1;
    }
  }
  __syncthreads();
  const bool overflow = sh.overflow != 0;
  H = hist;
  if (multi) {
    cluster_sum(hist, acc + kBins, tot, kBins, C);
    H = tot;
  }
  find_digit(sh, H, kBins, remaining);
  __syncthreads();
  const uint32_t p22 = (d0 << 11) | (uint32_t)sh.digit;
  remaining -= sh.above;
  __syncthreads();
  for (int i = threadIdx.x; i < 1024; i += kT) hist[i] = 0;
  __syncthreads();

  // ---- pass 3: low 10 bits of the candidates whose top 22 bits are p22
  if (!overflow) {
    for (int i = lane; i < ncw; i += 32) {
      const uint32_t key = seg.get1(wl[i]);
      if ((key >> 10) == p22) atomicAdd(&hist[key & 1023u], 1u);
    }
  } else {
    for (int c = 4 * threadIdx.x; c < len; c += 4 * kT) {
      const uint4 kk = seg.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + u < len && (lane_of(kk, u) >> 10) == p22) atomicAdd(&hist[lane_of(kk, u) & 1023u], 1u);
    }
  }
  __syncthreads();
  H = hist;
  if (multi) {
    cluster_sum(hist, acc + 2 * kBins, tot, 1024, C);
    H = tot;
  }
  find_digit(sh, H, 1024, remaining);
  __syncthreads();
  // the k-th largest key; `remaining` of the `equal_total` keys equal to it are
  // kept (lowest columns first), every larger key is kept
  const uint32_t thr = (p22 << 10) | (uint32_t)sh.digit;
  remaining -= sh.above;
  const int equal_total = sh.equal;
  const bool take_all_equal = remaining >= equal_total;

  // ---- per-warp counts: bin-d0 keys above / equal to the threshold
  {
    int gt = 0, eq = 0;
    if (!overflow) {
      for (int i = lane; i < ncw; i += 32) {
        const uint32_t key = seg.get1(wl[i]);
        gt += key > thr;
        eq += key == thr;
      }
    } else {
      for (int c = w0 + 4 * lane; c < w1; c += kSeg) {  // no collectives inside
        const uint4 kk = seg.get4(c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t key = lane_of(kk, u);
          const bool in = c + u < w1 && (key >> 21) == d0;
          gt += in && key > thr;
          eq += in && key == thr;
        }
      }
    }
    gt = __reduce_add_sync(0xFFFFFFFFu, gt);
    eq = __reduce_add_sync(0xFFFFFFFFu, eq);
    if (lane == 0) {
      sh.wgt[warp] += gt;
      sh.weq[warp] = eq;
    }
  }
  __syncthreads();

  // ---- first output slot of every warp
  const int g = lane < kW ? sh.wgt[lane] : 0;
  const int e = lane < kW ? sh.weq[lane] : 0;
  int cta_base = 0, cta_eq_before = 0;
  if (multi) {
    cg::cluster_group cl = cg::this_cluster();
    const int gtot = __reduce_add_sync(0xFFFFFFFFu, g), etot = __reduce_add_sync(0xFFFFFFFFu, e);
    if (threadIdx.x == 0) {
      sh.cta_gt = gtot;
      sh.cta_eq = etot;
    }
    cl.sync();
    // lane q < C reads CTA q's counts
    int qg = 0, qe = 0;
    if (lane < C) {
      qg = *cl.map_shared_rank(&sh.cta_gt, lane);
      qe = *cl.map_shared_rank(&sh.cta_eq, lane);
    }
    __syncwarp();
    cluster_arrive();  // done with remote shared memory (waited for before exit)
    int qei = qe;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, qei, s);
      if (lane >= s) qei += t;
    }
    const int qeb = qei - qe;  // tied keys in the CTAs before CTA `lane`
    const int qtake = take_all_equal ? qe : min(max(remaining - qeb, 0), qe);
    int qs = lane < part ? qg + qtake : 0;
    qs = __reduce_add_sync(0xFFFFFFFFu, qs);
    cta_base = qs;
    cta_eq_before = __shfl_sync(0xFFFFFFFFu, qeb, part);
  }
  int base, eq_before, mine;
  {
    int ei = e;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, ei, s);
      if (lane >= s) ei += t;
    }
    const int eb = cta_eq_before + ei - e;
    const int take = take_all_equal ? e : min(max(remaining - eb, 0), e);
    const int cnt = g + take;
    int ci = cnt;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, ci, s);
      if (lane >= s) ci += t;
    }
    base = cta_base + __shfl_sync(0xFFFFFFFFu, ci - cnt, warp);
    eq_before = __shfl_sync(0xFFFFFFFFu, eb, warp);
    mine = __shfl_sync(0xFFFFFFFFu, cnt, warp);
  }

  // ---- ordered write of this warp's selected columns
  if (mine > 0) {
    int run = 0, eq_run = eq_before;
    for (int c0 = w0; c0 < w1 && run < mine; c0 += kSeg) {  // warp-uniform
      const int c = c0 + 4 * lane;
      const uint4 kk = seg.get4(c);
      const int lim = w1 - c;
      bool ge[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ge[u] = (u < lim) & (lane_of(kk, u) >= thr);
      if (!__any_sync(0xFFFFFFFFu, ge[0] | ge[1] | ge[2] | ge[3])) continue;
      bool sel[4];
      if (take_all_equal) {
#pragma unroll
        for (int u = 0; u < 4; ++u) sel[u] = ge[u];
      } else {
        bool eqf[4];
        int lane_eq_before = 0, step_eq = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          eqf[u] = ge[u] && lane_of(kk, u) == thr;
          const unsigned b = __ballot_sync(0xFFFFFFFFu, eqf[u]);
          lane_eq_before += __popc(b & lt);
          step_eq += __popc(b);
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
          if (pos < k) o[pos] = s0 + c + u;
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
  // no CTA leaves while another may still read its shared memory
  __syncwarp();
  if (multi) cluster_wait();
}

}  // namespace

namespace {

// Shared-memory plan of one launch: the segment cache, per-warp candidate
// lists and the histograms.  One CTA a row aims at two CTAs per SM (lists of
// at least 64 entries a warp); a cluster launch keeps one CTA per SM (its
// solo rows then never share an SM) and kCpwMax-entry lists.
struct TopkPlan {
  int64_t cap, cpw;
  size_t smem;
};

TopkPlan plan_for(int C, int64_t row_stride) {
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
    if (4 * cap + fixed + 4LL * kW * 64 <= two_per_sm) {
      cpw = ((two_per_sm - 4 * cap - fixed) / (4LL * kW)) & ~int64_t(3);
      if (cpw > kCpwMax) cpw = kCpwMax;
    }
  }
  const int64_t room = (kSmemMax - fixed - 4LL * kW * cpw) / 4;
  if (cap > room) cap = room & ~int64_t(3);
  return TopkPlan{cap, cpw, (size_t)(4 * (cap + kW * cpw) + fixed)};
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
  e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  e = cudaOccupancyMaxActiveClusters(&n, topk_kernel<true>, &cfg);
  if (e != cudaSuccess) return e;
  cache[used % 32] = Entry{dev, c, smem, n};
  if (used < 32) ++used;
  *out = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                        const int32_t* visible, int32_t k, int32_t* out, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  if (num_rows > 0x7FFFFFFFLL / kMaxCluster || row_stride > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  unsigned int* fault = nullptr;
  cudaError_t e = fault_word_address(&fault);
  if (e != cudaSuccess) return e;
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
  const TopkPlan pl = plan_for(C, row_stride);
  TopkArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.visible = visible;
  a.out = out;
  a.fault = fault;
  a.k = k;
  a.cap = (int32_t)pl.cap;
  a.cpw = (int32_t)pl.cpw;
  // segment starts are multiples of 4 columns: 16-byte aligned when rows are
  a.bulk = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (row_stride & 3) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_rows * C), 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
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
    e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<true>, a);
  } else {
    e = cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<false>, a);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
