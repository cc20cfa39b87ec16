// Per-row top-k selection over [0, n) of a logits row: the CTA-level body
// shared by the top-k kernel (topk.cu) and the fused scoring + selection
// kernel (umma_kernel.cuh).
//
// vLLM #62589 "Details": the decode top-k reads only [0, visible_blocks[row]);
// SGLang #48649: rows whose visible count fits in k select every column.
// Selection rule: the k columns first in (logit descending, column ascending);
// the set is written in ascending column order, -1 in unused slots.
//
// A row is split over C CTAs (C = 1, or a thread-block cluster of 2, 4 or 8
// when there are few rows for the GPU and the row is longer than 16384
// columns), each owning a contiguous segment of the row.  A segment of at
// most 8192 columns (16 a thread) is selected with its keys in registers
// (select_row_reg below).  Longer segments take the compaction path, per CTA:
//  1. The segment is copied into shared memory (16 KB bulk copies with an
//     mbarrier per chunk, or plain loads) and turned in place into
//     order-preserving uint32 keys while the top 11 key bits are counted in a
//     histogram.  Columns past the cache (rows longer than it) are read from
//     global memory in every pass.
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
#pragma once
#include <cooperative_groups.h>

#include "device_common.cuh"
#include "sm100_ptx.cuh"

namespace qsa {
namespace sel {

namespace cg = cooperative_groups;

constexpr int kBins = 2048;                   // 11-bit digits (the last one has 10 bits)
constexpr int kChunk = 4096;                  // floats per bulk copy (16 KB)
constexpr int kMaxChunks = 10;
constexpr int kCacheMax = kChunk * kMaxChunks;  // cached columns per CTA (160 KB)
constexpr int kCpwMax = 512;                  // candidate list entries per warp, at most
constexpr int kSoloMax = 16384;               // rows up to this long: one CTA even in a cluster
constexpr int kAccWords = 2 * 2048 + 1024;    // cluster accumulators of the three digits
constexpr int kSeg = 128;                     // columns a warp covers per step
constexpr int kMaxCluster = 8;
constexpr int kMaxWarps = 32;                 // selecting threads per CTA: 256, 512 or 1024
constexpr long long kSpinCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr int kBarrier = 2;                   // named barrier of the selecting threads

struct Shared {
  uint64_t bar[kMaxChunks];
  int32_t warp_tot[kMaxWarps];
  int32_t wgt[kMaxWarps], weq[kMaxWarps];  // per warp: keys above / equal to the threshold
  int32_t digit, above, equal;
  int32_t overflow;          // a warp's candidates did not fit its list
  int32_t cta_gt, cta_eq;    // read by the other CTAs of the cluster
  int32_t timed_out;
};

// One row's selection: columns [0, n) of `row`, k slots at `out`.
struct RowTask {
  const float* row;
  int n;
  int32_t* out;
};

struct Config {
  int k;
  int cap;    // cached columns per CTA (multiple of 4, <= kCacheMax)
  int cpw;    // candidate list entries per warp (multiple of 4)
  int bulk;   // segments start 16-byte aligned: bulk copies fill the cache
  unsigned int* fault;  // bit 1 set when a copy wait gives up
  int pcap;   // candidates (a column and a key each) the sampled-pivot path holds (<= NT * KPT; below k: off)
};

// Dynamic shared memory one selecting CTA needs (bytes).
__host__ __device__ constexpr size_t smem_bytes(int nt, int cap, int cpw, bool cluster) {
  return 4 * ((size_t)cap + (size_t)(nt / 32) * cpw + kBins + (cluster ? kAccWords : 0));
}

template <int NT>
__device__ __forceinline__ void bar_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kBarrier), "n"(NT) : "memory");
}

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

// Global loads of logits: through the read-only path when the logits come
// from an earlier kernel, coherent at L2 when other CTAs of the same kernel
// wrote them.
template <bool COHERENT>
__device__ __forceinline__ float4 ld_row4(const float* p) {
  return COHERENT ? __ldcg(reinterpret_cast<const float4*>(p)) : __ldg(reinterpret_cast<const float4*>(p));
}
template <bool COHERENT>
__device__ __forceinline__ float ld_row1(const float* p) {
  return COHERENT ? __ldcg(p) : __ldg(p);
}

// Keys of one CTA's segment: columns [0, nc4) from the shared-memory cache
// (keys once pass 1 has converted them; read through 32-bit shared-window
// addresses), the rest from global memory.
template <bool COHERENT>
struct Segment {
  const float* x;  // first column of the segment
  const uint32_t* cache;
  uint32_t cache_s;  // shared-window address of cache
  int len, nc4;
  bool vec;  // 16-byte global loads are aligned

  // keys of columns c .. c+3 (c a multiple of 4); lanes past len hold 0
  __device__ __forceinline__ uint4 get4(int c) const {
    if (c + 4 <= nc4) return lds128(cache_s + 4u * (uint32_t)c);
    if (vec && c + 4 <= len) return keys4(ld_row4<COHERENT>(x + c));
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = c + u < len ? topk_key(ld_row1<COHERENT>(x + c + u)) : 0u;
    return make_uint4(v[0], v[1], v[2], v[3]);
  }
  __device__ __forceinline__ uint32_t get1(int c) const {
    return c < nc4 ? cache[c] : topk_key(ld_row1<COHERENT>(x + c));
  }
};

// Exclusive prefix of v over the NT selecting threads, and the total.  The
// warp totals are read after the one barrier; callers put a barrier between
// two calls (every caller does), so the next call cannot overwrite them early.
template <int NT>
__device__ __forceinline__ int block_excl_sum(int v, int32_t* warp_tot, int* total) {
  constexpr int kW = NT / 32;
  const int lane = lane_id(), warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  bar_sync<NT>();
  const int t = lane < kW ? warp_tot[lane] : 0;
  int wincl = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
    if (lane >= o) wincl += u;
  }
  const int warp_excl = __shfl_sync(0xFFFFFFFFu, wincl - t, warp);
  *total = __shfl_sync(0xFFFFFFFFu, wincl, 31);
  return warp_excl + incl - v;
}

// The digit whose bin holds the `remaining`-th largest candidate; thread t
// owns bins/NT consecutive bins in descending order.  Sets sh.digit / above /
// equal; callers synchronise before reading them.
template <int NT>
__device__ __forceinline__ void find_digit(Shared& sh, const uint32_t* hist, int bins, int remaining) {
  const int per = bins / NT;
  const int top = bins - 1 - (int)threadIdx.x * per;
  int tot = 0;
  for (int j = 0; j < per; ++j) tot += (int)hist[top - j];
  int block_tot;
  int run = block_excl_sum<NT>(tot, sh.warp_tot, &block_tot);
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
// pushes.  Thread t handles bins [t * per, t * per + per), per = bins / NT.
template <int NT>
__device__ __forceinline__ void cluster_sum(const uint32_t* hist, uint32_t* acc, uint32_t* tot, int bins, int C) {
  const int per = bins / NT;  // 4 or 2
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
  bar_sync<NT>();
}

// ---- register-resident selection ---------------------------------------------
// A CTA's segment of at most NT * KPT columns (a row one CTA selects alone, or
// one CTA's share of a row a cluster splits): with q = ceil(len / NT) <= KPT,
// thread t holds the keys of segment columns [t * q, t * q + q) in registers
// (every thread has keys, however short the segment), so every digit's
// histogram is a scan of registers (the keys of the current prefix only), no
// candidate list is needed, and thread order is column order: one exclusive
// scan of each thread's (above, equal) counts gives every thread its first
// output slot.  In a cluster the histograms are summed over distributed shared
// memory and the CTAs' counts exchanged exactly as in the compaction path
// below (one cluster barrier per digit and one for the counts).
// (Staging the row and the output through shared memory for coalesced global
// accesses, and writing each warp's run of output slots coalesced with a
// shuffle search for each slot's owner lane, both measured slower for rows of
// 2K to 8K columns than these per-thread stores.)
// Shared memory at `dyn`: three histograms (2048 + 2048 + 1024 words), then in
// a cluster the per-digit accumulators (kAccWords).
constexpr int kRegHistWords = 2 * kBins + 1024;

// CAND: the n keys are those of the sampled-pivot path's candidates, whose
// columns are in the per-warp slices of `wcap` entries of ccol and whose keys
// are at the same places of the NT / 32 slices that follow them; slice w
// holds the candidates from order position sh.weq[w] on (order = column
// order).  The selected columns are the candidates' ccol entries.
template <int NT, int KPT, bool COHERENT, bool CLUSTER, bool CAND = false>
__device__ __forceinline__ void select_row_reg(const RowTask& task, const Config& cf, uint32_t* dyn, Shared& sh,
                                               int C, int part, const int32_t* ccol = nullptr, int wcap = 0) {
  static_assert(KPT % 4 == 0, "keys per thread in groups of 4");
  const int tid = (int)threadIdx.x;
  const int lane = lane_id();
  const bool multi = CLUSTER && C > 1;  // the same in every CTA of the cluster
  const int n = task.n, k = cf.k;
  // this CTA's segment [s0, s0 + len) of the row; boundaries on multiples of 4
  const int per_cta = ((n + C - 1) / C + 3) & ~3;
  const int s0 = min(n, part * per_cta);
  const int len = min(n, s0 + per_cta) - s0;
  const float* x = task.row + s0;
  uint32_t* h0 = dyn;
  uint32_t* h1 = h0 + kBins;
  uint32_t* h2 = h1 + kBins;
  uint32_t* acc = dyn + kRegHistWords;  // cluster: the three digits' accumulators
  for (int i = tid; i < kRegHistWords; i += NT) h0[i] = 0;
  if (multi)
    for (int i = tid; i < kAccWords; i += NT) acc[i] = 0;
  // this thread's keys; slots past its columns hold key 0 and are never counted
  const int q = (len + NT - 1) / NT;
  const int c0 = tid * q;
  const int mine = max(0, min(q, len - c0));  // valid keys of this thread
  uint32_t key[KPT];
  int cidx[CAND ? KPT : 1];  // CAND: slice index of each of this thread's candidates
  if (CAND) {
    // the slice w holding order position g: [lo, hi) = [weq[w], weq[w + 1])
    constexpr int kWs = NT / 32;
    int w = 0, lo = 0, hi = kWs > 1 ? sh.weq[1] : INT32_MAX;
    while (c0 >= hi && w + 1 < kWs) {
      ++w;
      lo = hi;
      hi = w + 1 < kWs ? sh.weq[w + 1] : INT32_MAX;
    }
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      cidx[j] = 0;
      if (j < mine) {
        while (c0 + j >= hi && w + 1 < kWs) {
          ++w;
          lo = hi;
          hi = w + 1 < kWs ? sh.weq[w + 1] : INT32_MAX;
        }
        cidx[j] = w * wcap + (c0 + j - lo);
      }
    }
    // their keys, written by the pivot pass beside their columns
    const uint32_t* ckey = reinterpret_cast<const uint32_t*>(ccol) + kWs * wcap;
#pragma unroll
    for (int j = 0; j < KPT; ++j) key[j] = j < mine ? ckey[cidx[j]] : 0u;
  } else if ((q & 3) == 0 && (reinterpret_cast<uintptr_t>(x + c0) & 15u) == 0) {
#pragma unroll
    for (int j = 0; j < KPT; j += 4) {
      uint4 kk = make_uint4(0u, 0u, 0u, 0u);
      if (j < mine) kk = keys4(ld_row4<COHERENT>(x + c0 + j));  // mine is a multiple of 4 here
      key[j] = kk.x;
      key[j + 1] = kk.y;
      key[j + 2] = kk.z;
      key[j + 3] = kk.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) key[j] = j < mine ? topk_key(ld_row1<COHERENT>(x + c0 + j)) : 0u;
  }
  bar_sync<NT>();  // histograms (and accumulators) zeroed
  if (multi) cluster_arrive();  // accumulators zeroed (waited for before the first push)
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (j < mine) atomicAdd(&h0[key[j] >> 21], 1u);
  bar_sync<NT>();
  if (multi) {
    cluster_wait();
    cluster_sum<NT>(h0, acc, h0, kBins, C);
  }
  // After each digit: when the bin holding the k-th largest key holds exactly
  // the keys still wanted, all of them are selected - the selection is every
  // key at or above the bin's lowest key - and no further digit is needed
  // (after 22 bits, the usual case).  The test reads the (cluster-summed)
  // histogram, so every thread and every CTA of a cluster takes the same
  // branch.  thr is then the bin's lowest key minus one (bins 0 excluded) and
  // no key equal to it is taken.
  int remaining = k;
  find_digit<NT>(sh, h0, kBins, remaining);
  bar_sync<NT>();
  const uint32_t d0 = (uint32_t)sh.digit;
  remaining -= sh.above;
  uint32_t thr;
  if (sh.equal == remaining && d0 != 0u) {
    thr = (d0 << 21) - 1u;
    remaining = 0;
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (j < mine && (key[j] >> 21) == d0) atomicAdd(&h1[(key[j] >> 10) & 2047u], 1u);
    bar_sync<NT>();  // every thread has read sh for d0; h1 complete
    if (multi) cluster_sum<NT>(h1, acc + kBins, h1, kBins, C);
    find_digit<NT>(sh, h1, kBins, remaining);
    bar_sync<NT>();
    const uint32_t p22 = (d0 << 11) | (uint32_t)sh.digit;
    remaining -= sh.above;
    if (sh.equal == remaining && p22 != 0u) {
      thr = (p22 << 10) - 1u;
      remaining = 0;
    } else {
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (j < mine && (key[j] >> 10) == p22) atomicAdd(&h2[key[j] & 1023u], 1u);
      bar_sync<NT>();
      if (multi) cluster_sum<NT>(h2, acc + 2 * kBins, h2, 1024, C);
      find_digit<NT>(sh, h2, 1024, remaining);
      bar_sync<NT>();
      // the k-th largest key; of the keys equal to it the `remaining` lowest columns are kept
      thr = (p22 << 10) | (uint32_t)sh.digit;
      remaining -= sh.above;
    }
  }
  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    gt += (int)(j < mine && key[j] > thr);
    eq += (int)(j < mine && key[j] == thr);
  }
  // exclusive scan of (above << 16 | equal): both totals stay below 2^16
  int tot;
  const int ex = block_excl_sum<NT>((gt << 16) | eq, sh.warp_tot, &tot);
  const int gt_before = ex >> 16, eq_before = ex & 0xFFFF;
  // the CTAs before this one in the cluster: keys above the threshold, keys equal to it
  int gt_ctas = 0, eq_ctas = 0;
  if (multi) {
    cg::cluster_group cl = cg::this_cluster();
    if (tid == 0) {
      sh.cta_gt = tot >> 16;
      sh.cta_eq = tot & 0xFFFF;
    }
    cl.sync();
    int qg = 0, qe = 0;
    if (lane < part) {  // part < C <= 8
      qg = *cl.map_shared_rank(&sh.cta_gt, lane);
      qe = *cl.map_shared_rank(&sh.cta_eq, lane);
    }
    __syncwarp();
    cluster_arrive();  // done with remote shared memory (waited for before exit)
    gt_ctas = __reduce_add_sync(0xFFFFFFFFu, qg);
    eq_ctas = __reduce_add_sync(0xFFFFFFFFu, qe);
  }
  // selected columns before this thread's: every larger key, and of the equal
  // keys (row order) the first `remaining`
  int pos = gt_ctas + gt_before + min(eq_ctas + eq_before, remaining);
  int eq_rank = eq_ctas + eq_before;
  int32_t* o = task.out;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const bool is_eq = j < mine && key[j] == thr;
    const bool take = (j < mine && key[j] > thr) || (is_eq && eq_rank < remaining);
    eq_rank += (int)is_eq;
    if (take) {
      if (pos < k) o[pos] = CAND ? ccol[cidx[CAND ? j : 0]] : s0 + c0 + j;
      ++pos;
    }
  }
  // no CTA leaves while another may still read its shared memory
  if (multi) {
    __syncwarp();
    cluster_wait();
  }
}

// ---- sampled-pivot selection -------------------------------------------------
// A row one CTA selects alone, longer than its keys-in-registers limit, with
// k well below its length (the long prefill and MTP rows):
//  1. A sample - every 8th block of 128 columns, or sparser for rows so long
//     that the sample would not fit the candidate slices - gives a threshold T below
//     the row's k-th largest key with a wide margin: the lower edge of the
//     22-bit key bin holding the sample's j-th largest key, j the k-th
//     place scaled to the sample plus four standard deviations and 16.
//  2. One pass over the row (each warp a contiguous segment, each lane 16
//     consecutive columns a step) writes the columns at or above T, and
//     their keys, into the warp's own slices of shared memory, in column
//     order (a lane's offset from one scan of its candidate count, its stores
//     one per set bit).
//  3. The exact selection runs on the candidates alone, keys in registers
//     (select_row_reg reading the warps' slices in order), and writes the
//     selected candidates' columns.  (Reading each candidate's logit again
//     from L2 instead cost ~5 us a row.)
// It gives up - the caller then runs the full path - when fewer than k
// columns reach T (every selected key must be a candidate) or a warp's slice
// overflows; the decisions read shared values, so every thread takes the
// same one.  Shared memory at `dyn`: the three histograms (kRegHistWords),
// then per warp `wcap` candidate columns, then per warp `wcap` their keys.

// The smallest float whose key (topk_key) is at least tk, for the compare
// x >= T on floats: -inf below every finite key, NaN above them (no float
// compares >= NaN).
__device__ __forceinline__ float key_floor_float(uint32_t tk) {
  if (tk <= 0x007FFFFFu) return -INFINITY;
  if (tk & 0x80000000u) return __uint_as_float(tk & 0x7FFFFFFFu);
  return __uint_as_float(~tk);
}

constexpr int kSampleEvery = 8;  // sampled blocks of kSeg columns: one in kSampleEvery
constexpr int kLaneCols = 16;    // consecutive columns a lane covers per step of the pivot pass

template <int NT, bool COHERENT, int KPT>
__device__ __forceinline__ bool select_row_pivot(const RowTask& task, const Config& cf, uint32_t* dyn, Shared& sh) {
  constexpr int kW = NT / 32;
  const int tid = (int)threadIdx.x, lane = lane_id(), warp = tid >> 5;
  const int n = task.n, k = cf.k;
  const int wcap = (cf.pcap / kW) & ~3;  // candidate slots of a warp
  const float* x = task.row;
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  uint32_t* h0 = dyn;
  uint32_t* h1 = h0 + kBins;
  int32_t* scol = reinterpret_cast<int32_t*>(dyn + kRegHistWords) + warp * wcap;  // this warp's slice
  uint32_t* skey = dyn + kRegHistWords + kW * wcap + warp * wcap;                  // and its keys
  // four columns c..c+3 (c a multiple of 4) up to `end`; past it NaN, which
  // compares false with every threshold
  auto load4 = [&](int c, int end) -> float4 {
    if (vec && c + 4 <= end) return ld_row4<COHERENT>(x + c);
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = c + u < end ? ld_row1<COHERENT>(x + c + u) : __uint_as_float(0x7FC00000u);
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  const int nblk = (n + kSeg - 1) / kSeg;
  // one block in `every` (more than kSampleEvery for rows whose sample would
  // not fit the candidate slices, where it is kept)
  const int maxblk = max(1, kW * wcap / kSeg);
  const int every = max(kSampleEvery, (nblk + maxblk - 1) / maxblk);
  const int nsb = (nblk + every - 1) / every;  // sampled blocks
  const int last = (nsb - 1) * every;
  const int S = (nsb - 1) * kSeg + min(kSeg, n - last * kSeg);  // sampled columns
  const double r = (double)k * S / n;
  const int64_t jj = (int64_t)ceil(r + 4.0 * sqrt(r) + 16.0);
  if (jj > S || wcap < 4) return false;  // nothing written yet; the same in every thread
  const int j = (int)jj;
  // the whole row streams into L2 at once (16 KB bulk prefetches of its
  // 16-byte aligned part) while the sample is read; both passes then read L2
  if (tid == 0 && vec) {
    const int n4 = n & ~3;
    for (int c = 0; c < n4; c += kChunk) ptx::bulk_prefetch_l2(x + c, 4u * (uint32_t)min(kChunk, n4 - c));
  }
  for (int i = tid; i < 2 * kBins; i += NT) h0[i] = 0;
  bar_sync<NT>();  // histograms zeroed
  // (1) sample histogram of the top 11 bits (warp w takes sampled blocks w,
  // w + kW, ... four at a time; the keys stay in shared memory, in the
  // candidate slices the main pass fills later), then of the next 11 in d0's
  // bin from the kept keys
  uint32_t* skeep = dyn + kRegHistWords;  // sample key i at skeep[i]: block i / kSeg, column 4 lane + e
  for (int b0 = warp * every; b0 < nblk; b0 += 4 * kW * every) {
    float4 f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + u * kW * every;
      f[u] = b < nblk ? load4(b * kSeg + 4 * lane, n) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + u * kW * every;
      if (b >= nblk) break;
      const int c = b * kSeg + 4 * lane;
      const uint4 kk = keys4(f[u]);
      *reinterpret_cast<uint4*>(skeep + (b / every) * kSeg + 4 * lane) = kk;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c + e < n) atomicAdd(&h0[lane_of(kk, e) >> 21], 1u);
    }
  }
  bar_sync<NT>();
  find_digit<NT>(sh, h0, kBins, j);
  bar_sync<NT>();
  const uint32_t d0 = (uint32_t)sh.digit;
  const int j1 = j - sh.above;
  for (int i = tid; i < nsb * kSeg; i += NT) {
    const int c = (i / kSeg) * every * kSeg + (i % kSeg);  // the row column of sample key i
    const uint32_t key = skeep[i];
    if (c < n && (key >> 21) == d0) atomicAdd(&h1[(key >> 10) & 2047u], 1u);
  }
  bar_sync<NT>();
  find_digit<NT>(sh, h1, kBins, j1);
  bar_sync<NT>();
  const float T = key_floor_float((d0 << 21) | ((uint32_t)sh.digit << 10));
  // (2) the columns >= T, per warp in column order
  constexpr int kWarpStep = 32 * kLaneCols;
  const int wseg = (n + kW * kWarpStep - 1) / (kW * kWarpStep) * kWarpStep;
  const int w0 = min(n, warp * wseg), w1 = min(n, w0 + wseg);
  int ncw = 0;  // this warp's candidates (warp-uniform)
  for (int c0 = w0; c0 < w1; c0 += kWarpStep) {  // warp-uniform trip count
    const int c = c0 + kLaneCols * lane;
    float4 f[kLaneCols / 4];
#pragma unroll
    for (int u = 0; u < kLaneCols / 4; ++u) f[u] = load4(c + 4 * u, w1);
    uint32_t m = 0;  // bit i: column c + i is a candidate
#pragma unroll
    for (int u = 0; u < kLaneCols / 4; ++u)
      m |= (uint32_t)(f[u].x >= T) << (4 * u) | (uint32_t)(f[u].y >= T) << (4 * u + 1) |
           (uint32_t)(f[u].z >= T) << (4 * u + 2) | (uint32_t)(f[u].w >= T) << (4 * u + 3);
    const int nc = __popc(m);
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    int pos = ncw + incl - nc;
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1u;
      if (pos < wcap) {
        // the value at column c + i, picked by selects (no indexed registers)
        const float4 fv = (i >> 2) == 0 ? f[0] : ((i >> 2) == 1 ? f[1] : ((i >> 2) == 2 ? f[2] : f[3]));
        const float val = (i & 3) == 0 ? fv.x : ((i & 3) == 1 ? fv.y : ((i & 3) == 2 ? fv.z : fv.w));
        scol[pos] = c + i;
        skey[pos] = topk_key(val);
      }
      ++pos;
    }
    ncw += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) sh.wgt[warp] = ncw;
  bar_sync<NT>();
  // exclusive prefix of the warps' counts (every warp computes it), the total
  int wc = lane < kW ? sh.wgt[lane] : 0, wi = wc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
    if (lane >= o) wi += t;
  }
  const int M = __shfl_sync(0xFFFFFFFFu, wi, 31);
  const bool over = __any_sync(0xFFFFFFFFu, wc > wcap);
  if (warp == 0 && lane < kW) sh.weq[lane] = wi - wc;  // slice base of warp `lane` in the candidate order
  bar_sync<NT>();
  if (M < k || over) return false;  // every thread has read the counts (barrier above)
  const RowTask ctask{task.row, M, task.out};
  const int32_t* cc = reinterpret_cast<const int32_t*>(dyn + kRegHistWords);
  if (KPT > 8 && M <= NT * 8)  // the same in every thread
    select_row_reg<NT, (KPT > 8 ? 8 : KPT), COHERENT, false, true>(ctask, cf, dyn, sh, 1, 0, cc, wcap);
  else
    select_row_reg<NT, KPT, COHERENT, false, true>(ctask, cf, dyn, sh, 1, 0, cc, wcap);
  return true;
}

// Selects one row.  Called by threads [0, NT) of the CTA (every one of them,
// with the same arguments); in a cluster (CLUSTER, CL > 1 CTAs) by every CTA,
// `rank` being this CTA's.  Dynamic shared memory `dyn` (16-byte aligned,
// smem_bytes(NT, cap, cpw, CLUSTER) bytes):
//   cache [cap] | candidate lists [NT/32][cpw] | hist [kBins]
//   | cluster only: accumulators [kAccWords]
// COHERENT: the logits were written by other CTAs of the running kernel
// (plain loads coherent at L2; cf.bulk must be 0).  KPT > 0: a row one CTA
// selects alone and that has at most NT * KPT columns takes select_row_reg
// (`dyn` must then hold kRegHistWords words, kRegHistWords + kAccWords in a
// cluster).  The caller separates
// two calls on the same shared memory with a barrier of the NT threads.
template <int NT, bool CLUSTER, bool COHERENT, int KPT = 0>
__device__ __forceinline__ void select_row(const RowTask& task, const Config& cf, uint32_t* dyn, Shared& sh,
                                           int CL, int rank) {
  constexpr int kW = NT / 32;
  const int tid = (int)threadIdx.x;
  uint32_t* cache = dyn;  // floats as copied, keys after pass 1
  int32_t* cand = reinterpret_cast<int32_t*>(cache + cf.cap);
  uint32_t* hist = reinterpret_cast<uint32_t*>(cand + kW * cf.cpw);
  // cluster: per-digit accumulators of this CTA's bins (2048, 2048, 1024); the
  // summed histogram overwrites the local one, which is pushed by then
  uint32_t* acc = hist + kBins;
  uint32_t* tot = hist;

  const int lane = lane_id(), warp = tid >> 5;
  const int k = cf.k;
  int32_t* o = task.out;
  const int n = task.n;
  if (n <= k) {  // the same for every CTA of the cluster: no cluster barrier is pending
    if (rank == 0)
      for (int i = tid; i < k; i += NT) o[i] = i < n ? i : -1;
    return;
  }
  // A row of at most kSoloMax columns is done by the cluster's first CTA
  // alone (measured faster than any exchange), the others leave at once;
  // the decision depends on the row only, so it is the same in every CTA.
  const bool multi = CLUSTER && n > kSoloMax;
  if (CLUSTER && !multi && rank != 0) return;
  if (KPT > 0) {  // segments of at most NT * KPT columns: keys in registers
    constexpr int K4 = KPT > 0 ? KPT : 4;
    if (!multi && n <= NT * KPT) {  // one CTA (its own instantiation: no cluster code in it)
      select_row_reg<NT, K4, COHERENT, false>(task, cf, dyn, sh, 1, 0);
      return;
    }
    if (multi && (((n + CL - 1) / CL + 3) & ~3) <= NT * KPT) {  // the same in every CTA of the cluster
      select_row_reg<NT, K4, COHERENT, CLUSTER>(task, cf, dyn, sh, CL, rank);
      return;
    }
    // one CTA, a longer row: the sampled pivot, unless it gives up
    if (!multi && cf.pcap >= cf.k && select_row_pivot<NT, COHERENT, K4>(task, cf, dyn, sh)) return;
  }
  const int C = multi ? CL : 1;
  const int part = multi ? rank : 0;
  // this CTA's segment [s0, s0 + len) of the row; boundaries on multiples of 4
  const int per_cta = ((n + C - 1) / C + 3) & ~3;
  const int s0 = min(n, part * per_cta);
  const int len = min(n, s0 + per_cta) - s0;
  const float* x = task.row + s0;
  const int nc4 = min(len, cf.cap) & ~3;
  const int nchunks = cf.bulk ? (nc4 + kChunk - 1) / kChunk : 0;
  const Segment<COHERENT> seg{x, cache, ptx::smem_u32(cache), len, nc4,
                              (reinterpret_cast<uintptr_t>(x) & 15u) == 0};

  for (int i = tid; i < kBins; i += NT) hist[i] = 0;
  if (multi)
    for (int i = tid; i < kAccWords; i += NT) acc[i] = 0;
  if (tid == 0) {
    for (int i = 0; i < nchunks; ++i) ptx::mbar_init(&sh.bar[i], 1);
    sh.timed_out = 0;
    sh.overflow = 0;
    ptx::fence_mbar_init();
  }
  if (tid < kW) sh.weq[tid] = 0;
  bar_sync<NT>();  // barriers initialised, histogram zeroed
  if (multi) cluster_arrive();  // accumulators zeroed (waited for before the first push)
  if (tid == 0) {
    const uint64_t policy = ptx::policy_evict_first();  // each logit is read by one CTA
    for (int i = 0; i < nchunks; ++i) {
      const uint32_t bytes = 4u * (uint32_t)min(kChunk, nc4 - i * kChunk);
      ptx::mbar_arrive_expect_tx(&sh.bar[i], bytes);
      ptx::bulk_load(cache + (int64_t)i * kChunk, x + (int64_t)i * kChunk, bytes, &sh.bar[i], policy);
    }
  }

  // ---- pass 1: keys in place, histogram of the top 11 bits
  if (!cf.bulk) {
    // plain loads, kBatch groups of 4 columns in flight per thread; the keys
    // of the cached columns go to the cache
    constexpr int kBatch = 4;
    for (int c0 = 4 * tid; c0 < len; c0 += 4 * NT * kBatch) {
      uint4 kk[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int c = c0 + u * 4 * NT;
        kk[u] = make_uint4(0u, 0u, 0u, 0u);
        if (c < len) {
          if (seg.vec && c + 4 <= len) {
            kk[u] = keys4(ld_row4<COHERENT>(x + c));
          } else {
            uint32_t v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = c + e < len ? topk_key(ld_row1<COHERENT>(x + c + e)) : 0u;
            kk[u] = make_uint4(v[0], v[1], v[2], v[3]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int c = c0 + u * 4 * NT;
        if (c >= len) break;
        if (c + 4 <= nc4) sts128(seg.cache_s + 4u * (uint32_t)c, kk[u]);
        if (c + 4 <= len) {
          atomicAdd(&hist[kk[u].x >> 21], 1u);
          atomicAdd(&hist[kk[u].y >> 21], 1u);
          atomicAdd(&hist[kk[u].z >> 21], 1u);
          atomicAdd(&hist[kk[u].w >> 21], 1u);
        } else {
#pragma unroll
          for (int e = 0; e < 3; ++e)
            if (c + e < len) atomicAdd(&hist[lane_of(kk[u], e) >> 21], 1u);
        }
      }
    }
  } else {
    int ready = -1;
    for (int c = 4 * tid; c < len; c += 4 * NT) {
      uint4 kk;
      if (c + 4 <= nc4) {
        const int ch = c / kChunk;
        while (ready < ch && ready + 1 < nchunks) {
          ++ready;
          if (!ptx::mbar_try_wait(&sh.bar[ready], 0)) {
            const long long t0 = clock64();
            bool ok = false;
            while (!(ok = ptx::mbar_try_wait(&sh.bar[ready], 0)) && clock64() - t0 < kSpinCycles) {
            }
            if (!ok) {
              sh.timed_out = 1;
              atomicOr(cf.fault, 2u);
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
  bar_sync<NT>();  // keys cached, histogram complete
  int remaining = k;
  const uint32_t* H = hist;
  if (multi) {
    cluster_wait();
    cluster_sum<NT>(hist, acc, tot, kBins, C);
    H = tot;
  }
  find_digit<NT>(sh, H, kBins, remaining);
  bar_sync<NT>();
  const uint32_t d0 = (uint32_t)sh.digit;
  remaining -= sh.above;
  bar_sync<NT>();  // digit read; the local histogram is free again
  for (int i = tid; i < kBins; i += NT) hist[i] = 0;
  bar_sync<NT>();

  // ---- pass 2 (ordered, warp-contiguous): keys above bin d0 per warp, and
  // the candidates of bin d0 into the warp's list with a histogram of their
  // next 11 bits
  const int wseg = (len + kW * kSeg - 1) / (kW * kSeg) * kSeg;
  const int w0 = warp * wseg, w1 = min(len, w0 + wseg);
  const unsigned lt = (1u << lane) - 1u;
  int32_t* wl = cand + warp * cf.cpw;  // this warp's candidate columns
  int ncw = 0;                         // candidates of this warp (warp-uniform)
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
            if (pos < cf.cpw) wl[pos] = c + u;
            ++pos;
            atomicAdd(&hist[(lane_of(kk, u) >> 10) & 2047u], 1u);
          }
        ncw += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    gt0 = __reduce_add_sync(0xFFFFFFFFu, gt0);
    if (lane == 0) {
      sh.wgt[warp] = gt0;
      if (ncw > cf.cpw) sh.overflow = 1;
    }
  }
  bar_sync<NT>();
  const bool overflow = sh.overflow != 0;
  H = hist;
  if (multi) {
    cluster_sum<NT>(hist, acc + kBins, tot, kBins, C);
    H = tot;
  }
  find_digit<NT>(sh, H, kBins, remaining);
  bar_sync<NT>();
  const uint32_t p22 = (d0 << 11) | (uint32_t)sh.digit;
  remaining -= sh.above;
  bar_sync<NT>();
  for (int i = tid; i < 1024; i += NT) hist[i] = 0;
  bar_sync<NT>();

  // ---- pass 3: low 10 bits of the candidates whose top 22 bits are p22
  if (!overflow) {
    for (int i = lane; i < ncw; i += 32) {
      const uint32_t key = seg.get1(wl[i]);
      if ((key >> 10) == p22) atomicAdd(&hist[key & 1023u], 1u);
    }
  } else {
    for (int c = 4 * tid; c < len; c += 4 * NT) {
      const uint4 kk = seg.get4(c);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + u < len && (lane_of(kk, u) >> 10) == p22) atomicAdd(&hist[lane_of(kk, u) & 1023u], 1u);
    }
  }
  bar_sync<NT>();
  H = hist;
  if (multi) {
    cluster_sum<NT>(hist, acc + 2 * kBins, tot, 1024, C);
    H = tot;
  }
  find_digit<NT>(sh, H, 1024, remaining);
  bar_sync<NT>();
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
  bar_sync<NT>();

  // ---- first output slot of every warp
  const int g = lane < kW ? sh.wgt[lane] : 0;
  const int e = lane < kW ? sh.weq[lane] : 0;
  int cta_base = 0, cta_eq_before = 0;
  if (multi) {
    cg::cluster_group cl = cg::this_cluster();
    const int gtot = __reduce_add_sync(0xFFFFFFFFu, g), etot = __reduce_add_sync(0xFFFFFFFFu, e);
    if (tid == 0) {
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
  if (sh.timed_out && tid == 0)
    for (int i = 0; i < nchunks; ++i) {
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(&sh.bar[i], 0) && clock64() - t0 < kSpinCycles) {
      }
    }
  // no CTA leaves while another may still read its shared memory
  __syncwarp();
  if (multi) cluster_wait();
}

}  // namespace sel
}  // namespace qsa
