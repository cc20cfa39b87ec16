// tcgen05 scorer: 128 keys in M, a request's rows x heads in N.
//
// The pages stack a request's rows x heads into the M dimension of one MFMA
// so a key tile is read once for all of them (ROCm/ATOM #2651 "Changes":
// BMT rows x heads = one 16-row tile, per-head ReLU before the head sum).  On
// sm_100-class tensor cores M is 128 wide, so here the roles swap: each tile
// of 128 consecutive key columns is the A operand (M = 128 lanes of TMEM, one
// key per lane) and the group's rows x heads are the B operand (N = 16..256,
// zero or don't-care padded).  The epilogue then owns one key per thread and
// reduces heads in registers, and its stores of one row are 32 consecutive
// floats per warp.
//
// Structure (one persistent CTA per SM, 16 warps; 15 in the converter form;
// two CTAs of 8 warps per SM in the lean form):
//  * schedule: every CTA derives, from the visible counts, the tile count of
//    each row group (tiles past the group's widest visible column are never
//    scheduled - the early exit of vLLM #62589 "Overview") and takes an equal
//    contiguous share of the flattened (group, tile) list, plus an equal share
//    of the pure -inf tail (columns past each group's last tile).  Up to 256
//    rows, warp 0 builds the schedule and loads its first block-table entries
//    while the previous kernel in the stream is still running (programmatic
//    dependent launch); keys, q and weights are read after it completes.
//  * warp 0 (TMA): per tile, lanes fetch the block-table entries of the tile's
//    pages and each issues the page's two 64-column K-halves as 3-D tensor
//    copies into a 128-byte-swizzled stage (aiter #4221 KVBlockSize>=1 commit:
//    block = table[b][col / page_cols], slot = col % page_cols).  A new group's
//    q is loaded by a 2-D tensor copy once the previous group's MMAs are done.
//  * warp 1 (MMA): the warp walks the tiles and an elected lane issues 8
//    tcgen05.mma (K = 16 each; 4 of K = 32 with fp8 q) per tile into one of
//    the TMEM accumulators, then commits the stage back to the producer.
//  * warps 2-13 (epilogue, three warps per TMEM lane quadrant, each taking
//    every third row block of the group): tcgen05.ld of the tile's columns,
//    per head ReLU * weight, head sum, +0.0, -inf past the row's visible
//    count, store.  Warps 14-15 write the -inf tail.
//  * converter form (fp8 keys, bf16 q): warps 2-9 are the epilogue in two sets
//    of four taking alternate tiles; warps 10-13 widen each e4m3 key row to
//    f16 (into TMEM, the MMA's A operand, or shared memory for N > 128) and
//    scale each group's q into f16; warp 14 is a second MMA warp, the two
//    taking alternate tiles.
//  * FUSE instantiations (qsa_paged_mqa_topk) then select the rows of the row
//    groups whose last tile this CTA stored (see "fused selection" below).
// Every barrier wait gives up after about a second, sets the device fault
// word (qsa_device_status) and lets the CTA drain and exit.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "qsa_internal.h"
#include "sm100_ptx.cuh"
#include "topk_select.cuh"

namespace qsa {
namespace umma {

constexpr int kKindBf16 = 0;                // bf16 keys, bf16 q
constexpr int kKindFp8Keys = 1;             // fp8 keys widened to f16 by converter warps, bf16 q scaled to f16
constexpr int kKindFp8Q = 2;                // fp8 keys, fp8 q: kind::f8f6f4 MMA
constexpr int kBM = 128;                    // keys per tile (MMA M)
constexpr int kHalfBytes = kBM * 128;       // one 64-element K-half of a bf16 key tile
constexpr int kTileBytes = 2 * kHalfBytes;  // 32 KB
// A bf16 key tile as the copies leave it: for each group of 8 keys, their
// 64-element K-half 0 (a 1 KB 128-byte-swizzle atom), then their K-half 1, so
// one copy moves whole keys (both halves of a page's rows) and the MMA reads
// K-half h of 8-key group i at h * 1024 + i * 2048.
constexpr uint32_t kBf16AtomStride = 2048;
constexpr int kFp8StageBytes = kBM * 128;  // 128 fp8 keys of 128 bytes
constexpr int kFp8ConvStages = 3;          // f16 operand stages in shared memory fed by the converter
constexpr int kFp8TmemStages = 4;          // ... or in TMEM (64 columns each)
constexpr int kFp8StageAlloc = kFp8StageBytes + 1024;  // + the block's 128 fp32 scales, 1024-aligned
constexpr int kScaleRing = 8;                          // per-tile scale slots (see the converter)
// fp8 q: the copies put each tile's key scales in their own slot of a ring (a
// slot per tile, reused kQ8Ring tiles later), so a key stage is free as soon
// as the MMA has read it; at most kQ8Ring - 2 key stages (see the producer).
constexpr int kQ8Ring = 10;
// Warp roles: 0 TMA, 1 MMA, then the epilogue warps (three per TMEM lane
// quadrant, or one with the fp8 -> f16 converter or in the lean form), then
// 8 converter warps (fp8 keys with bf16 q) or 2 spare warps that write the
// -inf tail (ptxas 13.0 for aarch64 hosts crashes on this kernel when no warps
// follow the epilogue).  The lean form (8 warps, at most 128 registers a
// thread and half an SM's shared memory) serves decode-sized groups: two of
// its CTAs fit an SM, so a call's CTAs are resident, with their schedule built
// and their first block-table entries loaded, while the kernel before them
// still runs, and stream keys the moment it completes.
template <bool CONV, bool LEAN = false>
struct Roles {
  static constexpr int kEpiWarps = CONV ? 8 : (LEAN ? 4 : 12);
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kConvWarps = CONV ? 4 : 2;
  // epilogue sets taking alternate tiles (the converter form's 64-head
  // epilogue at one warp a lane quadrant would pace its pipeline)
  static constexpr int kSets = CONV ? 2 : 1;
  static constexpr int kConvThreads = 32 * kConvWarps;
  // MMA warps: the converter form has a second one (the last warp), the two
  // taking alternate tiles so that one's barrier waits overlap the other's
  // MMAs (a tile there is only 8 x 32 cycles of tensor work)
  static constexpr int kMmaWarps = CONV ? 2 : 1;
  static constexpr int kThreads = 64 + kEpiThreads + kConvThreads + 32 * (kMmaWarps - 1);
};
constexpr long long kSpinCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr int kFastSchedRows = 256;              // up to this many rows one warp builds the schedule
constexpr int64_t kPrefetchLines = 8192;         // block-table lines warmed in L2 before the wait (1 MB)
constexpr int kMaxSmem = 232448;                 // 227 KB opt-in limit per CTA
constexpr int kLeanSmem = 115712;                // two CTAs an SM: 2 x (this + 1 KB reserved) <= 228 KB
constexpr int kLeanMaxN = 64;                    // lean form: groups of at most 64 rows x heads
// Fused selection: at most kFuseMaxGroups row groups (their counters live in
// the caller's workspace, the list of groups a CTA completed in shared memory).
constexpr int kFuseWords = 4 + kFuseMaxGroups;   // won count, claim key, claimed row, last flag; won groups
constexpr int kSelSharedBytes = 512;             // sel::Shared at the start of the stage area
constexpr int kFuseKeys = 16;                    // keys per thread of the register selection path
static_assert(sizeof(sel::Shared) <= kSelSharedBytes, "selection state must fit its slot");


struct UmmaParams {
  unsigned int* fault;    // device fault word: bit 0 set when a bounded wait gives up
  const uint8_t* scales;  // fp8: scale of (page, slot) at scales + page * scale_stride + 4 * slot
  int64_t scale_stride;
  const float* weights;
  const uint16_t* q;  // bf16 q, [row x head][128] (the converter form reads it for its scales)
  const int32_t* block_table;
  const int32_t* visible;
  const int32_t* next_n_lens;  // live rows per request, or null (all live)
  float* out;
  int64_t out_cols;
  int64_t capacity;
  int32_t num_rows, rows_per_req, num_heads, page_cols, max_pages, num_pages;
  int32_t group_rows, groups_per_req, num_groups, tiles_cap, box_rows;
  int32_t bpt_shift;  // log2(pages per 128-column tile) when page_cols < 128, else 0
  int32_t pc_shift;   // log2(page_cols) when page_cols is a power of two, else -1
  int32_t stream_out;  // logits far larger than L2: write them with evict-first stores
  int32_t keep_keys;   // several row groups reuse each key tile: keep keys in L2
  // fused selection (kernels instantiated with FUSE only)
  int32_t* topk_out;    // [num_rows][topk_k] selected columns
  uint32_t* fuse_sync;  // caller workspace: done[G] | cursor[G] | finished; zero between calls
  int32_t topk_k, topk_cap, topk_cpw, topk_pcap;
};

// Shared-memory layout of one CTA (byte offsets from a 1024-aligned base);
// computed on the host and passed in, so N and the stage count are runtime.
struct Layout {
  int32_t n;            // MMA N (rows x heads of a group, padded to 16..256)
  int32_t stages;       // TMA stages in flight (bf16 key tiles, or fp8 key tiles)
  int32_t stage_bytes;  // 32 KB (bf16 tile) or 16 KB (fp8 tile)
  int32_t a_stages;     // fp8: f16 operand stages written by the converter; bf16: 0
  int32_t a_tmem;       // fp8 with N <= 128: the widened keys (MMA operand A) in TMEM, not smem
  int32_t naccs;        // TMEM accumulators of N columns: 4 (converter form, N <= 64) or 2
  int32_t a_col;        // a_tmem: TMEM column of the first A stage (after the accumulators)
  int32_t tmem_cols;    // naccs x N (+ the A stages) columns, power of two >= 32
  uint32_t idesc;       // tcgen05 instruction descriptor for M = 128, this N
  int32_t a_off, b_off, ring_off, bar_off, misc_off, epi_off, sched_off, fuse_off, total;
};

inline Layout make_layout(int N, int groups, int kind, bool fused = false, bool lean = false) {
  const bool conv = kind == kKindFp8Keys, q8 = kind == kKindFp8Q;
  Layout L;
  L.n = N;
  // fp8 keys widened by the converter: into TMEM beside the accumulators
  // while they fit there (N <= 128), sparing shared memory 64 KB of traffic
  // a tile (the widened keys' stores and the MMA's reads of them)
  L.a_tmem = conv && N <= 128 ? 1 : 0;
  L.naccs = L.a_tmem && N <= 64 ? 4 : 2;
  L.a_col = L.naccs * N;
  L.tmem_cols = 32;  // allocated as a power of two
  while (L.tmem_cols < L.a_col + (L.a_tmem ? kFp8TmemStages * 64 : 0)) L.tmem_cols *= 2;
  // the converter form computes in f16 (widened keys, q scaled into f16)
  L.idesc = q8 ? ptx::idesc_e4m3_f32(kBM, N) : (conv ? ptx::idesc_f16_f32(kBM, N) : ptx::idesc_bf16_f32(kBM, N));
  // fp8 keys widened by the converter: the tile's scales ride in its stage
  L.stage_bytes = conv ? kFp8StageAlloc : (q8 ? kFp8StageBytes : kTileBytes);
  L.a_stages = conv ? (L.a_tmem ? kFp8TmemStages : kFp8ConvStages) : 0;
  const int a_bytes = L.a_tmem ? 0 : L.a_stages * kTileBytes;  // smem for the widened keys
  const int qbytes = N * (q8 ? 128 : 256);         // q: N rows of D elements
  const int nring = conv ? kScaleRing : (q8 ? kQ8Ring : 0);
  const int ring = nring * kBM * 4;
  const int tail = qbytes + ring + (2 * 8 + 2 * kFp8TmemStages + nring + 13) * 8 + 32 + 2 * 256 * 4 + 16 +
                   8 * (groups + 1) + (fused ? 16 + 4 * kFuseWords : 0);
  int st = ((lean ? kLeanSmem : kMaxSmem) - 1024 - tail - a_bytes) / L.stage_bytes;
  L.stages = st > 8 ? 8 : st;  // <= kQ8Ring - 2
  L.a_off = L.stages * L.stage_bytes;  // fp8 only: the converter's bf16 ring
  L.b_off = L.a_off + a_bytes;
  L.ring_off = L.b_off + qbytes;       // fp8 only: per-tile key scales
  L.bar_off = L.ring_off + ring;
  const int nbars = 2 * L.stages + 2 * L.a_stages + nring + 4 + 4 + 5;
  L.misc_off = L.bar_off + nbars * 8;           // tmem slot, abort flag
  L.epi_off = (L.misc_off + 16 + 15) & ~15;     // w_s[256], vis_s[256]
  L.sched_off = L.epi_off + 2 * 256 * 4 + 16;   // pref[G + 1], gmax[G]
  L.fuse_off = (L.sched_off + 8 * (groups + 1) + 15) & ~15;  // fused: kFuseWords ints
  L.total = 1024 + (fused ? L.fuse_off + 4 * kFuseWords : L.sched_off + 8 * (groups + 1));
  return L;
}

// Bounded wait on an mbarrier phase.  Returns false on abort or time-out.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* fault) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinCycles) {
      *abort_flag = 1;
      atomicOr(fault, 1u);
      return false;
    }
  }
}

// Largest g with pref[g] <= t (pref is non-decreasing, pref[0] = 0).
__device__ __forceinline__ int find_group(const int32_t* pref, int num_groups, int t) {
  int lo = 0, hi = num_groups;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Exclusive scan (one warp) of the per-group tile counts in pref[0..G), total
// in pref[G].
__device__ __forceinline__ void scan_tiles(int32_t* pref, int G, int lane) {
  const int per = (G + 31) / 32;
  const int lo = min(G, lane * per), hi = min(G, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += pref[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - s;
  for (int i = lo; i < hi; ++i) {
    const int t = pref[i];
    pref[i] = run;
    run += t;
  }
  if (lane == 31) pref[G] = incl;
}

__device__ __forceinline__ void epi_bar(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Two fp8 e4m3 codes (bytes 0 and 1, or 2 and 3, of w) -> f16x2, the lower
// code in the low half: the hardware conversion, exact (every e4m3 value,
// 2^-9 .. 448, is an f16).  The NaN codes S.1111.111 are not inputs of this
// path.
template <int HI>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  const uint16_t codes = (uint16_t)(HI ? (w >> 16) : (w & 0xFFFFu));
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// The converter form runs its MMA in f16 (the widened fp8 keys are exact
// there).  A q row-head (128 bf16 elements) enters as q * 2^-e, with e taken
// from its largest magnitude so that this lies in [2^14, 2^15): every bf16
// element at or above 2^-17 there (8 significant bits on f16's grid of
// 2^-24 and finer) is then an f16 exactly, and smaller ones, under 2^-31 of
// the largest, round at 2^-25.  The head's weight is multiplied by 2^e.
// Products with powers of two commute with fp32 rounding, so each head's
// term w * relu(s x) is the one the bf16 MMA gives, bit for bit, while 2^e w
// stays a normal fp32 number.  Rows of zeros, or with an infinity or NaN,
// take e = 0.
//
// e from the bit pattern of the largest magnitude (sign cleared), by integer
// arithmetic alone, so the converter (from its shared-memory copy of q) and
// the epilogue (from q in global memory) reach the same value.
__device__ __forceinline__ int q_row_exp(uint32_t amax_bits) {
  const uint32_t ex = amax_bits >> 7, mant = amax_bits & 0x7Fu;
  if (amax_bits == 0 || ex == 0xFFu) return 0;
  const int lg = ex != 0 ? (int)ex - 127 : (31 - __clz((int)mant)) - 133;  // floor(log2 |q|max)
  return lg - 14;
}

// 2^e as fp32, exactly, for e in [-149, 127].
__device__ __forceinline__ float pow2_exact(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}

// The head sum of one (row, key): sum over heads h of w[h] * relu(x[h]) in
// fp32, x[h] the accumulator bits x_of(h) (times sgn, +-1, for fp8 keys).
// Below 16 heads one chain of fmaf in head order.  From 16 heads four
// partial sums, of heads h = 0, 1, 2, 3 (mod 4), added as (s0 + s1) +
// (s2 + s3) so that a dependent chain is H / 4 long; they run as two pairs
// through packed fp32 FMAs (fma.rn.f32x2: one rounding a lane, as fmaf), the
// same arithmetic in half the instructions (ragged 32-head scoring
// 180 -> 165 us).  With fewer heads a pair chain measured no faster.  A zero
// sum is +0.0: every chain starts from +0.0, and in round-to-nearest a sum
// with +0.0 or an exact cancellation is +0.0.
template <int H, bool FP8, typename X>
__device__ __forceinline__ float head_sum(const float* w_row, const X& x_of, float sgn) {
  if constexpr (H < 16) {
    float s = 0.0f;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      float wh;
      if (H % 4 == 0) {  // weights four at a time
        const float4 w4 = reinterpret_cast<const float4*>(w_row)[h / 4];
        wh = (h & 3) == 0 ? w4.x : ((h & 3) == 1 ? w4.y : ((h & 3) == 2 ? w4.z : w4.w));
      } else {
        wh = w_row[h];
      }
      const float xv = FP8 ? sgn * __uint_as_float(x_of(h)) : __uint_as_float(x_of(h));
      s = fmaf(wh, relu_nan(xv), s);
    }
    return s;
  } else {
    const float2 sg = make_float2(sgn, sgn);
    float2 a = make_float2(0.0f, 0.0f), b = make_float2(0.0f, 0.0f);  // (s0, s1), (s2, s3)
#pragma unroll
    for (int h = 0; h < H; h += 4) {
      const float4 w4 = reinterpret_cast<const float4*>(w_row)[h / 4];
      float2 x01 = make_float2(__uint_as_float(x_of(h)), __uint_as_float(x_of(h + 1)));
      float2 x23 = make_float2(__uint_as_float(x_of(h + 2)), __uint_as_float(x_of(h + 3)));
      if (FP8) {
        x01 = __fmul2_rn(sg, x01);
        x23 = __fmul2_rn(sg, x23);
      }
      a = __ffma2_rn(make_float2(w4.x, w4.y), make_float2(relu_nan(x01.x), relu_nan(x01.y)), a);
      b = __ffma2_rn(make_float2(w4.z, w4.w), make_float2(relu_nan(x23.x), relu_nan(x23.y)), b);
    }
    return (a.x + a.y) + (b.x + b.y);
  }
}

// Largest magnitude bit pattern of the 8 bf16 elements in v.
__device__ __forceinline__ uint32_t bf16x8_amax_bits(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

// The 8 bf16 elements of v times 2^s1 * 2^s2 (two exact steps: the scale
// 2^-e itself may exceed fp32's range), rounded to f16.
__device__ __forceinline__ uint4 bf16x8_scaled_to_f16(uint4 v, float s1, float s2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * s1 * s2;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * s1 * s2;
    const __half2 h = __floats2half2_rn(lo, hi);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The -inf tail: group g's columns [T_g * 128, out_cols) for its rows, where
// T_g is its scheduled tile count.  The CTA takes a contiguous slice of all
// groups' tail tiles (flattened group-major) and writes each group's part as
// plain row ranges, 16-byte streaming stores when rows are 16-byte aligned.
template <int kNT>
__device__ __forceinline__ void fill_tail(const UmmaParams& p, const int32_t* pref, int G, int total, int tid) {
  const int64_t oc = p.out_cols;
  const int64_t Tc = p.tiles_cap;
  const int64_t F = (int64_t)G * Tc - total;
  int64_t f = F * blockIdx.x / gridDim.x;
  const int64_t f1 = F * (blockIdx.x + 1) / gridDim.x;
  if (f >= f1) return;
  // fill prefix fp(g) = g * Tc - pref[g] is non-decreasing; find the group of f
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)mid * Tc - pref[mid] <= f) lo = mid;
    else hi = mid;
  }
  const bool vec = (oc & 3) == 0 && (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
  const float4 ninf4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  for (int g = lo; f < f1 && g < G; ++g) {
    const int64_t fpg = (int64_t)g * Tc - pref[g];
    const int Tg = pref[g + 1] - pref[g];
    const int64_t fe = min(f1, fpg + (Tc - Tg));
    if (f >= fe) continue;
    const int64_t ca = (Tg + (f - fpg)) * kBM;
    const int64_t cb = min((Tg + (fe - fpg)) * kBM, oc);
    f = fe;
    if (ca >= cb) continue;
    const int jj = g % p.groups_per_req;
    const int64_t r0 = (int64_t)(g / p.groups_per_req) * p.rows_per_req + jj * p.group_rows;
    const int nr = min(p.group_rows, p.rows_per_req - jj * p.group_rows);
    for (int j = 0; j < nr; ++j) {
      float* o = p.out + (r0 + j) * oc;
      if (vec) {
        for (int64_t cc = ca + 4 * tid; cc < cb; cc += 4 * kNT) __stcs(reinterpret_cast<float4*>(o + cc), ninf4);
      } else {
        for (int64_t cc = ca + tid; cc < cb; cc += kNT) __stcs(o + cc, -INFINITY);
      }
    }
  }
}

// ---- fused selection -------------------------------------------------------
// Every CTA counts, per row group, the tiles whose logits it has stored
// (done[g], a release); the CTA whose count completes a group (an acquire)
// has every logit of the group's rows behind it and selects them once its own
// tiles are done.  Groups of one row: that is all, and the completing CTA
// puts the count back to zero.  Groups of several rows: the completing CTA
// selects row 0 and then takes rows from cursor[g]; the other CTAs that
// scored the group wait for it to complete (a bounded wait: a CTA that gives
// up leaves its rows to the others, never a row unselected) and take rows
// too; the last CTA to finish zeroes the counters.  Groups without tiles (no
// row sees a column) select nothing and need no logits.

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

constexpr long long kHelpSpinCycles = 200000;  // ~0.1 ms: a helper's wait for a group to complete

// The epilogue has stored `run` tiles of group g: add them to the group's
// count (one thread, after a barrier of the epilogue threads, so the count is
// a release of all of their stores) and record the group when it completes.
__device__ __forceinline__ void fuse_close(const UmmaParams& p, const int32_t* pref, int g, int run, int et,
                                           int32_t* fz, int nthreads) {
  epi_bar(nthreads);
  if (et == 0) {
    const uint32_t T = (uint32_t)(pref[g + 1] - pref[g]);
    const uint32_t old = atom_add_acq_rel_gpu(p.fuse_sync + g, (uint32_t)run);
    if (old + (uint32_t)run == T) fz[4 + fz[0]++] = g;
  }
}

__device__ __forceinline__ int group_nrows(const UmmaParams& p, int g) {
  const int jj = g % p.groups_per_req;
  return min(p.group_rows, p.rows_per_req - jj * p.group_rows);
}

__device__ __forceinline__ int64_t group_row0(const UmmaParams& p, int g) {
  const int b = g / p.groups_per_req, jj = g - b * p.groups_per_req;
  return (int64_t)b * p.rows_per_req + (int64_t)jj * p.group_rows;
}

// Selection of the groups' rows by threads [0, NT) once the CTA's scoring is
// done; the stage area (`smem`, L.bar_off bytes, idle by now) holds the
// selection's shared memory.  [t_begin, t_end) are the CTA's tiles.
template <int NT>
__device__ __forceinline__ void fused_select(const UmmaParams& p, const int32_t* pref, int G, int t_begin,
                                             int t_end, uint8_t* smem, int32_t* fz) {
  const int tid = (int)threadIdx.x;
  const int k = p.topk_k;
  sel::Shared& sh = *reinterpret_cast<sel::Shared*>(smem);
  uint32_t* dyn = reinterpret_cast<uint32_t*>(smem + kSelSharedBytes);
  const sel::Config cf{k, p.topk_cap, p.topk_cpw, 0, p.fault, p.topk_pcap};
  uint32_t* done = p.fuse_sync;
  uint32_t* cursor = done + G;
  uint32_t* finished = done + 2 * G;
  // shared memory the tensor core and the copies used is written by plain stores now
  ptx::fence_proxy_async_smem();
  auto select = [&](int g, int j) {  // row j of group g
    const int64_t r = group_row0(p, g) + j;
    const int n = (int)row_visible(p.visible, p.next_n_lens, r, p.rows_per_req, p.capacity);
    const sel::RowTask task{p.out + r * p.out_cols, n, p.topk_out + r * k};
    sel::select_row<NT, false, true, kFuseKeys>(task, cf, dyn, sh, 1, 0);
    sel::bar_sync<NT>();
  };
  auto claim = [&](int g) -> int {  // next row of g nobody has taken (>= its row count: none)
    if (tid == 0) fz[2] = 1 + (int)atomicAdd(cursor + g, 1u);
    sel::bar_sync<NT>();
    const int j = fz[2];
    sel::bar_sync<NT>();
    return j;
  };

  // (0) groups without tiles: every row selects nothing
  for (int g = blockIdx.x; g < G; g += gridDim.x)
    if (pref[g + 1] == pref[g]) {
      int32_t* o = p.topk_out + group_row0(p, g) * k;
      for (int i = tid; i < group_nrows(p, g) * k; i += NT) o[i] = -1;
    }
  const bool multi = p.group_rows > 1;
  // (1) the groups this CTA completed
  const int nwon = fz[0];
  for (int w = 0; w < nwon; ++w) {
    const int g = fz[4 + w];
    if (!multi && tid == 0) done[g] = 0u;  // every count of the group is in: reset for the next call
    select(g, 0);
    const int nr = group_nrows(p, g);
    if (nr > 1)
      for (int j = claim(g); j < nr; j = claim(g)) select(g, j);
  }
  if (!multi) return;
  // (2) rows of the other groups this CTA scored, once they complete
  if (t_begin < t_end) {
    const int g1 = find_group(pref, G, t_end - 1);
    for (int g = find_group(pref, G, t_begin); g <= g1; ++g) {
      bool mine = false;
      for (int w = 0; w < nwon; ++w) mine |= fz[4 + w] == g;
      if (mine || group_nrows(p, g) < 2) continue;
      if (tid == 0) {
        const uint32_t T = (uint32_t)(pref[g + 1] - pref[g]);
        const long long t0 = clock64();
        bool ok;
        while (!(ok = ld_acquire_gpu(done + g) == T) && clock64() - t0 < kHelpSpinCycles) {
        }
        fz[1] = ok ? 1 : 0;
      }
      sel::bar_sync<NT>();
      const bool ready = fz[1] != 0;
      sel::bar_sync<NT>();
      if (!ready) continue;
      const int nr = group_nrows(p, g);
      for (int j = claim(g); j < nr; j = claim(g)) select(g, j);
    }
  }
  // (3) the last CTA out zeroes the counters
  if (tid == 0) fz[3] = atom_add_acq_rel_gpu(finished, 1u) == gridDim.x - 1 ? 1 : 0;
  sel::bar_sync<NT>();
  if (fz[3]) {
    for (int i = tid; i < 2 * G; i += NT) done[i] = 0u;
    if (tid == 0) *finished = 0u;
  }
}

template <int H, int KIND, bool FUSE, bool LEAN = false>
__global__ void __launch_bounds__(Roles<KIND == kKindFp8Keys, LEAN>::kThreads, LEAN ? 2 : 1)
    umma_score_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const UmmaParams p, const Layout L) {
  constexpr bool FP8 = KIND != kKindBf16;      // fp8 keys (+ per-key scales)
  constexpr bool CONV = KIND == kKindFp8Keys;  // widened to f16 by the converter warps
  constexpr bool Q8 = KIND == kKindFp8Q;       // fp8 q: e4m3 x e4m3 MMA on the copied keys
  static_assert(!LEAN || (!CONV && !FUSE), "the lean form has no converter and no fused selection");
  using R = Roles<CONV, LEAN>;
  constexpr int kThreads = R::kThreads;
  constexpr int kEpiThreads = R::kEpiThreads;
  extern __shared__ uint8_t smem_raw[];
  const int N = L.n;
  const int kStages = L.stages;
  const int kAStages = L.a_stages;
  // 1024-byte aligned base, by an offset from the shared-memory symbol (not an
  // integer round trip) so every pointer below is known to address shared memory
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* S = smem;                          // TMA stages
  uint8_t* A = CONV ? smem + L.a_off : smem;  // MMA A-operand stages (128-byte swizzle)
  uint8_t* Bq = smem + L.b_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kStages;
  uint64_t* afull = empty + kStages;          // fp8: converter -> MMA
  uint64_t* aempty = afull + kAStages;        // fp8: MMA -> converter
  uint64_t* sfull = aempty + kAStages;        // fp8: scales of a tile ready, one per scale slot
  uint64_t* tfull = sfull + (CONV ? kScaleRing : (Q8 ? kQ8Ring : 0));
  float* scale_ring = reinterpret_cast<float*>(smem + L.ring_off);  // fp8: [slots][128]
  uint64_t* tempty = tfull + 4;
  uint64_t* qfull = tempty + 4;
  uint64_t* qempty = qfull + 1;
  uint64_t* mma_done = qempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
  float* w_s = reinterpret_cast<float*>(smem + L.epi_off);
  int32_t* vis_s = reinterpret_cast<int32_t*>(w_s + 256);
  int32_t* pref = reinterpret_cast<int32_t*>(smem + L.sched_off);
  int32_t* gmax = pref + p.num_groups + 1;
  int32_t* fz = reinterpret_cast<int32_t*>(smem + L.fuse_off);  // FUSE: won groups and claim slots

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.num_groups;

  uint64_t* setup = mma_done + 1;  // one-warp schedule and TMEM allocation done
  uint64_t* qready = setup + 1;    // converter form: the group's q scaled into f16 in place
  // Few rows: warp 0 alone builds the schedule from visible counts it loads
  // first thing, and starts producing at once; the other warps wait on
  // `setup`.  Many rows: every thread takes part, with CTA barriers.
  const bool fast = p.num_rows <= kFastSchedRows;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      // freed by the converter (widened keys), or by the MMA
      ptx::mbar_init(&empty[s], CONV ? R::kConvThreads : 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      ptx::mbar_init(&afull[s], R::kConvThreads);
      ptx::mbar_init(&aempty[s], 1);
    }
    if (CONV)
      for (int s = 0; s < kScaleRing; ++s) ptx::mbar_init(&sfull[s], R::kConvThreads);
    if (Q8)
      for (int s = 0; s < kQ8Ring; ++s) ptx::mbar_init(&sfull[s], 1);
    for (int a = 0; a < L.naccs; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      // released by each thread of the set that read it (one arrival a warp
      // after __syncwarp measured slower: 422 against 413 us prefill scoring)
      ptx::mbar_init(&tempty[a], kEpiThreads / R::kSets);
    }
    ptx::mbar_init(qfull, 1);
    ptx::mbar_init(qempty, R::kMmaWarps);
    ptx::mbar_init(mma_done, R::kMmaWarps);
    ptx::mbar_init(setup, 2);
    ptx::mbar_init(qready, CONV ? R::kConvWarps : 1);
    *abort_flag = 0;
    if (FUSE) fz[0] = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&kv_map);
    ptx::prefetch_tmap(&q_map);
  }
  // Warm L2 with the visible counts and the block table (a share of their
  // 128-byte lines per CTA, at most kPrefetchLines in all) while the previous
  // kernel finishes.
  if (warp >= 2) {
    const int64_t vis_lines = ((int64_t)p.num_rows * 4 + 127) / 128;
    const int64_t bt_bytes = (int64_t)(p.num_rows / p.rows_per_req) * p.max_pages * 4;
    const int64_t bt_lines = min((bt_bytes + 127) / 128, kPrefetchLines);
    for (int64_t l = blockIdx.x + (int64_t)gridDim.x * (threadIdx.x - 64); l < vis_lines + bt_lines;
         l += (int64_t)gridDim.x * (kThreads - 64)) {
      const char* a = l < vis_lines ? reinterpret_cast<const char*>(p.visible) + l * 128
                                    : reinterpret_cast<const char*>(p.block_table) + (l - vis_lines) * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
  // Everything above overlaps the previous kernel in the stream.  Few rows:
  // warp 0 also loads the visible counts (and next_n_lens), builds the
  // schedule and loads its first block-table entries before it waits for that
  // kernel - none of the three may be written by it - and every other load,
  // and every store, comes after the wait.  Many rows: nothing is loaded
  // before the wait.
  if (!fast) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
  }
  int32_t vfast[kFastSchedRows / 32], nfast[kFastSchedRows / 32];
  if (fast && warp == 0) {
    // in-range address in every lane; rows past num_rows are masked at use, so
    // nothing waits for these loads until they are used
#pragma unroll
    for (int u = 0; u < kFastSchedRows / 32; ++u) {
      const int r = min(u * 32 + lane, p.num_rows - 1);
      vfast[u] = __ldg(p.visible + r);
      nfast[u] = p.next_n_lens != nullptr ? __ldg(p.next_n_lens + r / p.rows_per_req) : p.rows_per_req;
    }
  }
  if (!fast && warp == 1) {
    ptx::tmem_alloc(tmem_slot, (uint32_t)L.tmem_cols);
    ptx::tmem_relinquish();
  }
  if (!fast)
    for (int g = threadIdx.x; g < G; g += kThreads) gmax[g] = 0;
  __syncthreads();  // barriers initialised
  uint32_t tmem_base = 0;
  bool setup_ok = true;
  if (fast) {
    if (warp == 0) {
      for (int g = lane; g < G; g += 32) gmax[g] = 0;
      __syncwarp();
#pragma unroll
      for (int u = 0; u < kFastSchedRows / 32; ++u) {
        const int r = u * 32 + lane;
        const int b = r / p.rows_per_req, i = r - b * p.rows_per_req;
        const bool live = i < (int)clamp64(nfast[u], 0, p.rows_per_req);
        const int32_t vc = live ? (int32_t)clamp64(vfast[u], 0, p.capacity) : 0;
        if (r < p.num_rows && vc > 0) atomicMax(&gmax[b * p.groups_per_req + i / p.group_rows], vc);
      }
      __syncwarp();
      for (int g = lane; g < G; g += 32) pref[g] = (gmax[g] + kBM - 1) / kBM;
      __syncwarp();
      scan_tiles(pref, G, lane);
      __syncwarp();
      // warp 0 arrives on `setup` once its first copies are issued (below):
      // until then the other warps stay parked and leave it the issue slots
    } else {
      ptx::grid_dep_wait();
      ptx::grid_dep_launch();
      if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, (uint32_t)L.tmem_cols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(setup);
      }
      setup_ok = wait_phase(setup, 0, abort_flag, p.fault);
      ptx::tc_fence_after();
      tmem_base = *tmem_slot;
    }
  } else {
    // Per-group widest visible count and tile count from the visible counts
    // (device data, no host sync): every thread takes rows, four loads in flight.
    for (int r0 = 0; r0 < p.num_rows; r0 += 4 * kThreads) {
      int32_t v[4], nn[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = min(r0 + u * kThreads + (int)threadIdx.x, p.num_rows - 1);
        v[u] = __ldg(p.visible + r);
        nn[u] = p.next_n_lens != nullptr ? __ldg(p.next_n_lens + r / p.rows_per_req) : p.rows_per_req;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r0 + u * kThreads + threadIdx.x;
        const int b = r / p.rows_per_req, i = r - b * p.rows_per_req;
        const bool live = i < (int)clamp64(nn[u], 0, p.rows_per_req);
        const int32_t vc = live ? (int32_t)clamp64(v[u], 0, p.capacity) : 0;
        if (r < p.num_rows && vc > 0) atomicMax(&gmax[b * p.groups_per_req + i / p.group_rows], vc);
      }
    }
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += kThreads) pref[g] = (gmax[g] + kBM - 1) / kBM;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    tmem_base = *tmem_slot;
    if (warp == 0) scan_tiles(pref, G, lane);
    __syncthreads();
  }
  const int total = setup_ok ? pref[G] : 0;
  // equal shares, the first total % gridDim.x CTAs one tile more: they are
  // the first to be placed on SMs that the previous kernel has left
  const int t_share = total / (int)gridDim.x, t_extra = total % (int)gridDim.x;
  const int t_begin = (int)blockIdx.x * t_share + min((int)blockIdx.x, t_extra);
  const int t_end = t_begin + t_share + ((int)blockIdx.x < t_extra ? 1 : 0);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t policy = p.keep_keys ? ptx::policy_evict_last() : ptx::policy_evict_first();
    const int pc = p.page_cols;
    const int bsh = p.bpt_shift;
    const int bpt = 1 << bsh;                   // boxes (pages) per full tile, <= 16
    const int tiles_per_batch = 32 >> bsh;      // one box per lane per batch
    // page index and slot of column c (a power-of-two page size below 128
    // columns always; otherwise a 32-bit division)
    auto page_of = [&](int c) { return p.pc_shift >= 0 ? c >> p.pc_shift : c / pc; };
    auto req_of = [&](int g) { return p.groups_per_req == 1 ? g : g / p.groups_per_req; };
    const uint32_t box_bytes = (uint32_t)p.box_rows * (FP8 ? 128u : 256u);  // one copy per page (box)
    // Block-table entry of this lane's box in the batch starting at tile tb
    // (null: no box).  Lane l covers tile tb + l / bpt, box l % bpt.
    auto lane_entry = [&](int tb) -> const int32_t* {
      const int tl = tb + (lane >> bsh), box = lane & (bpt - 1);
      if (tl >= t_end) return nullptr;
      const int gl = find_group(pref, G, tl);
      const int c0 = (tl - pref[gl]) * kBM;
      const int lim = gmax[gl] - c0;
      const int nbox = pc >= kBM ? 1 : min(bpt, (lim + pc - 1) >> p.pc_shift);
      if (box >= nbox) return nullptr;
      const int lp = page_of(c0) + box;
      return p.block_table + (int64_t)req_of(gl) * p.max_pages + lp;
    };
    // Every lane loads from a valid address (the table's first entry when it
    // has no box) and nothing reads the value until its copy is issued, so
    // the load stays in flight while the current batch is issued.  (A select
    // on the loaded value would wait for it right here.)
    auto load_entry = [&](const int32_t* e) -> int32_t { return __ldg(e != nullptr ? e : p.block_table); };
    int stage = 0;
    uint32_t phase = 0;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int qg = -1;
    uint32_t q_loads = 0;
    uint32_t filled_mask = 0, last_phase_bits = 0;
    uint32_t sfilled_mask = 0, s_last_phase_bits = 0;  // fp8 q: scale slots with copies issued
    bool ok = true;
    bool released = !fast;  // fast schedule: `setup` not yet arrived on by this warp
    const int32_t* cur_e = t_begin < t_end ? lane_entry(t_begin) : nullptr;
    int32_t cur = load_entry(cur_e);
    if (fast) {  // the first table entries are in flight; keys and q only after the wait
      ptx::grid_dep_wait();
      ptx::grid_dep_launch();
    }
    for (int tb = t_begin; tb < t_end && ok; tb += tiles_per_batch) {
      // the next batch's block-table entries load while this batch is issued
      const int32_t* nxt_e = lane_entry(tb + tiles_per_batch);
      const int32_t nxt = load_entry(nxt_e);
      for (int i = 0; i < tiles_per_batch && tb + i < t_end; ++i) {
        const int t = tb + i;
        while (t >= pref[g + 1]) ++g;
        const int b = req_of(g), jj = g - b * p.groups_per_req;
        const int r0 = b * p.rows_per_req + jj * p.group_rows;
        const int c0 = (t - pref[g]) * kBM;
        const int lim = gmax[g] - c0;  // visible columns in this tile (>= 1)
        const int nbox = pc >= kBM ? 1 : min(bpt, (lim + pc - 1) >> p.pc_shift);
        if (g != qg) {
          if (q_loads > 0) ok = wait_phase(qempty, (q_loads - 1) & 1, abort_flag, p.fault);
          if (!ok) break;
          if (lane == 0) {
            if (Q8) {  // one 128-byte row (all of D) per row-head
              ptx::mbar_arrive_expect_tx(qfull, (uint32_t)N * 128u);
              ptx::tma_load_2d(Bq, &q_map, 0, r0 * H, qfull);
            } else {  // two 64-element K-halves
              ptx::mbar_arrive_expect_tx(qfull, 2u * N * 128u);
              ptx::tma_load_2d(Bq, &q_map, 0, r0 * H, qfull);
              ptx::tma_load_2d(Bq + N * 128, &q_map, 64, r0 * H, qfull);
            }
          }
          qg = g;
          ++q_loads;
        }
        ok = wait_phase(&empty[stage], phase ^ 1u, abort_flag, p.fault);
        if (!ok) break;
        // fp8 q: the tile's scale slot.  It is free: the stage wait above means
        // the MMA of tile rel - kStages is done, so the epilogue has released
        // the accumulator of tile rel - kStages - 2 and read every scale up to
        // that tile, and rel - kQ8Ring <= rel - kStages - 2.
        const int rel = t - t_begin;
        const int slot = Q8 ? rel % kQ8Ring : 0;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&full[stage], nbox * box_bytes + (CONV ? nbox * p.box_rows * 4u : 0u));
          if (Q8) ptx::mbar_arrive_expect_tx(&sfull[slot], nbox * p.box_rows * 4u);
        }
        __syncwarp();
        if ((lane >> bsh) == i && cur_e != nullptr) {
          const int32_t pg = cur < 0 ? 0 : (cur >= p.num_pages ? p.num_pages - 1 : cur);  // clamp: no fault
          const int box = lane & (bpt - 1);
          const int y = pc >= kBM ? c0 - page_of(c0) * pc : 0;
          uint8_t* dst = S + stage * L.stage_bytes + (uint32_t)box * (uint32_t)p.box_rows * (FP8 ? 128u : 256u);
          if (FP8) ptx::tma_load_3d(dst, &kv_map, 0, y, pg, &full[stage], policy);
          else ptx::tma_load_5d(dst, &kv_map, 0, 0, 0, y >> 3, pg, &full[stage], policy);
          // the box's scales (plain bulk copy: 16-byte aligned source,
          // destination and size) land after the key rows of the stage for
          // the converter, in the tile's scale slot with fp8 q
          if (CONV)
            ptx::bulk_load(S + stage * L.stage_bytes + kFp8StageBytes + box * p.box_rows * 4,
                           p.scales + (int64_t)pg * p.scale_stride + (int64_t)y * 4, (uint32_t)p.box_rows * 4u,
                           &full[stage], policy);
          if (Q8)
            ptx::bulk_load(scale_ring + slot * kBM + box * p.box_rows,
                           p.scales + (int64_t)pg * p.scale_stride + (int64_t)y * 4, (uint32_t)p.box_rows * 4u,
                           &sfull[slot], policy);
        }
        if (!released) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(setup);
          released = true;
        }
        filled_mask |= 1u << stage;
        last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
        if (Q8) {
          sfilled_mask |= 1u << slot;
          s_last_phase_bits = (s_last_phase_bits & ~(1u << slot)) | ((uint32_t)((rel / kQ8Ring) & 1) << slot);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      cur = nxt;
      cur_e = nxt_e;
    }
    if (!released && lane == 0) ptx::mbar_arrive(setup);  // no tile, or gave up before the first
    // Drain: every copy this warp issued has landed before the CTA tears down.
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < kStages; ++s)
        if (filled_mask & (1u << s)) {
          const long long t0 = clock64();
          while (!ptx::mbar_try_wait(&full[s], (last_phase_bits >> s) & 1u) && clock64() - t0 < kSpinCycles) {
          }
        }
      for (int s = 0; Q8 && s < kQ8Ring; ++s)
        if (sfilled_mask & (1u << s)) {
          const long long t0 = clock64();
          while (!ptx::mbar_try_wait(&sfull[s], (s_last_phase_bits >> s) & 1u) && clock64() - t0 < kSpinCycles) {
          }
        }
    }
  } else if (warp == 1 || (R::kMmaWarps > 1 && warp == 2 + R::kEpiWarps + R::kConvWarps)) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and one elected lane issues each tcgen05
    // instruction (the operands stay warp-uniform).  Waits are warp-wide: a
    // lane's failed wait ends the loop for every lane.  With two MMA warps,
    // warp mw issues the tiles with (t - t_begin) % 2 == mw; both follow the
    // group changes (each releases the q buffer for its own MMAs).
    const int mw = warp == 1 ? 0 : 1;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, p.fault));
    };
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int qg = -1;
    uint32_t q_uses = 0;
    const uint32_t a_base = ptx::smem_u32(A);
    const uint32_t b_base = ptx::smem_u32(Bq);
    bool ok = true;
    for (int t = t_begin; t < t_end && ok; ++t) {
      while (t >= pref[g + 1]) ++g;
      if (g != qg) {
        if (qg >= 0) ptx::mma_commit_elect(qempty);  // q buffer free once earlier MMAs finish
        ok = warp_wait(CONV ? qready : qfull, q_uses & 1u);
        if (!ok) break;
        ++q_uses;
        qg = g;
      }
      if (R::kMmaWarps > 1 && ((t - t_begin) & 1) != mw) {  // the other MMA warp's tile
        if (++stage == (CONV ? kAStages : kStages)) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == L.naccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
        continue;
      }
      ok = warp_wait(&tempty[acc], acc_phase ^ 1u) && warp_wait(CONV ? &afull[stage] : &full[stage], phase);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(acc * N);
      if (Q8) {
        // the fp8 key rows as copied: 128 bytes (all of D) a key, 4 MMAs of K = 32
        const uint32_t a0 = a_base + stage * (uint32_t)L.stage_bytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = ptx::sw128_desc(a0 + (uint32_t)k * 32u);
          const uint64_t bd = ptx::sw128_desc(b_base + (uint32_t)k * 32u);
          ptx::mma_e4m3_elect(d, ad, bd, L.idesc, k > 0 ? 1u : 0u);
        }
      } else if (CONV && L.a_tmem) {
        // the widened keys in TMEM: K elements 16k .. 16k + 15 of every
        // key row in columns 8k .. 8k + 7 of the stage
        const uint32_t at = tmem_base + (uint32_t)(L.a_col + stage * 64);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = ptx::sw128_desc(b_base + (k >> 2) * (N * 128) + (uint32_t)(k & 3) * 32u);
          ptx::mma_bf16_ts_elect(d, at + 8u * (uint32_t)k, bd, L.idesc, k > 0 ? 1u : 0u);
        }
      } else {
        const uint32_t a0 = a_base + stage * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (uint32_t)(k & 3) * 32u;
          // copied bf16 keys: halves interleaved per 8-key group; widened
          // fp8 keys in shared memory: one 16 KB block per K-half
          const uint64_t ad = CONV ? ptx::sw128_desc(a0 + (k >> 2) * kHalfBytes + koff)
                                   : ptx::sw128_desc(a0 + (k >> 2) * 1024u + koff, kBf16AtomStride);
          const uint64_t bd = ptx::sw128_desc(b_base + (k >> 2) * (N * 128) + koff);
          ptx::mma_bf16_elect(d, ad, bd, L.idesc, k > 0 ? 1u : 0u);
        }
      }
      ptx::mma_commit_elect(CONV ? &aempty[stage] : &empty[stage]);
      ptx::mma_commit_elect(&tfull[acc]);
      if (++stage == (CONV ? kAStages : kStages)) {
        stage = 0;
        phase ^= 1u;
      }
      if (++acc == L.naccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // every MMA issued above has completed before TMEM is released
    ptx::mma_commit_elect(mma_done);
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(mma_done, 0) && clock64() - t0 < kSpinCycles) {
    }
    __syncwarp();
  } else if (warp < 2 + R::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    constexpr int kSets = R::kSets;                      // sets taking alternate tiles
    constexpr int kHalves = R::kEpiWarps / (4 * kSets);  // a set's warps sharing one TMEM lane quadrant
    const int et = threadIdx.x - 64;                     // 0 .. kEpiThreads - 1
    const int quad = warp & 3;                           // TMEM lane quadrant this warp may access
    const int set = (warp - 2) / (4 * kHalves);          // this warp's set
    const int half = ((warp - 2) >> 2) % kHalves;        // which of the set's quadrant warps
    const int m = quad * 32 + lane;            // key row of the tile = TMEM lane
    const int64_t oc = p.out_cols;
    const bool stream_out = p.stream_out != 0;
    int32_t* const vis_min_s = vis_s + 256;  // smallest visible count of the group's rows

    // (1) computed tiles.  Column n of the accumulator is (row n / H, head
    // n % H).  A "unit" is the smallest run of 16-column TMEM loads that holds
    // whole rows: one load (16 / H rows) for H <= 16, H / 16 loads (one row)
    // for H > 16.  The warps of a quadrant take alternate units.
    constexpr int kRowsPerUnit = H >= 16 ? 1 : 16 / H;
    constexpr int kLdPerUnit = H >= 16 ? H / 16 : 1;
    constexpr int kUnitsPerBatch = 4 / kLdPerUnit;  // four loads in flight
    // tile i of the CTA: set i % kSets, accumulator i % naccs, in its
    // (i / naccs)-th use
    const int lg_accs = L.naccs == 4 ? 2 : 1;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int eg = -1, r0 = 0, nr = 0, b = 0;
    int run = 0;  // FUSE: tiles of group eg stored in this CTA's current run
    bool ok = true;
    // After a failed wait a thread keeps walking the tiles without work, so
    // every epilogue thread meets the same barriers at group changes.
    for (int t = t_begin; t < t_end; ++t) {
      while (t >= pref[g + 1]) ++g;
      if (g != eg) {
        if (FUSE && eg >= 0) fuse_close(p, pref, eg, run, et, fz, kEpiThreads);
        run = 0;
        epi_bar(kEpiThreads);
        b = g / p.groups_per_req;
        const int jj = g % p.groups_per_req;
        r0 = b * p.rows_per_req + jj * p.group_rows;
        nr = min(p.group_rows, p.rows_per_req - jj * p.group_rows);
        if (et == 0) *vis_min_s = INT32_MAX;
        for (int i = et; i < nr * H; i += kEpiThreads) {
          float w = p.weights[(int64_t)r0 * H + i];
          if (CONV) {
            // the row-head's q enters the f16 MMA as q * 2^-e: its weight
            // takes 2^e (e from q in global memory, as the converter found it)
            const uint4* qr = reinterpret_cast<const uint4*>(p.q + ((int64_t)r0 * H + i) * 128);
            uint32_t amax = 0;
#pragma unroll 4
            for (int j = 0; j < 16; ++j) amax = max(amax, bf16x8_amax_bits(__ldg(qr + j)));
            w *= pow2_exact(q_row_exp(amax));
          }
          w_s[i] = w;
        }
        epi_bar(kEpiThreads);
        for (int i = et; i < nr; i += kEpiThreads) {
          const int32_t v = (int32_t)row_visible(p.visible, p.next_n_lens, r0 + i, p.rows_per_req, p.capacity);
          vis_s[i] = v;
          atomicMin(vis_min_s, v);
        }
        epi_bar(kEpiThreads);
        eg = g;
      }
      ++run;
      if (!ok) continue;
      const int ti = t - t_begin;
      if (kSets > 1 && ti % kSets != set) continue;  // the other set's tile
      const int acc = ti & (L.naccs - 1);
      const uint32_t acc_phase = (uint32_t)(ti >> lg_accs) & 1u;
      const int tile_c0 = (t - pref[g]) * kBM;  // first column of the tile
      const int64_t c = (int64_t)tile_c0 + m;
      // every row of the group sees the whole tile: no mask, no bounds test
      const bool unmasked = (int64_t)tile_c0 + kBM <= min((int64_t)*vis_min_s, oc);
      // fp8: this key's dequantisation scale.  relu(s x) = |s| relu(sign(s) x)
      // for every s, so the sign goes inside the ReLU and |s| is applied once
      // per row after the head sum.
      float sgn = 1.0f, mag = 1.0f;
      if (CONV) {
        ok = wait_phase(&sfull[ti % kScaleRing], (uint32_t)(ti / kScaleRing) & 1u, abort_flag, p.fault);
        if (!ok) continue;
        const float sc = scale_ring[(ti % kScaleRing) * kBM + m];
        sgn = sc < 0.0f ? -1.0f : 1.0f;
        mag = fabsf(sc);
      } else if (Q8) {
        // the tile's scales, copied into their slot of the scale ring;
        // waiting on the slot's completed fill orders the copied bytes
        ok = wait_phase(&sfull[ti % kQ8Ring], (uint32_t)(ti / kQ8Ring) & 1u, abort_flag, p.fault);
        if (!ok) continue;
        const float sc = scale_ring[(ti % kQ8Ring) * kBM + m];
        sgn = sc < 0.0f ? -1.0f : 1.0f;
        mag = fabsf(sc);
      }
      ok = wait_phase(&tfull[acc], acc_phase, abort_flag, p.fault);
      if (!ok) continue;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * N);
      float* const ob = p.out + (int64_t)r0 * oc + c;  // row r0, this key's column
      const int nunits = H >= 16 ? nr : (nr + kRowsPerUnit - 1) / kRowsPerUnit;
      for (int u0 = half; u0 < nunits; u0 += kHalves * kUnitsPerBatch) {
        uint32_t v[4][16];
        // fewer than 16 heads (several rows a unit): when every unit of the
        // batch is present and whole and every row sees the whole tile, no
        // per-unit, per-row or per-column test (uniform; prefill scoring
        // 717 -> 480 us against the tested path below)
        const int ulast = u0 + kHalves * (kUnitsPerBatch - 1);
        const bool whole = H < 16 && unmasked && (ulast + 1) * kRowsPerUnit <= nr;
        if (whole) {
#pragma unroll
          for (int q = 0; q < kUnitsPerBatch; ++q)
#pragma unroll
            for (int l = 0; l < kLdPerUnit; ++l)
              ptx::tmem_ld16(tb + (uint32_t)(16 * ((u0 + kHalves * q) * kLdPerUnit + l)), v[q * kLdPerUnit + l]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < kUnitsPerBatch; ++q) {
            const int u = u0 + kHalves * q;
            float* const obu = ob + (int64_t)(u * kRowsPerUnit) * oc;
#pragma unroll
            for (int rr = 0; rr < kRowsPerUnit; ++rr) {
              const int j = u * kRowsPerUnit + rr;
              float part = head_sum<H, FP8>(
                  w_s + j * H,
                  [&](int h) { return H < 16 ? v[q][rr * H + h] : v[q * kLdPerUnit + h / 16][h % 16]; }, sgn);
              if (FP8) part = part * mag + 0.0f;  // +0.0 for zero: see the tested path
              float* const dst = obu + (int64_t)rr * oc;
              if (stream_out) __stcs(dst, part);
              else *dst = part;
            }
          }
          continue;
        }
#pragma unroll
        for (int q = 0; q < kUnitsPerBatch; ++q)
          if (u0 + kHalves * q < nunits)
#pragma unroll
            for (int l = 0; l < kLdPerUnit; ++l)
              ptx::tmem_ld16(tb + (uint32_t)(16 * ((u0 + kHalves * q) * kLdPerUnit + l)), v[q * kLdPerUnit + l]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < kUnitsPerBatch; ++q) {
          const int u = u0 + kHalves * q;
          if (u >= nunits) break;
          // the unit's first row; its rows are constant offsets from it
          float* const obu = ob + (int64_t)(u * kRowsPerUnit) * oc;
#pragma unroll
          for (int rr = 0; rr < kRowsPerUnit; ++rr) {
            const int j = u * kRowsPerUnit + rr;
            if (j >= nr) break;
            float part = head_sum<H, FP8>(
                w_s + j * H,
                [&](int h) { return H < 16 ? v[q][rr * H + h] : v[q * kLdPerUnit + h / 16][h % 16]; }, sgn);
            // a zero logit is +0.0 (head_sum's is), so only fp8's final
            // scale (|s| * a negative sum when s = 0) can make -0.0
            if (FP8) part = part * mag + 0.0f;
            float* const dst = obu + (int64_t)rr * oc;
            if (unmasked) {
              if (stream_out) __stcs(dst, part);
              else *dst = part;
            } else if (c < oc) {
              const float val = c < vis_s[j] ? part : -INFINITY;
              if (stream_out) __stcs(dst, val);
              else *dst = val;
            }
          }
        }
      }
      // this thread's loads are done (tcgen05.wait::ld above) and fenced
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
    }
    if (FUSE && eg >= 0) fuse_close(p, pref, eg, run, et, fz, kEpiThreads);

    // (2) fp8: this CTA's share of the -inf tail, after its tiles (the
    // converter warps are busy until then).  bf16: the spare warps write it.
    if (CONV && ok && setup_ok) fill_tail<kEpiThreads>(p, pref, G, total, et);
  } else if (CONV) {
    // ------------------------------------------------------------ fp8 -> f16 converter
    // Thread m widens key row m.  The TMA stage holds 128-byte fp8 rows in
    // the 128-byte swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)).
    // The widened row goes to TMEM lane m (row m of the MMA's A operand, two
    // K elements a column), or, for N > 128, to the two K-half blocks of a
    // shared-memory operand stage in the same swizzle (bank-conflict free on
    // both sides).  Row m is in this warp's TMEM lane quadrant.
    static_assert(!CONV || R::kConvThreads == kBM, "one converter thread a key row");
    const int m = (warp & 3) * 32 + lane;
    const int sw = m & 7;
    const bool a_tmem = L.a_tmem != 0;
    const uint32_t a_lane = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)L.a_col;
    const int cw = warp - (2 + R::kEpiWarps);  // converter warp 0..3
    int stage = 0, a = 0;
    uint32_t phase = 0, aphase = 0;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int qg = -1;
    uint32_t q_uses = 0;
    bool ok = true;
    for (int t = t_begin; t < t_end && ok; ++t) {
      while (t >= pref[g + 1]) ++g;
      if (g != qg) {
        // a new group's q (bf16, landed by the producer once the MMAs of the
        // last group were done): scaled into f16 in place, each row-head by
        // its 2^-e.  Half-warp h of this warp takes row-head n = 2 (cw + 4 i)
        // + h; lane l of it the 16 bytes at chunk l % 8 of K-half l / 8 (the
        // swizzle only permutes a row's chunks, and the conversion is per
        // element).
        ok = __all_sync(0xffffffffu, wait_phase(qfull, q_uses & 1u, abort_flag, p.fault));
        if (!ok) break;
        const int l16 = lane & 15;
        for (int n0 = 2 * cw; n0 < N; n0 += 2 * R::kConvWarps) {
          const int n = n0 + (lane >> 4);
          uint4* qp = reinterpret_cast<uint4*>(Bq + (l16 >> 3) * (N * 128) + n * 128 + (l16 & 7) * 16);
          const uint4 v = *qp;
          uint32_t amax = bf16x8_amax_bits(v);
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const int ne = -q_row_exp(amax);
          *qp = bf16x8_scaled_to_f16(v, pow2_exact(ne / 2), pow2_exact(ne - ne / 2));
        }
        ptx::fence_proxy_async_smem();  // generic-proxy writes -> visible to tcgen05.mma
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(qready);
        ++q_uses;
        qg = g;
      }
      ok = wait_phase(&full[stage], phase, abort_flag, p.fault) &&
           wait_phase(&aempty[a], aphase ^ 1u, abort_flag, p.fault);
      // the warp goes on together (the TMEM stores below are warp-wide)
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();  // after the MMA's reads of the stage's last use
      const uint8_t* src = S + stage * L.stage_bytes + m * 128;
      uint4 in[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) in[i] = *reinterpret_cast<const uint4*>(src + ((i ^ sw) << 4));
      {
        // Tile i's scales go to ring slot i % kScaleRing, last used by tile
        // i - kScaleRing (kScaleRing even: same epilogue set as tile i).  It
        // is free: before this point the converter waited, for tiles j = i - 1
        // and i, until the MMA of tile j - a_stages had completed, and that
        // MMA had waited for the epilogue to release accumulator use
        // j - a_stages - naccs.  One of those two uses has the parity of i and
        // is not before i - kScaleRing; its set works through its tiles in
        // order and reads a tile's scales before releasing it.
        static_assert(kScaleRing % 2 == 0 && kScaleRing >= kFp8TmemStages + 4 &&
                          kScaleRing >= kFp8ConvStages + 2 + 1,
                      "scale slot reuse");
        const int i = t - t_begin;
        scale_ring[(i % kScaleRing) * kBM + m] =
            *reinterpret_cast<const float*>(S + stage * L.stage_bytes + kFp8StageBytes + m * 4);
        ptx::mbar_arrive(&sfull[i % kScaleRing]);
        ptx::mbar_arrive(&empty[stage]);  // this thread's reads of the stage are done
      }
      if (a_tmem) {
        // columns 8j .. 8j + 7 of the stage: the 16 elements of fp8 chunk j,
        // two to a column, the lower K index in the low half
        const uint32_t ta = a_lane + (uint32_t)(a * 64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[16];
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint4 w = in[2 * c + jj];
            o[8 * jj + 0] = e4m3x2_to_f16x2<0>(w.x);
            o[8 * jj + 1] = e4m3x2_to_f16x2<1>(w.x);
            o[8 * jj + 2] = e4m3x2_to_f16x2<0>(w.y);
            o[8 * jj + 3] = e4m3x2_to_f16x2<1>(w.y);
            o[8 * jj + 4] = e4m3x2_to_f16x2<0>(w.z);
            o[8 * jj + 5] = e4m3x2_to_f16x2<1>(w.z);
            o[8 * jj + 6] = e4m3x2_to_f16x2<0>(w.w);
            o[8 * jj + 7] = e4m3x2_to_f16x2<1>(w.w);
          }
          ptx::tmem_st16(ta + 16u * (uint32_t)c, o);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();  // the stores -> the MMA, through the barrier
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint8_t* dst = A + a * kTileBytes + (i >> 2) * kHalfBytes + m * 128;
          const int j = i & 3;  // 16-byte fp8 chunk j of the half: bf16 chunks 2j, 2j + 1
          uint4 o0, o1;
          o0.x = e4m3x2_to_f16x2<0>(in[i].x);
          o0.y = e4m3x2_to_f16x2<1>(in[i].x);
          o0.z = e4m3x2_to_f16x2<0>(in[i].y);
          o0.w = e4m3x2_to_f16x2<1>(in[i].y);
          o1.x = e4m3x2_to_f16x2<0>(in[i].z);
          o1.y = e4m3x2_to_f16x2<1>(in[i].z);
          o1.z = e4m3x2_to_f16x2<0>(in[i].w);
          o1.w = e4m3x2_to_f16x2<1>(in[i].w);
          *reinterpret_cast<uint4*>(dst + (((2 * j) ^ sw) << 4)) = o0;
          *reinterpret_cast<uint4*>(dst + (((2 * j + 1) ^ sw) << 4)) = o1;
        }
        ptx::fence_proxy_async_smem();  // generic-proxy writes -> visible to tcgen05.mma
      }
      ptx::mbar_arrive(&afull[a]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++a == kAStages) {
        a = 0;
        aphase ^= 1u;
      }
    }
  }

  if (!CONV && warp >= 2 + R::kEpiWarps && setup_ok) {
    // ------------------------------------------------------------ bf16 spare warps
    // the -inf tail, while the pipeline starts up and streams keys
    fill_tail<R::kConvThreads>(p, pref, G, total, (int)threadIdx.x - 64 - kEpiThreads);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, (uint32_t)L.tmem_cols);
  if (FUSE) {
    // selection of the rows of completed groups: all 512 threads, or the
    // first 256 of the converter kernel's 448
    constexpr int NT = kThreads >= 512 ? 512 : 256;
    if (threadIdx.x < NT) fused_select<NT>(p, pref, G, t_begin, t_end, smem, fz);
  }
}

// Launch helpers, one translation unit per key type (umma_bf16.cu, umma_fp8.cu).
cudaError_t launch_bf16(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                        const Layout& L, int grid, cudaStream_t s);
cudaError_t launch_fp8(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                       const Layout& L, int grid, cudaStream_t s);
cudaError_t launch_q8(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                      const Layout& L, int grid, cudaStream_t s);
// The lean form (umma_lean.cu): bf16 keys, or fp8 keys with fp8 q.
cudaError_t launch_lean(int heads, int kind, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                        const Layout& L, int grid, cudaStream_t s);
// Scoring followed by the selection of every row in the same kernel (umma_*_topk.cu).
cudaError_t launch_bf16_topk(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                             const Layout& L, int grid, cudaStream_t s);
cudaError_t launch_fp8_topk(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                            const Layout& L, int grid, cudaStream_t s);
cudaError_t launch_q8_topk(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                           const Layout& L, int grid, cudaStream_t s);

template <int H, int KIND, bool FUSE, bool LEAN>
cudaError_t launch_h(const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up, const Layout& L,
                     int grid, cudaStream_t s) {
  auto kern = umma_score_kernel<H, KIND, FUSE, LEAN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return e;
  // programmatic stream serialisation: the launch may begin while the
  // previous kernel finishes; the kernel waits for it before touching memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(Roles<KIND == kKindFp8Keys, LEAN>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, kv, qm, up, L);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KIND, bool FUSE = false, bool LEAN = false>
cudaError_t launch_any(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                       const Layout& L, int grid, cudaStream_t s) {
  switch (heads) {
    case 1: return launch_h<1, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    case 2: return launch_h<2, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    case 4: return launch_h<4, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    case 8: return launch_h<8, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    case 16: return launch_h<16, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    case 32: return launch_h<32, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
    default: return launch_h<64, KIND, FUSE, LEAN>(kv, qm, up, L, grid, s);
  }
}

}  // namespace umma
}  // namespace qsa
