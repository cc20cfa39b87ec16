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
// Structure (one persistent CTA per SM, 6 warps):
//  * schedule: every CTA derives, from the visible counts, the tile count of
//    each row group (tiles past the group's widest visible column are never
//    scheduled - the early exit of vLLM #62589 "Overview") and takes an equal
//    contiguous share of the flattened (group, tile) list, plus an equal share
//    of the pure -inf tail (columns past each group's last tile).
//  * warp 0 (TMA): per tile, lanes fetch the block-table entries of the tile's
//    pages and each issues the page's two 64-column K-halves as 3-D tensor
//    copies into a 128-byte-swizzled stage (aiter #4221 KVBlockSize>=1 commit:
//    block = table[b][col / page_cols], slot = col % page_cols).  A new group's
//    q is loaded by a 2-D tensor copy once the previous group's MMAs are done.
//  * warp 1 (MMA): one thread issues 8 tcgen05.mma (K = 16 each) per tile into
//    one of two TMEM accumulators and commits the stage back to the producer.
//  * warps 2-5 (epilogue): tcgen05.ld of the tile's columns, per head
//    ReLU * weight, head sum, +0.0, -inf past the row's visible count, store.
// Every barrier wait gives up after about a second, sets the device fault
// word (qsa_device_status) and lets the CTA drain and exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "qsa_internal.h"
#include "sm100_ptx.cuh"

namespace qsa {
namespace {

constexpr int kBM = 128;                    // keys per tile (MMA M)
constexpr int kHalfBytes = kBM * 128;       // one 64-element K-half of a bf16 key tile
constexpr int kTileBytes = 2 * kHalfBytes;  // 32 KB
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr long long kSpinCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr int kMaxSmem = 232448;                 // 227 KB opt-in limit per CTA

__device__ unsigned int g_fault_word = 0;

struct UmmaParams {
  const float* weights;
  const int32_t* block_table;
  const int32_t* visible;
  float* out;
  int64_t out_cols;
  int64_t capacity;
  int32_t num_rows, rows_per_req, num_heads, page_cols, max_pages, num_pages;
  int32_t group_rows, groups_per_req, num_groups, tiles_cap, box_rows;
};

template <int N>
struct Cfg {
  static constexpr int kStages = N <= 32 ? 6 : (N == 64 ? 5 : 4);
  static constexpr int kTmemCols = 2 * N < 32 ? 32 : 2 * N;
  static constexpr int kIdesc = ptx::idesc_bf16_f32(kBM, N);
  static constexpr int kAOff = 0;
  static constexpr int kBOff = kStages * kTileBytes;
  static constexpr int kBarOff = kBOff + N * 256;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 3;  // full, empty, tfull, tempty, qfull, qempty, done
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // tmem slot, abort flag
  static constexpr int kEpiOff = kMiscOff + 16;             // w_s[256], vis_s[256]
  static constexpr int kSchedOff = kEpiOff + 2 * 256 * 4;   // pref[G + 1], gmax[G]
  static int smem_bytes(int groups) { return 1024 + kSchedOff + 8 * (groups + 1); }
};

struct Sync {
  volatile int* abort;
};

// Bounded wait on an mbarrier phase.  Returns false on abort or time-out.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinCycles) {
      *abort_flag = 1;
      atomicOr(&g_fault_word, 1u);
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

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    umma_score_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const UmmaParams p) {
  using C = Cfg<N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* A = smem + C::kAOff;
  uint8_t* Bq = smem + C::kBOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + 1;
  uint64_t* mma_done = qempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  float* w_s = reinterpret_cast<float*>(smem + C::kEpiOff);
  int32_t* vis_s = reinterpret_cast<int32_t*>(w_s + 256);
  int32_t* pref = reinterpret_cast<int32_t*>(smem + C::kSchedOff);
  int32_t* gmax = pref + p.num_groups + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.num_groups;
  const int H = p.num_heads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kEpiThreads);
    }
    ptx::mbar_init(qfull, 1);
    ptx::mbar_init(qempty, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&kv_map);
    ptx::prefetch_tmap(&q_map);
  }
  // Per-group tile counts from the visible counts (device data, no host sync).
  for (int g = threadIdx.x; g < G; g += kThreads) {
    const int b = g / p.groups_per_req, j = g % p.groups_per_req;
    const int r0 = b * p.rows_per_req + j * p.group_rows;
    const int nr = min(p.group_rows, p.rows_per_req - j * p.group_rows);
    int64_t mv = 0;
    for (int i = 0; i < nr; ++i) {
      const int64_t v = clamp64(p.visible[r0 + i], 0, p.capacity);
      mv = v > mv ? v : mv;
    }
    gmax[g] = (int32_t)mv;
    pref[g] = (int32_t)((mv + kBM - 1) / kBM);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (warp == 0) {  // exclusive scan of the tile counts, total in pref[G]
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
  __syncthreads();
  const int total = pref[G];
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t policy = ptx::policy_evict_first();
    const int pc = p.page_cols;
    const int boxes_full = pc >= kBM ? 1 : kBM / pc;
    const uint32_t box_bytes = (uint32_t)p.box_rows * 128u;
    int stage = 0;
    uint32_t phase = 0;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int qg = -1;
    uint32_t q_loads = 0;
    uint32_t filled_mask = 0, last_phase_bits = 0;
    bool ok = true;
    for (int t = t_begin; t < t_end && ok; ++t) {
      while (t >= pref[g + 1]) ++g;
      const int b = g / p.groups_per_req, jj = g % p.groups_per_req;
      const int r0 = b * p.rows_per_req + jj * p.group_rows;
      const int c0 = (t - pref[g]) * kBM;
      const int lim = gmax[g] - c0;  // visible columns in this tile (>= 1)
      const int nbox = pc >= kBM ? 1 : min(boxes_full, (lim + pc - 1) / pc);
      int32_t page = 0;
      if (lane < nbox) {
        const int64_t lp = pc >= kBM ? (int64_t)c0 / pc : (int64_t)c0 / pc + lane;
        const int32_t v = __ldg(p.block_table + (int64_t)b * p.max_pages + lp);
        page = v < 0 ? 0 : (v >= p.num_pages ? p.num_pages - 1 : v);
      }
      if (g != qg) {
        if (q_loads > 0) ok = wait_phase(qempty, (q_loads - 1) & 1, abort_flag);
        if (!ok) break;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(qfull, 2u * N * 128u);
          ptx::tma_load_2d(Bq, &q_map, 0, r0 * H, qfull);
          ptx::tma_load_2d(Bq + N * 128, &q_map, 64, r0 * H, qfull);
        }
        qg = g;
        ++q_loads;
      }
      ok = wait_phase(&empty[stage], phase ^ 1u, abort_flag);
      if (!ok) break;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2u * nbox * box_bytes);
      __syncwarp();
      if (lane < nbox) {
        const int y = pc >= kBM ? c0 % pc : 0;
        const uint32_t row_off = pc >= kBM ? 0u : (uint32_t)lane * (uint32_t)pc * 128u;
        uint8_t* dst = A + stage * kTileBytes + row_off;
        ptx::tma_load_3d(dst, &kv_map, 0, y, page, &full[stage], policy);
        ptx::tma_load_3d(dst + kHalfBytes, &kv_map, 64, y, page, &full[stage], policy);
      }
      filled_mask |= 1u << stage;
      last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // Drain: every copy this warp issued has landed before the CTA tears down.
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < C::kStages; ++s)
        if (filled_mask & (1u << s)) {
          const long long t0 = clock64();
          while (!ptx::mbar_try_wait(&full[s], (last_phase_bits >> s) & 1u) && clock64() - t0 < kSpinCycles) {
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
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
          if (qg >= 0) ptx::mma_commit(qempty);  // q buffer free once earlier MMAs finish
          ok = wait_phase(qfull, q_uses & 1u, abort_flag);
          if (!ok) break;
          ++q_uses;
          qg = g;
        }
        ok = wait_phase(&tempty[acc], acc_phase ^ 1u, abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        ok = wait_phase(&full[stage], phase, abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * N);
        const uint32_t a0 = a_base + stage * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (uint32_t)(k & 3) * 32u;
          const uint64_t ad = ptx::sw128_desc(a0 + (k >> 2) * kHalfBytes + koff);
          const uint64_t bd = ptx::sw128_desc(b_base + (k >> 2) * (N * 128) + koff);
          ptx::mma_bf16(d, ad, bd, C::kIdesc, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&empty[stage]);
        ptx::mma_commit(&tfull[acc]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued above has completed before TMEM is released
      ptx::mma_commit(mma_done);
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(mma_done, 0) && clock64() - t0 < kSpinCycles) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0..127
    const int quad = warp & 3;        // TMEM lane quadrant this warp may access
    const int m = quad * 32 + lane;   // key row of the tile = TMEM lane
    const int64_t oc = p.out_cols;

    // (1) this CTA's share of the -inf tail: group g's tiles [T_g, tiles_cap)
    {
      const int64_t Tc = p.tiles_cap;
      const int64_t F = (int64_t)G * Tc - total;
      int64_t f = F * blockIdx.x / gridDim.x;
      const int64_t f_end = F * (blockIdx.x + 1) / gridDim.x;
      if (f < f_end) {
        // fill prefix fp(g) = g * Tc - pref[g] is non-decreasing; find the group of f
        int lo = 0, hi = G;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if ((int64_t)mid * Tc - pref[mid] <= f) lo = mid;
          else hi = mid;
        }
        int g = lo;
        for (; f < f_end; ++f) {
          while (g + 1 < G && (int64_t)(g + 1) * Tc - pref[g + 1] <= f) ++g;
          const int Tg = pref[g + 1] - pref[g];
          const int64_t tile = Tg + (f - ((int64_t)g * Tc - pref[g]));
          const int64_t c = tile * kBM + et;
          if (c >= oc) continue;
          const int b = g / p.groups_per_req, jj = g % p.groups_per_req;
          const int r0 = b * p.rows_per_req + jj * p.group_rows;
          const int nr = min(p.group_rows, p.rows_per_req - jj * p.group_rows);
          for (int j = 0; j < nr; ++j) p.out[(int64_t)(r0 + j) * oc + c] = -INFINITY;
        }
      }
    }

    // (2) computed tiles
    int acc = 0;
    uint32_t acc_phase = 0;
    int g = t_begin < t_end ? find_group(pref, G, t_begin) : 0;
    int eg = -1, r0 = 0, nr = 0;
    bool ok = true;
    for (int t = t_begin; t < t_end && ok; ++t) {
      while (t >= pref[g + 1]) ++g;
      if (g != eg) {
        epi_bar();
        const int b = g / p.groups_per_req, jj = g % p.groups_per_req;
        r0 = b * p.rows_per_req + jj * p.group_rows;
        nr = min(p.group_rows, p.rows_per_req - jj * p.group_rows);
        for (int i = et; i < nr * H; i += kEpiThreads) w_s[i] = p.weights[(int64_t)r0 * H + i];
        for (int i = et; i < nr; i += kEpiThreads) vis_s[i] = (int32_t)clamp64(p.visible[r0 + i], 0, p.capacity);
        epi_bar();
        eg = g;
      }
      const int64_t c = (int64_t)(t - pref[g]) * kBM + m;
      ok = wait_phase(&tfull[acc], acc_phase, abort_flag);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * N);
      const int ncols = nr * H;
      float part = 0.0f;
      for (int col0 = 0; col0 < ncols; col0 += 16) {
        uint32_t v[16];
        ptx::tmem_ld16(tb + (uint32_t)col0, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = col0 + i;
          if (n < ncols) {
            part = fmaf(w_s[n], relu_keep_nan(__uint_as_float(v[i])), part);
            if ((n + 1) % H == 0) {
              const int j = n / H;
              if (c < oc) p.out[(int64_t)(r0 + j) * oc + c] = c < vis_s[j] ? part + 0.0f : -INFINITY;
              part = 0.0f;
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int pick_n(int rows_per_group, int heads) {
  const int need = rows_per_group * heads;
  for (int n : {16, 32, 64, 128, 256})
    if (need <= n) return n;
  return 0;
}

void group_shape(const qsa_paged_desc& d, int* G_rows, int* N) {
  int g = 256 / d.num_heads;
  if (g < 1) g = 1;
  if (g > d.rows_per_req) g = d.rows_per_req;
  *G_rows = g;
  *N = pick_n(g, d.num_heads);
}

int smem_for(int N, int groups) {
  switch (N) {
    case 16: return Cfg<16>::smem_bytes(groups);
    case 32: return Cfg<32>::smem_bytes(groups);
    case 64: return Cfg<64>::smem_bytes(groups);
    case 128: return Cfg<128>::smem_bytes(groups);
    default: return Cfg<256>::smem_bytes(groups);
  }
}

template <int N>
cudaError_t launch_n(const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up, int grid, int smem,
                     cudaStream_t s) {
  auto kern = umma_score_kernel<N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(kv, qm, up);
  return cudaGetLastError();
}

}  // namespace

bool umma_supports(const qsa_paged_desc& d, const char** why) {
  if (d.kv_dtype != QSA_KV_BF16) {
    *why = "fp8 keys are served by the CUDA-core scorer in this build";
    return false;
  }
  const int pc = d.page_cols;
  if (pc % 8 != 0 || !(kBM % pc == 0 || pc % kBM == 0)) {
    *why = "page_cols must be a multiple of 8 that divides 128 or is a multiple of 128";
    return false;
  }
  if (d.out_cols > (int64_t)0x7FFFFF00LL) {
    *why = "out_cols too large for the tile index";
    return false;
  }
  int Gr, N;
  group_shape(d, &Gr, &N);
  if (N == 0) {
    *why = "rows x heads of a group exceed 256";
    return false;
  }
  const int64_t groups = (int64_t)d.num_requests * ((d.rows_per_req + Gr - 1) / Gr);
  if (groups > (1 << 20) || smem_for(N, (int)groups) > kMaxSmem) {
    *why = "too many row groups for the on-chip schedule";
    return false;
  }
  const int64_t qrows = (int64_t)d.num_requests * d.rows_per_req * d.num_heads;
  if (qrows > 0x7FFFFFFFLL) {
    *why = "too many q rows for the tensor map";
    return false;
  }
  return true;
}

cudaError_t launch_umma(const ScoreParams& p, cudaStream_t stream, const char** msg) {
  if (p.num_rows == 0 || p.out_cols == 0) return cudaSuccess;
  qsa_paged_desc d{};
  d.num_requests = p.num_requests;
  d.rows_per_req = p.rows_per_req;
  d.num_heads = p.num_heads;
  d.head_dim = 128;
  d.page_cols = p.page_cols;
  d.kv_dtype = p.fp8 ? QSA_KV_FP8_E4M3 : QSA_KV_BF16;
  d.out_cols = p.out_cols;
  if (!umma_supports(d, msg)) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) {
    *msg = "cuTensorMapEncodeTiled is unavailable from the driver";
    return cudaErrorInvalidValue;
  }
  int Gr, N;
  group_shape(d, &Gr, &N);
  UmmaParams up;
  up.weights = p.weights;
  up.block_table = p.block_table;
  up.visible = p.visible;
  up.out = p.out;
  up.out_cols = p.out_cols;
  up.capacity = p.capacity;
  up.num_rows = p.num_rows;
  up.rows_per_req = p.rows_per_req;
  up.num_heads = p.num_heads;
  up.page_cols = p.page_cols;
  up.max_pages = p.max_pages;
  up.num_pages = p.num_pages;
  up.group_rows = Gr;
  up.groups_per_req = (p.rows_per_req + Gr - 1) / Gr;
  up.num_groups = p.num_requests * up.groups_per_req;
  up.tiles_cap = (int32_t)((p.out_cols + kBM - 1) / kBM);
  up.box_rows = p.page_cols < kBM ? p.page_cols : kBM;

  CUtensorMap kv_map, q_map;
  {
    cuuint64_t dims[3] = {128, (cuuint64_t)p.page_cols, (cuuint64_t)p.num_pages};
    cuuint64_t strides[2] = {256, (cuuint64_t)p.key_page_stride};
    cuuint32_t box[3] = {64, (cuuint32_t)up.box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint8_t*>(p.kv), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "key-cache tensor map rejected by the driver";
      return cudaErrorInvalidValue;
    }
  }
  {
    cuuint64_t dims[2] = {128, (cuuint64_t)p.num_rows * (cuuint64_t)p.num_heads};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {64, (cuuint32_t)N};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *msg = "q tensor map rejected by the driver";
      return cudaErrorInvalidValue;
    }
  }
  DeviceInfo info;
  cudaError_t e = device_info(&info);
  if (e != cudaSuccess) return e;
  const int64_t upper = (int64_t)up.num_groups * up.tiles_cap;
  const int grid = (int)(upper < info.num_sms ? (upper < 1 ? 1 : upper) : info.num_sms);
  const int smem = smem_for(N, up.num_groups);
  switch (N) {
    case 16: return launch_n<16>(kv_map, q_map, up, grid, smem, stream);
    case 32: return launch_n<32>(kv_map, q_map, up, grid, smem, stream);
    case 64: return launch_n<64>(kv_map, q_map, up, grid, smem, stream);
    case 128: return launch_n<128>(kv_map, q_map, up, grid, smem, stream);
    default: return launch_n<256>(kv_map, q_map, up, grid, smem, stream);
  }
}

cudaError_t read_fault_word(uint32_t* flags, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof v);
  if (e != cudaSuccess) return e;
  *flags = v;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_fault_word, &z, sizeof z);
  }
  return e;
}

}  // namespace qsa
