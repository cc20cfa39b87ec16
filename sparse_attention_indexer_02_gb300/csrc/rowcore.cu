// CUDA-core scorer: one query row at a time (the one-row decode kernel).
//
// vLLM #62589 "Dispatch"/"Details": for single-row decode the 16-row MMA tile
// is mostly padding, so rows are scored one by one with fp32 CUDA-core math
// and column blocks at or past the row's visible count exit at once.  This
// kernel also serves every shape the tcgen05 scorer does not (any head count,
// any page size), so it is the library's general path.
//
// Work split: a CTA owns one row and a chunk of kChunk columns.  Blocks are
// numbered chunk-major (block = chunk * R + row), so the low column chunks -
// the ones that hold visible columns - of every row launch first and the pure
// -inf chunks fill in behind them.  Inside a CTA, 8 lanes share one key (16
// head-dim elements each), so one warp reads 4 whole keys with 16-byte
// coalesced loads; kUnroll keys per lane group are in flight at once, and the
// page ids of the next step are fetched while the current keys load.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "device_common.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLanesPerKey = 8;
constexpr int kKeysPerWarp = 32 / kLanesPerKey;               // 4
constexpr int kUnroll = 4;                                    // keys per lane group per step
constexpr int kKeysPerStep = kKeysPerWarp * kWarps * kUnroll;  // 128
constexpr int kChunk = 512;                                   // columns per CTA
constexpr int kHeadDim = 128;

struct RowcoreArgs {
  ScoreParams p;
  int32_t chunks_per_row;
  int32_t heads_pad;  // num_heads rounded up to the register tile HR
};

// Head-dim element held in register i (0..15) by lane `sub` of a key group.
// bf16: bytes [16 sub, 16 sub + 16) and [128 + 16 sub, ...) of the 256-byte key.
// fp8 : bytes [16 sub, 16 sub + 16) of the 128-byte key.
template <bool FP8>
__device__ __forceinline__ int dim_of(int sub, int i) {
  if (FP8) return 16 * sub + i;
  return i < 8 ? 8 * sub + i : 64 + 8 * sub + (i - 8);
}

template <bool FP8>
struct KeyRaw {
  uint4 a, b;   // bf16: two 16-byte pieces; fp8: a only
  float scale;  // fp8 only
};

template <bool FP8>
__device__ __forceinline__ void load_key(const ScoreParams& p, int32_t page, int32_t slot, int sub,
                                         KeyRaw<FP8>& k) {
  if (FP8) {
    const uint8_t* base = p.kv + (int64_t)page * p.key_page_stride + (int64_t)slot * kHeadDim;
    k.a = ld_stream_v4(base + 16 * sub);
    k.scale = __ldg(reinterpret_cast<const float*>(p.scales + (int64_t)page * p.scale_page_stride +
                                                   4 * (int64_t)slot));
  } else {
    const uint8_t* base = p.kv + (int64_t)page * p.key_page_stride + (int64_t)slot * (2 * kHeadDim);
    k.a = ld_stream_v4(base + 16 * sub);
    k.b = ld_stream_v4(base + 128 + 16 * sub);
  }
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes), __NV_E4M3);
  return __half22float2(__half2(h));
}

// Partial dots of HR heads over the lane's 16 elements; key words are widened
// to fp32 pair by pair as they are consumed.
template <int HR, bool FP8>
__device__ __forceinline__ void partial_dots(const KeyRaw<FP8>& k, const float (&qr)[HR][16],
                                             float (&dot)[HR]) {
#pragma unroll
  for (int h = 0; h < HR; ++h) dot[h] = 0.0f;
  if (FP8) {
    const uint32_t w[4] = {k.a.x, k.a.y, k.a.z, k.a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 lo = e4m3x2_to_float2(w[j] & 0xFFFFu);
      const float2 hi = e4m3x2_to_float2(w[j] >> 16);
#pragma unroll
      for (int h = 0; h < HR; ++h) {
        dot[h] = fmaf(qr[h][4 * j + 0], lo.x, dot[h]);
        dot[h] = fmaf(qr[h][4 * j + 1], lo.y, dot[h]);
        dot[h] = fmaf(qr[h][4 * j + 2], hi.x, dot[h]);
        dot[h] = fmaf(qr[h][4 * j + 3], hi.y, dot[h]);
      }
    }
  } else {
    const uint32_t w[8] = {k.a.x, k.a.y, k.a.z, k.a.w, k.b.x, k.b.y, k.b.z, k.b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float lo = bf16_lo(w[j]), hi = bf16_hi(w[j]);
#pragma unroll
      for (int h = 0; h < HR; ++h) {
        dot[h] = fmaf(qr[h][2 * j + 0], lo, dot[h]);
        dot[h] = fmaf(qr[h][2 * j + 1], hi, dot[h]);
      }
    }
  }
}

template <int HR, bool FP8>
__global__ void __launch_bounds__(kThreads, HR >= 8 ? 1 : 2) rowcore_kernel(const RowcoreArgs args) {
  const ScoreParams& p = args.p;
  extern __shared__ float smem[];
  const int Hp = args.heads_pad;
  float* q_s = smem;                        // [Hp][128]
  float* w_s = q_s + Hp * kHeadDim;         // [Hp]
  float* out_s = w_s + ((Hp + 3) & ~3);     // [kChunk]

  const int64_t bid = blockIdx.x;
  const int64_t row = bid % p.num_rows;
  const int64_t chunk = bid / p.num_rows;
  const int64_t c0 = chunk * kChunk;
  const int64_t c_end = c0 + kChunk < p.out_cols ? c0 + kChunk : p.out_cols;
  const int64_t vis = row_visible(p.visible, p.next_n_lens, row, p.rows_per_req, p.capacity);
  float* out_row = p.out + row * p.out_cols;

  if (c0 >= vis) {  // column chunk past the visible range: mask only, no key traffic
    for (int64_t c = c0 + threadIdx.x; c < c_end; c += kThreads) out_row[c] = -INFINITY;
    return;
  }

  // q (bf16 -> fp32) and weights of this row, zero-padded to Hp heads.
  for (int i = threadIdx.x; i < Hp * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim;
    float v = 0.0f;
    if (h < p.num_heads) {
      if (p.q8) {  // e4m3 code -> half (exact) -> float
        const uint8_t code = reinterpret_cast<const uint8_t*>(p.q)[(row * p.num_heads) * kHeadDim + i];
        v = __half2float(__half(__nv_cvt_fp8_to_halfraw(code, __NV_E4M3)));
      } else {
        const uint32_t bits = p.q[(row * p.num_heads) * kHeadDim + i];
        v = __uint_as_float(bits << 16);
      }
    }
    q_s[i] = v;
  }
  for (int h = threadIdx.x; h < Hp; h += kThreads)
    w_s[h] = h < p.num_heads ? p.weights[row * p.num_heads + h] : 0.0f;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane % kLanesPerKey;
  const int kslot = lane / kLanesPerKey;
  const int64_t b = row / p.rows_per_req;
  const int32_t* bt = p.block_table + b * (int64_t)p.max_pages;
  const int64_t c_lim = c_end < vis ? c_end : vis;
  // Only the 8-head tile ever loops over head passes (H > 8); smaller tiles
  // hold every head in registers, so their single pass is a compile-time fact.
  const int passes = HR == 8 ? Hp / HR : 1;

  float qr[HR][16];
  if (passes == 1) {
#pragma unroll
    for (int h = 0; h < HR; ++h)
#pragma unroll
      for (int i = 0; i < 16; ++i) qr[h][i] = q_s[h * kHeadDim + dim_of<FP8>(sub, i)];
  }

  auto col_of = [&](int64_t cs, int u) -> int64_t {
    return cs + (int64_t)(u * kWarps + warp) * kKeysPerWarp + kslot;
  };
  auto page_of = [&](int64_t c) -> int32_t {
    int32_t pg = __ldg(bt + c / p.page_cols);
    return pg < 0 ? 0 : (pg >= p.num_pages ? p.num_pages - 1 : pg);
  };

  int32_t pages[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t c = col_of(c0, u);
    pages[u] = c < c_lim ? page_of(c) : 0;
  }

  for (int64_t cs = c0; cs < c_lim; cs += kKeysPerStep) {
    KeyRaw<FP8> raw[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = col_of(cs, u);
      if (c < c_lim) {
        load_key<FP8>(p, pages[u], (int32_t)(c % p.page_cols), sub, raw[u]);
      } else {
        raw[u].a = make_uint4(0, 0, 0, 0);
        raw[u].b = make_uint4(0, 0, 0, 0);
        raw[u].scale = 0.0f;
      }
    }
    // page ids of the next step, overlapped with this step's key loads
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = col_of(cs + kKeysPerStep, u);
      pages[u] = c < c_lim ? page_of(c) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = col_of(cs, u);
      // Skip only when the warp's first key is past the limit, so the skip is
      // warp-uniform and every lane reaches the shuffles below; keys past the
      // limit inside a live warp were zero-filled and are not stored.
      if (c - kslot >= c_lim) continue;
      float logit = 0.0f;
      for (int ps = 0; ps < passes; ++ps) {
        if (HR == 8 && passes > 1) {
#pragma unroll
          for (int h = 0; h < HR; ++h)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              qr[h][i] = q_s[(ps * HR + h) * kHeadDim + dim_of<FP8>(sub, i)];
        }
        float dot[HR];
        partial_dots<HR, FP8>(raw[u], qr, dot);
        // sum the 8 partial dots of each head across the key's lane group
#pragma unroll
        for (int h = 0; h < HR; ++h) {
          dot[h] += __shfl_xor_sync(0xFFFFFFFFu, dot[h], 4);
          dot[h] += __shfl_xor_sync(0xFFFFFFFFu, dot[h], 2);
          dot[h] += __shfl_xor_sync(0xFFFFFFFFu, dot[h], 1);
        }
#pragma unroll
        for (int h = 0; h < HR; ++h) {
          float d = dot[h];
          if (FP8) d *= raw[u].scale;  // dequantise before the ReLU
          logit = fmaf(w_s[ps * HR + h], relu_keep_nan(d), logit);
        }
      }
      if (sub == 0 && c < c_lim) out_s[c - c0] = logit + 0.0f;
    }
  }
  __syncthreads();
  for (int64_t c = c0 + threadIdx.x; c < c_end; c += kThreads)
    out_row[c] = c < vis ? out_s[c - c0] : -INFINITY;
}

template <int HR, bool FP8>
cudaError_t launch_t(const RowcoreArgs& a, int64_t grid, size_t smem, cudaStream_t s) {
  auto kern = rowcore_kernel<HR, FP8>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rowcore(const ScoreParams& p, cudaStream_t stream, const char** msg) {
  if (p.num_rows == 0 || p.out_cols == 0) return cudaSuccess;
  RowcoreArgs a;
  a.p = p;
  const int64_t chunks = (p.out_cols + kChunk - 1) / kChunk;
  const int64_t grid = chunks * p.num_rows;
  if (grid > 0x7FFFFFFFLL) {
    *msg = "rowcore: rows x column chunks exceeds the grid limit";
    return cudaErrorInvalidValue;
  }
  a.chunks_per_row = (int32_t)chunks;
  const int H = p.num_heads;
  int HR = H <= 1 ? 1 : (H <= 2 ? 2 : (H <= 4 ? 4 : 8));
  a.heads_pad = (H + HR - 1) / HR * HR;
  const size_t smem = sizeof(float) * ((size_t)a.heads_pad * kHeadDim + ((a.heads_pad + 3) & ~3) + kChunk);
  const bool f8 = p.fp8 != 0;
  switch (HR) {
    case 1: return f8 ? launch_t<1, true>(a, grid, smem, stream) : launch_t<1, false>(a, grid, smem, stream);
    case 2: return f8 ? launch_t<2, true>(a, grid, smem, stream) : launch_t<2, false>(a, grid, smem, stream);
    case 4: return f8 ? launch_t<4, true>(a, grid, smem, stream) : launch_t<4, false>(a, grid, smem, stream);
    default: return f8 ? launch_t<8, true>(a, grid, smem, stream) : launch_t<8, false>(a, grid, smem, stream);
  }
}

}  // namespace qsa
