// Internal declarations shared by the library's translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

// Parameters of one scoring launch, resolved on the host from qsa_paged_desc.
struct ScoreParams {
  const uint16_t* q;        // bf16 bits [R][H][128], or e4m3 codes when q8
  const float* weights;     // [R][H]
  const uint8_t* kv;        // paged keys
  const uint8_t* scales;    // fp8 scales base (NULL for bf16)
  const int32_t* block_table;
  const int32_t* visible;
  const int32_t* next_n_lens;  // [num_requests] live rows of each request, or null (all live)
  float* out;
  int64_t out_cols;
  int64_t key_page_stride;
  int64_t scale_page_stride;
  int64_t capacity;         // min(out_cols, max_pages * page_cols): largest legal visible count
  int32_t num_requests, rows_per_req, num_rows, num_heads, page_cols, max_pages, num_pages;
  int32_t fp8;
  int32_t q8;               // q as e4m3 codes [R][H][128] (fp8 keys only)
};

// Selection fused into a tcgen05 scoring launch (qsa_paged_mqa_topk).
constexpr int kFuseMaxGroups = 256;  // row groups a fused launch takes at most
struct FuseArgs {
  int32_t* topk_out;  // [num_rows][k]
  uint32_t* sync;     // 2 * groups + 1 words, zero (and zero again once the launch completes)
  int32_t k;
};

// Each launcher returns cudaSuccess or the launch error; `msg` gets a reason
// when a shape is rejected (then the return is cudaErrorInvalidValue).
cudaError_t launch_rowcore(const ScoreParams& p, cudaStream_t stream, const char** msg);
bool umma_supports(const qsa_paged_desc& d, const char** why);
// The lean form of the tcgen05 scorer serves `d` (with fp8 q when q8).
bool umma_lean_supports(const qsa_paged_desc& d, bool q8, const char** why);
// Row groups the tcgen05 scorer splits `d` into (rows x heads of a group <= 256).
int64_t umma_num_groups(const qsa_paged_desc& d);
cudaError_t launch_umma(const ScoreParams& p, cudaStream_t stream, const char** msg,
                        const FuseArgs* fuse = nullptr, bool lean = false);
// Device address of the fault word on the current device (bit 0: a scoring
// kernel's bounded wait gave up; bit 1: a top-k kernel's).
cudaError_t fault_word_address(unsigned int** out);
// Reads (and optionally clears) the device fault word the kernels set when a
// bounded wait gives up.  Synchronises the device.
cudaError_t read_fault_word(uint32_t* flags, bool clear);
// Top-k of every row over [0, n_r): n_r = visible[r] clamped to [0, min(capacity,
// row_stride)], and 0 for a dead row (next_n_lens non-null: row r is dead when
// r % rows_per_req >= next_n_lens[r / rows_per_req]).  max_visible > 0 is the
// caller's bound on the n_r, a dispatch hint only: a row above it is still
// selected exactly, more slowly.
cudaError_t launch_topk(const float* logits, int64_t num_rows, int64_t row_stride, const int32_t* visible,
                        const int32_t* next_n_lens, int32_t rows_per_req, int64_t capacity, int64_t max_visible,
                        int32_t k, int32_t* out, cudaStream_t stream);

// Cached per-device properties (queried once per device).
struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;
};
cudaError_t device_info(DeviceInfo* info);

// page_stream.cu: qsa_page_stream's launch (arguments already validated).
cudaError_t launch_page_stream(const uint8_t* base, int64_t page_stride, int32_t page_bytes, const int32_t* pages,
                               int64_t num_listed, int64_t pool_pages, uint32_t* checksum, cudaStream_t stream);

}  // namespace qsa
