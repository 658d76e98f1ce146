// Host-side interface between the C ABI (pa_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

struct MetadataParams {
  const void* req_pool_indices;  // int64 or int32 (idx64)
  const void* seq_lens;          // int64 or int32 (idx64)
  const int32_t* req_to_token;
  int64_t req_to_token_rows;
  int64_t req_to_token_stride;
  const int64_t* full_to_swa_mapping;  // nullptr: no sliding-window outputs
  int64_t mapping_len;
  const int64_t* out_cache_loc;
  int64_t num_out_tokens;  // valid prefix of out_cache_loc (already min'ed)
  const void* qlens;  // int64 or int32 (idx64)
  int32_t* cache_seqlens;
  int32_t* cu_seqlens_k;
  int32_t* cu_seqlens_q;
  int32_t* page_table;
  int64_t page_table_stride;
  int32_t* swa_page_table;
  int64_t swa_page_table_stride;
  int64_t* swa_out_cache_loc;
  int64_t swa_out_len;
  int32_t bs;
  int32_t seqlen_offset;
  int32_t max_seq_pages;
  int32_t page_size;
  int32_t q_mode;
  int32_t q_stride;
  bool idx64;  // index inputs are int64 (else int32)
  unsigned int* err;
  unsigned long long* ts;  // stage timestamps (instrumented builds only), else nullptr
};

struct SplitKParams {
  const void* q;  // bf16 [bs, Hq, 128]
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  int64_t page_table_stride;
  const int32_t* cache_seqlens;
  int64_t num_pages;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t max_seq_pages;
  int32_t pages_per_split;
  int32_t num_splits;
  float q_scale;  // sm_scale * log2(e)
  // Several query tokens per request (tensor-core producer only): query rows of request
  // b are cu_seqlens_q[b] .. cu_seqlens_q[b+1], at most max_q_len of them; nullptr for
  // one query per request (row b).
  const int32_t* cu_seqlens_q;
  int32_t max_q_len;
  // Sliding window (tensor-core producer only): > 0 restricts query i of a request to
  // its `window` newest positions, starts the split partition at the page of the
  // request's first visible position, and skips pages whose table entry is -1.
  // pages_per_split is then counted over the window's pages.  0: whole context.
  int32_t window;
  int32_t bs;        // requests (the persistent form walks them itself)
  int32_t work_slot;  // persistent form: the work-claim counter this launch uses
  int32_t sm_count;  // SMs of the device (grids of at most this many blocks take the
                     // deep-pipeline configuration)
  int32_t hold_loads;  // instrumented build only: the TMA warp issues nothing (timeout test)
  int32_t no_persist;  // instrumented build only: one block per item (A/B test)
  float* m_out;
  float* l_out;
  float* acc_out;
  unsigned int* err;
  unsigned long long* ts;  // stage timestamps (instrumented builds only), else nullptr
};

struct ReduceParams {
  const float* m;
  const float* l;
  const float* acc;
  int64_t num_rows;  // bs * Hq
  int32_t num_splits;
  void* out;   // bf16 [num_rows, 128]
  float* lse;  // [num_rows] or nullptr
  unsigned long long* ts;  // stage timestamps (instrumented builds only), else nullptr
};

// Step of the last failed launch on this host thread (for pa_last_error_string).
inline thread_local const char* g_fail_site = "launch";
inline cudaError_t fail_at(cudaError_t e, const char* site) {
  if (e != cudaSuccess) g_fail_site = site;
  return e;
}

// PA_OK for cudaSuccess; otherwise records `where`, the failed step and the CUDA error
// for pa_last_error_string on this host thread and returns PA_ERR_CUDA.
pa_status from_cuda(cudaError_t e, const char* where);

cudaError_t launch_metadata(const MetadataParams& p, cudaStream_t stream, bool use_pdl);

// bs, grid and shapes are validated by the caller.
cudaError_t launch_splitk_bf16(const SplitKParams& p, int bs, int group, int page_size,
                               cudaStream_t stream, bool use_pdl);
cudaError_t launch_splitk_int8(const SplitKParams& p, int bs, int group, int page_size,
                               cudaStream_t stream, bool use_pdl);

cudaError_t launch_splitk_mma_bf16(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl);
cudaError_t launch_splitk_mma_int8(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl);
// Sliding-window variants (SplitKParams::window > 0).
cudaError_t launch_splitk_mma_window_bf16(const SplitKParams& p, int bs, int group,
                                          int page_size, cudaStream_t stream, bool use_pdl);
cudaError_t launch_splitk_mma_window_int8(const SplitKParams& p, int bs, int group,
                                          int page_size, cudaStream_t stream, bool use_pdl);

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream, bool use_pdl);

}  // namespace pa
