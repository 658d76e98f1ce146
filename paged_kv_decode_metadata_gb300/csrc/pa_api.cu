// C ABI of the decode-step library: argument checks, split heuristic, workspace
// layout and the three-launch decode step.  See include/pa.h for the contract.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>

#include "../../include/pa.h"
#include "../../include/pa_timestamps.h"
#include "pa_internal.h"

namespace {
// Last CUDA failure seen by an entry point on this host thread (pa_last_error_string).
thread_local char g_last_error[256] = "no CUDA error";
}  // namespace

namespace pa {

pa_status from_cuda(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return PA_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s [%s]: %s (%s)", where, g_fail_site,
           cudaGetErrorString(e), cudaGetErrorName(e));
  g_fail_site = "launch";
  return PA_ERR_CUDA;
}

}  // namespace pa

namespace {

// Device-side error word.  Kernels receive its device address; host code fetches
// that address once per device with cudaGetSymbolAddress.
__device__ unsigned int g_pa_error_flags;

constexpr int kMaxDevices = 64;
std::atomic<unsigned int*> g_err_ptr[kMaxDevices];
std::atomic<int32_t> g_producer{PA_PRODUCER_AUTO};
// Stage timestamp buffer (9 uint64) of the instrumented build; nullptr otherwise.
std::atomic<unsigned long long*> g_ts{nullptr};
// Instrumented build: non-zero makes later producer launches issue no copies.
std::atomic<int32_t> g_hold_loads{0};
// Instrumented build: non-zero keeps later producer launches at one block per item.
std::atomic<int32_t> g_no_persist{0};
std::atomic<int> g_sm_count[kMaxDevices];

cudaError_t error_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned int* p = g_err_ptr[dev].load();
  if (p == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_pa_error_flags);
    if (e != cudaSuccess) return e;
    p = static_cast<unsigned int*>(addr);
    g_err_ptr[dev].store(p);
  }
  *out = p;
  return cudaSuccess;
}

int sm_count_of_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_sm_count[dev].load();
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(n);
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using pa::from_cuda;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

pa_status check_metadata(const void* req_pool_indices, const void* seq_lens,
                         const int32_t* req_to_token, int64_t req_to_token_rows,
                         int64_t req_to_token_stride, const int64_t* mapping,
                         int64_t mapping_len, int32_t* cache_seqlens, int32_t* cu_seqlens_k,
                         int32_t* page_table, int64_t page_table_stride,
                         int32_t* swa_page_table, int64_t swa_page_table_stride, int32_t bs,
                         int32_t max_seq_pages, int32_t page_size) {
  if (bs < 0 || max_seq_pages < 0 || page_size < 1) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (!req_pool_indices || !seq_lens || !cache_seqlens || !cu_seqlens_k || !page_table)
    return PA_ERR_INVALID;
  if (bs >= (1 << 30)) return PA_ERR_INVALID;
  if (page_table_stride < max_seq_pages) return PA_ERR_INVALID;
  if (max_seq_pages > 0) {
    if (!req_to_token || req_to_token_rows < 1) return PA_ERR_INVALID;
    if (static_cast<int64_t>(max_seq_pages - 1) * page_size >= req_to_token_stride)
      return PA_ERR_INVALID;
  }
  if ((mapping == nullptr) != (swa_page_table == nullptr)) return PA_ERR_INVALID;
  if (mapping != nullptr) {
    if (mapping_len < 1 || swa_page_table_stride < max_seq_pages) return PA_ERR_INVALID;
  }
  return PA_OK;
}

pa_status check_attention(const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale, int32_t kv_dtype,
                          const int32_t* page_table, int64_t page_table_stride,
                          const int32_t* cache_seqlens, int32_t bs, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                          int64_t num_pages, int32_t max_seq_pages, int32_t num_splits) {
  if (bs < 0) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_INT8) return PA_ERR_INVALID;
  if (!q || !k_cache || !v_cache || !page_table || !cache_seqlens) return PA_ERR_INVALID;
  if (kv_dtype == PA_KV_INT8 && (!k_scale || !v_scale)) return PA_ERR_INVALID;
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID;
  if (num_pages < 1 || max_seq_pages < 1 || page_table_stride < max_seq_pages)
    return PA_ERR_INVALID;
  if (num_splits < 1 || num_splits > 4096) return PA_ERR_INVALID;
  if (bs > 65535 || num_kv_heads > 65535) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
  if (kv_dtype == PA_KV_INT8 && (!aligned16(k_scale) || !aligned16(v_scale)))
    return PA_ERR_INVALID;
  const int group = num_q_heads / num_kv_heads;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return PA_ERR_UNSUPPORTED;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
    return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_seq_pages) * page_size > INT32_MAX) return PA_ERR_INVALID;
  return PA_OK;
}

// Limits of the producer that will run (the selected implementation, the query tile,
// the window bounds), checked before any launch.  The decode-step entry points call it
// before they enqueue the metadata kernel, so a step rejected here changes no output.
pa_status check_producer(int group, bool multi, int32_t max_q_len, int32_t window,
                         int32_t max_seq_pages, int32_t page_size) {
  const bool use_fma = g_producer.load() == PA_PRODUCER_FMA;
  if (multi) {
    if (max_q_len < 1) return PA_ERR_INVALID;
    if (use_fma || static_cast<int64_t>(group) * max_q_len > 16) return PA_ERR_UNSUPPORTED;
  }
  if (use_fma && group > 8) return PA_ERR_UNSUPPORTED;
  if (window != 0) {
    if (window < 0) return PA_ERR_INVALID;
    if (use_fma) return PA_ERR_UNSUPPORTED;
    // keeps every window bound the kernel forms within int32
    if (static_cast<int64_t>(max_seq_pages) * page_size > (int64_t{1} << 29))
      return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

pa_status launch_metadata_checked(const pa::MetadataParams& p, cudaStream_t stream,
                                  int32_t use_pdl) {
  cudaError_t e = pa::launch_metadata(p, stream, use_pdl != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  return from_cuda(e, "metadata launch");
}

}  // namespace

extern "C" {

pa_status pa_build_metadata_full(
    const void* req_pool_indices, const void* seq_lens, int32_t index_bits,
    const int32_t* req_to_token, int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    const int64_t* out_cache_loc, int64_t out_cache_loc_len, const void* qlens,
    int32_t* cache_seqlens, int32_t* cu_seqlens_k, int32_t* cu_seqlens_q,
    int32_t* page_table, int64_t page_table_stride, int32_t* swa_page_table,
    int64_t swa_page_table_stride, int64_t* swa_out_cache_loc, int64_t swa_out_len,
    int32_t bs, int32_t seqlen_offset, int32_t max_seq_pages, int32_t page_size,
    int32_t q_mode, int32_t q_stride, void* stream, int32_t use_pdl) {
  if (index_bits != 32 && index_bits != 64) return PA_ERR_INVALID;
  pa_status st = check_metadata(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                                req_to_token_stride, full_to_swa_mapping,
                                full_to_swa_mapping_len, cache_seqlens, cu_seqlens_k,
                                page_table, page_table_stride, swa_page_table,
                                swa_page_table_stride, bs, max_seq_pages, page_size);
  if (st != PA_OK || bs == 0) return st;
  if (q_mode < 0 || q_mode > 2) return PA_ERR_INVALID;
  if (q_mode != 0 && cu_seqlens_q == nullptr) return PA_ERR_INVALID;
  if (q_mode == 1 && qlens == nullptr) return PA_ERR_INVALID;
  if (swa_out_cache_loc != nullptr) {
    if (full_to_swa_mapping == nullptr || swa_out_len < 0 || out_cache_loc_len < 0)
      return PA_ERR_INVALID;
    if (out_cache_loc_len > 0 && out_cache_loc == nullptr) return PA_ERR_INVALID;
    if (cdiv(swa_out_len, 256) > (1 << 30)) return PA_ERR_INVALID;
  }
  pa::MetadataParams p = {};
  p.req_pool_indices = req_pool_indices;
  p.seq_lens = seq_lens;
  p.req_to_token = req_to_token;
  p.req_to_token_rows = req_to_token_rows;
  p.req_to_token_stride = req_to_token_stride;
  p.full_to_swa_mapping = full_to_swa_mapping;
  p.mapping_len = full_to_swa_mapping_len;
  p.out_cache_loc = out_cache_loc;
  p.num_out_tokens = swa_out_cache_loc != nullptr
                         ? (out_cache_loc_len < swa_out_len ? out_cache_loc_len : swa_out_len)
                         : 0;
  p.qlens = qlens;
  p.cache_seqlens = cache_seqlens;
  p.cu_seqlens_k = cu_seqlens_k;
  p.cu_seqlens_q = cu_seqlens_q;
  p.page_table = page_table;
  p.page_table_stride = page_table_stride;
  p.swa_page_table = swa_page_table;
  p.swa_page_table_stride = swa_page_table_stride;
  p.swa_out_cache_loc = swa_out_cache_loc;
  p.swa_out_len = swa_out_cache_loc != nullptr ? swa_out_len : 0;
  p.bs = bs;
  p.seqlen_offset = seqlen_offset;
  p.max_seq_pages = max_seq_pages;
  p.page_size = page_size;
  p.q_mode = q_mode;
  p.q_stride = q_stride;
  p.idx64 = index_bits == 64;
  p.ts = g_ts.load();
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e, "error word lookup");
  return launch_metadata_checked(p, static_cast<cudaStream_t>(stream), use_pdl);
}

pa_status pa_build_metadata(const int64_t* req_pool_indices, const int64_t* seq_lens,
                            const int32_t* req_to_token, int64_t req_to_token_rows,
                            int64_t req_to_token_stride,
                            const int64_t* full_to_swa_mapping,
                            int64_t full_to_swa_mapping_len, int32_t* cache_seqlens,
                            int32_t* cu_seqlens_k, int32_t* page_table,
                            int64_t page_table_stride, int32_t* swa_page_table,
                            int64_t swa_page_table_stride, int32_t bs,
                            int32_t seqlen_offset, int32_t max_seq_pages,
                            int32_t page_size, void* stream, int32_t use_pdl) {
  return pa_build_metadata_full(
      req_pool_indices, seq_lens, 64, req_to_token, req_to_token_rows, req_to_token_stride,
      full_to_swa_mapping, full_to_swa_mapping_len, nullptr, 0, nullptr, cache_seqlens,
      cu_seqlens_k, nullptr, page_table, page_table_stride, swa_page_table,
      swa_page_table_stride, nullptr, 0, bs, seqlen_offset, max_seq_pages, page_size,
      PA_Q_MODE_NONE, 0, stream, use_pdl);
}

}  // extern "C"

namespace {

pa_status decode_splitk_impl(const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, int32_t kv_dtype,
                             const int32_t* page_table, int64_t page_table_stride,
                             const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                             int32_t max_q_len, int32_t bs, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int64_t num_pages, int32_t max_seq_pages, int32_t window,
                             int32_t num_splits, float sm_scale, float* scratch_m,
                             float* scratch_l, float* scratch_acc, void* stream,
                             int32_t use_pdl) {
  pa_status st = check_attention(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                                 page_table_stride, cache_seqlens, bs, num_q_heads,
                                 num_kv_heads, head_dim, page_size, num_pages, max_seq_pages,
                                 num_splits);
  if (st != PA_OK || bs == 0) return st;
  if (!scratch_m || !scratch_l || !scratch_acc || !aligned16(scratch_acc))
    return PA_ERR_INVALID;
  const int group = num_q_heads / num_kv_heads;
  const bool use_fma = g_producer.load() == PA_PRODUCER_FMA;
  st = check_producer(group, cu_seqlens_q != nullptr, max_q_len, window, max_seq_pages,
                      page_size);
  if (st != PA_OK) return st;
  const int32_t q_rows = cu_seqlens_q != nullptr ? max_q_len : 1;
  int32_t split_pages = max_seq_pages;  // pages the split partition spans
  if (window != 0) {
    const int64_t longest = static_cast<int64_t>(max_seq_pages) * page_size + q_rows;
    if (window > longest) window = static_cast<int32_t>(longest);  // same positions
    split_pages = pa_window_pages(window, q_rows, page_size, max_seq_pages);
  }
  pa::SplitKParams p = {};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.page_table = page_table;
  p.page_table_stride = page_table_stride;
  p.cache_seqlens = cache_seqlens;
  p.num_pages = num_pages;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_seq_pages = max_seq_pages;
  p.pages_per_split = static_cast<int32_t>(cdiv(split_pages, num_splits));
  p.window = window;
  p.bs = bs;
  p.sm_count = sm_count_of_current_device();
  p.hold_loads = g_hold_loads.load();
  p.no_persist = g_no_persist.load();
  p.num_splits = num_splits;
  p.q_scale = sm_scale * 1.4426950408889634f;  // log2(e): the kernel works in base 2
  p.cu_seqlens_q = cu_seqlens_q;
  p.max_q_len = q_rows;
  p.m_out = scratch_m;
  p.l_out = scratch_l;
  p.acc_out = scratch_acc;
  p.ts = g_ts.load();
  cudaError_t e = error_word(&p.err);
  if (e != cudaSuccess) return from_cuda(e, "error word lookup");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (window > 0) {
    e = kv_dtype == PA_KV_INT8
            ? pa::launch_splitk_mma_window_int8(p, bs, group, page_size, s, use_pdl != 0)
            : pa::launch_splitk_mma_window_bf16(p, bs, group, page_size, s, use_pdl != 0);
  } else if (kv_dtype == PA_KV_INT8) {
    e = use_fma ? pa::launch_splitk_int8(p, bs, group, page_size, s, use_pdl != 0)
                : pa::launch_splitk_mma_int8(p, bs, group, page_size, s, use_pdl != 0);
  } else {
    e = use_fma ? pa::launch_splitk_bf16(p, bs, group, page_size, s, use_pdl != 0)
                : pa::launch_splitk_mma_bf16(p, bs, group, page_size, s, use_pdl != 0);
  }
  if (e == cudaSuccess) e = pa::fail_at(cudaGetLastError(), "error state after launch");
  return from_cuda(e, "split-K producer launch");
}

}  // namespace

extern "C" {

pa_status pa_decode_splitk(const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int32_t kv_dtype,
                           const int32_t* page_table, int64_t page_table_stride,
                           const int32_t* cache_seqlens, int32_t bs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           int64_t num_pages, int32_t max_seq_pages, int32_t num_splits,
                           float sm_scale, float* scratch_m, float* scratch_l,
                           float* scratch_acc, void* stream, int32_t use_pdl) {
  return decode_splitk_impl(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                            page_table_stride, cache_seqlens, nullptr, 1, bs, num_q_heads,
                            num_kv_heads, head_dim, page_size, num_pages, max_seq_pages, 0,
                            num_splits, sm_scale, scratch_m, scratch_l, scratch_acc, stream,
                            use_pdl);
}

pa_status pa_decode_splitk_multi(const void* q, const void* k_cache, const void* v_cache,
                                 const float* k_scale, const float* v_scale, int32_t kv_dtype,
                                 const int32_t* page_table, int64_t page_table_stride,
                                 const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                                 int32_t bs, int32_t max_q_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                 int64_t num_pages, int32_t max_seq_pages, int32_t num_splits,
                                 float sm_scale, float* scratch_m, float* scratch_l,
                                 float* scratch_acc, void* stream, int32_t use_pdl) {
  if (cu_seqlens_q == nullptr) return PA_ERR_INVALID;
  return decode_splitk_impl(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                            page_table_stride, cache_seqlens, cu_seqlens_q, max_q_len, bs,
                            num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                            max_seq_pages, 0, num_splits, sm_scale, scratch_m, scratch_l,
                            scratch_acc, stream, use_pdl);
}

pa_status pa_decode_splitk_window(const void* q, const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale, int32_t kv_dtype,
                                  const int32_t* page_table, int64_t page_table_stride,
                                  const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                                  int32_t bs, int32_t max_q_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                  int64_t num_pages, int32_t max_seq_pages,
                                  int32_t sliding_window, int32_t num_splits, float sm_scale,
                                  float* scratch_m, float* scratch_l, float* scratch_acc,
                                  void* stream, int32_t use_pdl) {
  if (sliding_window < 1) return PA_ERR_INVALID;
  return decode_splitk_impl(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                            page_table_stride, cache_seqlens, cu_seqlens_q,
                            cu_seqlens_q != nullptr ? max_q_len : 1, bs, num_q_heads,
                            num_kv_heads, head_dim, page_size, num_pages, max_seq_pages,
                            sliding_window, num_splits, sm_scale, scratch_m, scratch_l,
                            scratch_acc, stream, use_pdl);
}

int32_t pa_window_pages(int32_t sliding_window, int32_t max_q_len, int32_t page_size,
                        int32_t max_seq_pages) {
  if (sliding_window < 1 || max_q_len < 1 || page_size < 1 || max_seq_pages < 1) return 0;
  const int64_t pages = (static_cast<int64_t>(sliding_window) + max_q_len - 2) / page_size + 2;
  return static_cast<int32_t>(pages < max_seq_pages ? pages : max_seq_pages);
}

pa_status pa_reduce(const float* scratch_m, const float* scratch_l, const float* scratch_acc,
                    int32_t bs, int32_t num_q_heads, int32_t head_dim, int32_t num_splits,
                    void* out, float* lse, void* stream, int32_t use_pdl) {
  if (bs < 0 || num_q_heads < 1 || num_splits < 1 || num_splits > 4096) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (!scratch_m || !scratch_l || !scratch_acc || !out) return PA_ERR_INVALID;
  if (!aligned16(scratch_acc) || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return PA_ERR_INVALID;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  pa::ReduceParams p = {};
  p.m = scratch_m;
  p.l = scratch_l;
  p.acc = scratch_acc;
  p.num_rows = static_cast<int64_t>(bs) * num_q_heads;
  p.num_splits = num_splits;
  p.out = out;
  p.lse = lse;
  p.ts = g_ts.load();
  cudaError_t e = pa::launch_reduce(p, static_cast<cudaStream_t>(stream), use_pdl != 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  return from_cuda(e, "reducer launch");
}

size_t pa_workspace_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim,
                          int32_t num_splits) {
  if (bs <= 0 || num_q_heads <= 0 || head_dim <= 0 || num_splits <= 0) return 0;
  const size_t rows = static_cast<size_t>(bs) * num_q_heads * num_splits;
  return 2 * align256(rows * sizeof(float)) + align256(rows * head_dim * sizeof(float));
}

int32_t pa_choose_splits(int32_t bs, int32_t num_kv_heads, int32_t max_seq_pages,
                         int32_t page_size, int32_t kv_dtype, int32_t sm_count) {
  if (bs <= 0 || num_kv_heads <= 0 || max_seq_pages <= 0 || page_size <= 0) return 1;
  if (sm_count <= 0) sm_count = sm_count_of_current_device();
  if (sm_count <= 0) sm_count = 152;
  // About 2048 positions of the longest request per split, for both KV types (GB300
  // sweeps of the whole step: bf16 bs32 ctx 8K best at 5 splits; int8 bs64 ctx 8K
  // best at 4, ragged bs64 / bs32 up to 16K at 6-8, ragged bs64 up to 32K at 6-8 with
  // 16 within 1.2%; the persistent form balances the smaller items that gives).
  // kv_dtype is kept in the signature: the two types have differed.
  (void)kv_dtype;
  const int64_t tokens = static_cast<int64_t>(max_seq_pages) * page_size;
  int64_t want = cdiv(tokens, 2048);
  // ... but at least 2.5 waves of blocks at three resident blocks per SM, so the
  // scheduler can balance ragged requests and the last wave is not most of the step.
  const int64_t units = static_cast<int64_t>(bs) * num_kv_heads;
  const int64_t waves = cdiv(static_cast<int64_t>(sm_count) * 3 * 5, 2 * units);
  if (want < waves) want = waves;
  // At least two 64-token chunks per split keep the per-block prologue amortised.
  const int64_t chunks = cdiv(tokens, 64);
  const int64_t most = chunks / 2 > 0 ? chunks / 2 : 1;
  if (want > most) want = most;
  if (want < 1) want = 1;
  if (want > 4096) want = 4096;
  // Equal page-aligned split length; drop splits the longest request would leave empty.
  const int64_t pages_per_split = cdiv(max_seq_pages, want);
  return static_cast<int32_t>(cdiv(max_seq_pages, pages_per_split));
}

}  // extern "C"

namespace {

// Metadata, producer and reducer; window > 0 runs the sliding-window producer over
// swa_page_table (k/v/scales/num_pages then describe the sliding-window pool).
pa_status decode_step_impl(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_pages, int32_t window, int32_t num_splits,
    float sm_scale, void* workspace, size_t workspace_bytes, void* out, float* lse,
    void* stream, int32_t use_pdl) {
  if (bs < 0) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (num_splits < 0) return PA_ERR_INVALID;
  if (window > 0 && (full_to_swa_mapping == nullptr || swa_page_table == nullptr))
    return PA_ERR_INVALID;
  const int32_t split_pages =
      window > 0 ? pa_window_pages(window, 1, page_size, max_seq_pages) : max_seq_pages;
  const int32_t splits =
      num_splits > 0 ? num_splits
                     : pa_choose_splits(bs, num_kv_heads, split_pages, page_size, kv_dtype, 0);
  pa_status st = check_metadata(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                                req_to_token_stride, full_to_swa_mapping,
                                full_to_swa_mapping_len, cache_seqlens, cu_seqlens_k,
                                page_table, page_table_stride, swa_page_table,
                                swa_page_table_stride, bs, max_seq_pages, page_size);
  if (st != PA_OK) return st;
  const int32_t* attn_table = window > 0 ? swa_page_table : page_table;
  const int64_t attn_stride = window > 0 ? swa_page_table_stride : page_table_stride;
  st = check_attention(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, attn_table,
                       attn_stride, cache_seqlens, bs, num_q_heads, num_kv_heads,
                       head_dim, page_size, num_pages, max_seq_pages, splits);
  if (st != PA_OK) return st;
  if (!out || !workspace || !aligned16(workspace)) return PA_ERR_INVALID;
  if (workspace_bytes < pa_workspace_bytes(bs, num_q_heads, head_dim, splits))
    return PA_ERR_INVALID;
  st = check_producer(num_q_heads / num_kv_heads, false, 1, window, max_seq_pages, page_size);
  if (st != PA_OK) return st;
  const size_t rows = static_cast<size_t>(bs) * num_q_heads * splits;
  char* ws = static_cast<char*>(workspace);
  float* m = reinterpret_cast<float*>(ws);
  float* l = reinterpret_cast<float*>(ws + align256(rows * sizeof(float)));
  float* acc = reinterpret_cast<float*>(ws + 2 * align256(rows * sizeof(float)));

  st = pa_build_metadata(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                         req_to_token_stride, full_to_swa_mapping, full_to_swa_mapping_len,
                         cache_seqlens, cu_seqlens_k, page_table, page_table_stride,
                         swa_page_table, swa_page_table_stride, bs, seqlen_offset,
                         max_seq_pages, page_size, stream, use_pdl);
  if (st != PA_OK) return st;
  st = decode_splitk_impl(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, attn_table,
                          attn_stride, cache_seqlens, nullptr, 1, bs, num_q_heads,
                          num_kv_heads, head_dim, page_size, num_pages, max_seq_pages, window,
                          splits, sm_scale, m, l, acc, stream, use_pdl);
  if (st != PA_OK) return st;
  return pa_reduce(m, l, acc, bs, num_q_heads, head_dim, splits, out, lse, stream, use_pdl);
}

}  // namespace

extern "C" {

pa_status pa_decode_step(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_pages, int32_t num_splits,
    float sm_scale, void* workspace, size_t workspace_bytes, void* out, float* lse,
    void* stream, int32_t use_pdl) {
  return decode_step_impl(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                          req_to_token_stride, full_to_swa_mapping, full_to_swa_mapping_len,
                          seqlen_offset, max_seq_pages, cache_seqlens, cu_seqlens_k, page_table,
                          page_table_stride, swa_page_table, swa_page_table_stride, q, k_cache,
                          v_cache, k_scale, v_scale, kv_dtype, bs, num_q_heads, num_kv_heads,
                          head_dim, page_size, num_pages, 0, num_splits, sm_scale, workspace,
                          workspace_bytes, out, lse, stream, use_pdl);
}

pa_status pa_decode_step_host(
    const void* h_q, const int64_t* h_req_pool_indices, const int64_t* h_seq_lens,
    void* h_out, float* h_lse, const int64_t* req_pool_indices, const int64_t* seq_lens,
    const int32_t* req_to_token, int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_pages, int32_t num_splits,
    float sm_scale, void* workspace, size_t workspace_bytes, void* out, float* lse,
    void* stream, int32_t use_pdl) {
  if (bs < 0 || num_q_heads < 1 || head_dim < 1) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (!h_q || !h_req_pool_indices || !h_seq_lens || !h_out) return PA_ERR_INVALID;
  if (!q || !req_pool_indices || !seq_lens || !out) return PA_ERR_INVALID;
  if ((h_lse == nullptr) != (lse == nullptr)) return PA_ERR_INVALID;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(bs) * num_q_heads;
  const size_t qo_bytes = rows * static_cast<size_t>(head_dim) * 2;
  const size_t idx_bytes = static_cast<size_t>(bs) * sizeof(int64_t);
  cudaError_t e = cudaMemcpyAsync(const_cast<void*>(q), h_q, qo_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<int64_t*>(req_pool_indices), h_req_pool_indices, idx_bytes,
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(const_cast<int64_t*>(seq_lens), h_seq_lens, idx_bytes,
                        cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return from_cuda(e, "host-to-device input copy");
  pa_status st = decode_step_impl(
      req_pool_indices, seq_lens, req_to_token, req_to_token_rows, req_to_token_stride,
      full_to_swa_mapping, full_to_swa_mapping_len, seqlen_offset, max_seq_pages, cache_seqlens,
      cu_seqlens_k, page_table, page_table_stride, swa_page_table, swa_page_table_stride, q,
      k_cache, v_cache, k_scale, v_scale, kv_dtype, bs, num_q_heads, num_kv_heads, head_dim,
      page_size, num_pages, 0, num_splits, sm_scale, workspace, workspace_bytes, out, lse, stream,
      use_pdl);
  if (st != PA_OK) return st;
  e = cudaMemcpyAsync(h_out, out, qo_bytes, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && h_lse != nullptr)
    e = cudaMemcpyAsync(h_lse, lse, rows * sizeof(float), cudaMemcpyDeviceToHost, s);
  return from_cuda(e, "device-to-host output copy");
}

size_t pa_packed_input_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim) {
  if (bs <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return static_cast<size_t>(bs) * num_q_heads * head_dim * 2 + 2 * sizeof(int64_t) * bs;
}

size_t pa_packed_output_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim) {
  if (bs <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return static_cast<size_t>(bs) * num_q_heads * (head_dim * 2 + sizeof(float));
}

pa_status pa_decode_step_host_packed(
    const void* h_inputs, void* inputs, void* h_outputs, void* outputs,
    const int32_t* req_to_token, int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* k_cache,
    const void* v_cache, const float* k_scale, const float* v_scale, int32_t kv_dtype,
    int32_t bs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int64_t num_pages, int32_t num_splits, float sm_scale, void* workspace,
    size_t workspace_bytes, void* stream, int32_t use_pdl) {
  if (bs < 0 || num_q_heads < 1 || head_dim < 1) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (!h_inputs || !inputs || !h_outputs || !outputs) return PA_ERR_INVALID;
  if (!aligned16(inputs) || !aligned16(outputs)) return PA_ERR_INVALID;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qo_bytes = static_cast<size_t>(bs) * num_q_heads * head_dim * 2;
  char* in = static_cast<char*>(inputs);
  char* outs = static_cast<char*>(outputs);
  const int64_t* rpi = reinterpret_cast<const int64_t*>(in + qo_bytes);
  const int64_t* sl = rpi + bs;
  float* lse = reinterpret_cast<float*>(outs + qo_bytes);
  cudaError_t e = cudaMemcpyAsync(inputs, h_inputs, pa_packed_input_bytes(bs, num_q_heads, head_dim),
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return from_cuda(e, "host-to-device input copy");
  pa_status st = decode_step_impl(
      rpi, sl, req_to_token, req_to_token_rows, req_to_token_stride, full_to_swa_mapping,
      full_to_swa_mapping_len, seqlen_offset, max_seq_pages, cache_seqlens, cu_seqlens_k,
      page_table, page_table_stride, swa_page_table, swa_page_table_stride, in, k_cache, v_cache,
      k_scale, v_scale, kv_dtype, bs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
      0, num_splits, sm_scale, workspace, workspace_bytes, outs, lse, stream, use_pdl);
  if (st != PA_OK) return st;
  e = cudaMemcpyAsync(h_outputs, outputs, pa_packed_output_bytes(bs, num_q_heads, head_dim),
                      cudaMemcpyDeviceToHost, s);
  return from_cuda(e, "device-to-host output copy");
}

pa_status pa_decode_step_multi(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const int64_t* qlens,
    int32_t q_mode, int32_t q_stride, int32_t* cu_seqlens_q, const void* q, int32_t total_q,
    int32_t max_q_len, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, int32_t kv_dtype, int32_t bs, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, int64_t num_pages,
    int32_t num_splits, float sm_scale, void* workspace, size_t workspace_bytes, void* out,
    float* lse, void* stream, int32_t use_pdl) {
  if (bs < 0 || total_q < 0 || num_splits < 0) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  if (cu_seqlens_q == nullptr || max_q_len < 1) return PA_ERR_INVALID;
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID;
  // the multi-query producer's limits, before anything is enqueued
  pa_status st = check_producer(num_q_heads / num_kv_heads, true, max_q_len, 0, max_seq_pages,
                                page_size);
  if (st != PA_OK) return st;
  const int32_t splits =
      num_splits > 0 ? num_splits
                     : pa_choose_splits(bs, num_kv_heads, max_seq_pages, page_size, kv_dtype, 0);
  if (total_q > 0) {
    if (!out || !workspace || !aligned16(workspace)) return PA_ERR_INVALID;
    if (workspace_bytes < pa_workspace_bytes(total_q, num_q_heads, head_dim, splits))
      return PA_ERR_INVALID;
  }
  // the attention arguments are checked before anything is enqueued
  st = check_attention(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                                 page_table_stride, cache_seqlens, bs, num_q_heads,
                                 num_kv_heads, head_dim, page_size, num_pages, max_seq_pages,
                                 splits);
  if (st != PA_OK) return st;
  st = pa_build_metadata_full(req_pool_indices, seq_lens, 64, req_to_token, req_to_token_rows,
                              req_to_token_stride, full_to_swa_mapping,
                              full_to_swa_mapping_len, nullptr, 0, qlens, cache_seqlens,
                              cu_seqlens_k, cu_seqlens_q, page_table, page_table_stride,
                              swa_page_table, swa_page_table_stride, nullptr, 0, bs,
                              seqlen_offset, max_seq_pages, page_size, q_mode, q_stride, stream,
                              use_pdl);
  if (st != PA_OK || total_q == 0) return st;
  const size_t rows = static_cast<size_t>(total_q) * num_q_heads * splits;
  char* ws = static_cast<char*>(workspace);
  float* m = reinterpret_cast<float*>(ws);
  float* l = reinterpret_cast<float*>(ws + align256(rows * sizeof(float)));
  float* acc = reinterpret_cast<float*>(ws + 2 * align256(rows * sizeof(float)));
  st = decode_splitk_impl(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, page_table,
                          page_table_stride, cache_seqlens, cu_seqlens_q, max_q_len, bs,
                          num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                          max_seq_pages, 0, splits, sm_scale, m, l, acc, stream, use_pdl);
  if (st != PA_OK) return st;
  return pa_reduce(m, l, acc, total_q, num_q_heads, head_dim, splits, out, lse, stream, use_pdl);
}

pa_status pa_decode_step_window(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_swa, const void* v_swa, const float* k_swa_scale, const float* v_swa_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_swa_pages, int32_t sliding_window,
    int32_t num_splits, float sm_scale, void* workspace, size_t workspace_bytes, void* out,
    float* lse, void* stream, int32_t use_pdl) {
  if (sliding_window < 1) return PA_ERR_INVALID;
  return decode_step_impl(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                          req_to_token_stride, full_to_swa_mapping, full_to_swa_mapping_len,
                          seqlen_offset, max_seq_pages, cache_seqlens, cu_seqlens_k, page_table,
                          page_table_stride, swa_page_table, swa_page_table_stride, q, k_swa,
                          v_swa, k_swa_scale, v_swa_scale, kv_dtype, bs, num_q_heads,
                          num_kv_heads, head_dim, page_size, num_swa_pages, sliding_window,
                          num_splits, sm_scale, workspace, workspace_bytes, out, lse, stream,
                          use_pdl);
}

#ifdef PA_TIMESTAMPS
// Instrumented build only (include/pa_timestamps.h).
pa_status pa_set_timestamp_buffer(uint64_t* buffer) {
  g_ts.store(reinterpret_cast<unsigned long long*>(buffer));
  return PA_OK;
}

pa_status pa_set_test_hold_loads(int32_t hold) {
  g_hold_loads.store(hold != 0 ? 1 : 0);
  return PA_OK;
}

pa_status pa_set_test_no_persist(int32_t off) {
  g_no_persist.store(off != 0 ? 1 : 0);
  return PA_OK;
}
#endif

int32_t pa_select_producer(int32_t producer) {
  if (producer != PA_PRODUCER_AUTO && producer != PA_PRODUCER_FMA && producer != PA_PRODUCER_MMA)
    return g_producer.load();
  return g_producer.exchange(producer);
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_SCRATCH_LIMIT: return "step needs more scratch than the static array holds";
  }
  return "unknown status";
}

pa_status pa_read_error_flags(uint32_t* flags, int32_t reset) {
  if (flags == nullptr) return PA_ERR_INVALID;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return from_cuda(e, "cudaDeviceSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_pa_error_flags, sizeof(v));
  if (e != cudaSuccess) return from_cuda(e, "error word read");
  *flags = v;
  if (reset) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_pa_error_flags, &zero, sizeof(zero));
    if (e != cudaSuccess) return from_cuda(e, "error word reset");
  }
  return PA_OK;
}

const char* pa_last_error_string(void) { return g_last_error; }

}  // extern "C"
