// pa_decode_step_static_scratch: the decode step with its split-K scratch taken from
// a fixed array compiled into this library instead of a caller-provided workspace.
//
// It exists for callers that cannot allocate device memory at the point where they
// run a decode step: runtimes whose device memory is handed out entirely by their own
// allocator or fixed at start-up (a cudaMalloc behind the allocator's back takes memory
// it has already promised, or fails), code on a latency-critical path where cudaMalloc's
// implicit device synchronisation is not acceptable, and plain C hosts that link this
// library but have no device allocator of their own.  Such a caller still passes its
// inputs and outputs; only the scratch moves here.
//
// Costs and rules:
//   * Every GPU that loads the library holds PA_STATIC_SCRATCH_BYTES for the array
//     until the process exits.
//   * All calls share the one array and it keeps the last call's contents.  Nothing in
//     it has to start at zero: the producer writes every max and sum entry and every
//     accumulator row the reducer then reads.  Two calls whose work overlaps on the GPU
//     (different streams, or graphs replayed concurrently) race on the array and give
//     wrong results; order them on one stream.
//   * The first call on a device looks up the array's device address (once per device,
//     with that device current) and keeps it for the life of the process.  Make that
//     first call before any stream capture.  After a cudaDeviceReset the kept address
//     names nothing: the library must not be called on that device again.
//   * A step that needs more scratch than the array holds is rejected with
//     PA_ERR_SCRATCH_LIMIT before anything is launched.
//   * Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library call.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// The scratch array.  In host code this name is only a host-side stand-in, not a
// device address; host code must use the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_scratch_addr[kMaxDevices];

// Device address of the array on the current device, looked up once per device.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_static_scratch_addr[dev].load();
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_pa_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_addr[dev].store(p);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_step_static_scratch(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_pages, int32_t num_splits,
    float sm_scale, void* out, float* lse, void* stream, int32_t use_pdl) {
  if (bs < 0 || num_splits < 0) return PA_ERR_INVALID;
  if (bs == 0) return PA_OK;
  const int32_t splits =
      num_splits > 0 ? num_splits
                     : pa_choose_splits(bs, num_kv_heads, max_seq_pages, page_size, kv_dtype,
                                        0);
  const size_t need = pa_workspace_bytes(bs, num_q_heads, head_dim, splits);
  if (need == 0) return PA_ERR_INVALID;
  if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const cudaError_t e = static_scratch_address(&scratch);
  if (e != cudaSuccess) return pa::from_cuda(e, "static scratch address");
  return pa_decode_step(req_pool_indices, seq_lens, req_to_token, req_to_token_rows,
                        req_to_token_stride, full_to_swa_mapping, full_to_swa_mapping_len,
                        seqlen_offset, max_seq_pages, cache_seqlens, cu_seqlens_k, page_table,
                        page_table_stride, swa_page_table, swa_page_table_stride, q, k_cache,
                        v_cache, k_scale, v_scale, kv_dtype, bs, num_q_heads, num_kv_heads,
                        head_dim, page_size, num_pages, splits, sm_scale, scratch,
                        PA_STATIC_SCRATCH_BYTES, out, lse, stream, use_pdl);
}
