/*
 * pa.h -- C ABI of the GB300 (sm_103a) decode-step paged-KV attention library.
 *
 * One decode step runs three kernels chained with Programmatic Dependent Launch:
 *
 *   pa_build_metadata  -> pa_decode_splitk  -> pa_reduce
 *   (fused metadata)      (split-K producer)   (log-sum-exp reducer)
 *
 * pa_decode_step issues all three; pa_decode_splitk_multi (several query tokens per
 * request) and pa_decode_splitk_window / pa_decode_step_window (sliding-window layers)
 * are the producer's other forms.  Every entry point takes plain device pointers
 * and sizes, enqueues work on `stream` (a cudaStream_t passed as void*, NULL = the
 * legacy default stream) and returns without synchronising.  The step's own inputs
 * and outputs -- q, req_pool_indices, seq_lens, out, lse -- may instead point into
 * pinned host memory (cudaHostAlloc / cudaHostRegister; with unified addressing the
 * host pointer is the device pointer): the kernels then read and write them over the
 * host link, with no copy on the stream; the result is the same bit for bit.  The
 * K/V pools, scales, req_to_token, metadata outputs and scratch stay in device
 * memory.  No entry point
 * allocates memory: the caller owns every buffer, including the split-K scratch
 * (pa_decode_step_static_scratch uses a scratch array inside the library instead).
 * The metadata, producer, reducer and pa_decode_step(_window) launches are recorded
 * into CUDA graphs by this library's benchmark and tests.  The library keeps
 * per-device state for the life of the process (the device address of its error word,
 * kernel attributes, pa_decode_step_static_scratch's array address): after a
 * cudaDeviceReset, do not call it on that device again.  When use_pdl is non-zero the
 * kernel is launched with the programmatic-stream-serialisation attribute, so it
 * may start while the previous kernel in the stream finishes; each kernel waits
 * (griddepcontrol.wait) before it reads anything an earlier kernel wrote.
 *
 * Errors.  Arguments are checked on the host before any launch:
 *   PA_ERR_INVALID      a required pointer is NULL, a size is negative, a stride is
 *                       smaller than the width it must hold, a pointer is not
 *                       16-byte aligned where stated, or the workspace is too small;
 *   PA_ERR_UNSUPPORTED  a shape this build has no kernel for (see each function);
 *   PA_ERR_CUDA         the launch itself failed (cudaGetLastError after launch).
 * bs == 0 returns PA_OK and launches nothing.  Values that only the device can see
 * (a page index outside the pool, a pool row outside req_to_token, a token slot
 * outside full_to_swa_mapping, a cache length beyond the page table) never cause an
 * out-of-bounds access: the kernel substitutes a safe index, the affected outputs
 * are unspecified, and a bit is set in a device-side error word that
 * pa_read_error_flags returns.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Only the entry points below are exported from the shared library. */
#ifndef PA_API
#define PA_API __attribute__((visibility("default")))
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,
  PA_ERR_UNSUPPORTED = 2,
  PA_ERR_CUDA = 3,
  PA_ERR_SCRATCH_LIMIT = 4 /* pa_decode_step_static_scratch: step needs more scratch
                              than PA_STATIC_SCRATCH_BYTES */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_INT8 = 1 } pa_kv_dtype;

/* Implementations of the split-K producer (pa_select_producer). */
typedef enum {
  PA_PRODUCER_AUTO = 0, /* the tensor-core producer */
  PA_PRODUCER_FMA = 1,  /* CUDA-core FMA producer: G in {1, 2, 4, 8} */
  PA_PRODUCER_MMA = 2   /* tensor-core (mma.sync m16n8k16) producer: G in {1, 2, 4, 8, 16} */
} pa_producer;

/* Bits of the device-side error word (pa_read_error_flags). */
#define PA_DEVERR_PAGE_OUT_OF_RANGE 0x1u     /* page_table entry outside [0, num_pages) */
#define PA_DEVERR_POOL_ROW_OUT_OF_RANGE 0x2u /* req_pool_indices entry outside req_to_token */
#define PA_DEVERR_SLOT_OUT_OF_RANGE 0x4u     /* token slot outside full_to_swa_mapping */
#define PA_DEVERR_WAIT_TIMEOUT 0x8u          /* a shared-memory copy wait gave up (~2 s) */
#define PA_DEVERR_SEQLEN_OUT_OF_RANGE 0x10u  /* cache_seqlens < 0 or > max_seq_pages*page_size */

/* cu_seqlens_q modes of pa_build_metadata_full. */
#define PA_Q_MODE_NONE 0    /* leave cu_seqlens_q untouched (decode, target-verify) */
#define PA_Q_MODE_CUMSUM 1  /* cu_seqlens_q[0] = 0, [i+1] = sum_{j<=i} int32(qlens[j]) */
#define PA_Q_MODE_STRIDED 2 /* cu_seqlens_q[0] = 0, [i+1] = (i+1) * q_stride */

/*
 * pa_build_metadata -- the fused per-step metadata update.
 *
 * Follows sglang "trtllm_mha_graph_metadata.py" (module docstring; kernel
 * update_trtllm_mha_graph_metadata_kernel and its launcher), which replaces about
 * 25 small host-dispatched ops per graph replay with one launch:
 *
 *   cache_seqlens[i] = int32(seq_lens[i] + seqlen_offset)
 *   cu_seqlens_k[0]  = 0;  cu_seqlens_k[i+1] = cu_seqlens_k[i] + cache_seqlens[i]
 *                      (int32, wrapping)
 *   page_table[i,p]  = req_to_token[req_pool_indices[i], p*page_size] / page_size
 *                      for 0 <= p < max_seq_pages (C truncating division)
 *   swa_page_table[i,p] (when full_to_swa_mapping != NULL):
 *                      t = the same req_to_token entry;
 *                      s = t >= 0 ? full_to_swa_mapping[t] : -1;
 *                      s < 0 ? -1 : int32(s / page_size)
 *
 * Arguments (all device pointers, row-major):
 *   req_pool_indices [bs] int64     pool row of each request
 *   seq_lens         [bs] int64
 *   req_to_token     [req_to_token_rows, req_to_token_stride] int32 token slots
 *   full_to_swa_mapping [full_to_swa_mapping_len] int64 or NULL (no sliding window)
 *   cache_seqlens    [bs] int32 (out)
 *   cu_seqlens_k     [bs+1] int32 (out; entry 0 is written as 0)
 *   page_table       [bs, page_table_stride] int32 (out; columns >= max_seq_pages
 *                    are not touched)
 *   swa_page_table   [bs, swa_page_table_stride] int32 (out) -- NULL iff the
 *                    mapping is NULL
 *   page_size >= 1, max_seq_pages >= 0, (max_seq_pages-1)*page_size <
 *   req_to_token_stride when max_seq_pages > 0.
 * With use_pdl, the inputs (req_pool_indices, seq_lens, the req_to_token entries and
 * their full_to_swa_mapping entries) are read before the kernel waits on the previous
 * grid, and the outputs are written after it: the kernel launched just before must
 * not write those inputs after it triggers its dependents (a kernel that never
 * triggers early, as any kernel written without PDL, is always fine).
 * Errors: PA_ERR_INVALID as listed in the file comment.
 */
PA_API pa_status pa_build_metadata(const int64_t* req_pool_indices, const int64_t* seq_lens,
                            const int32_t* req_to_token, int64_t req_to_token_rows,
                            int64_t req_to_token_stride,
                            const int64_t* full_to_swa_mapping,
                            int64_t full_to_swa_mapping_len, int32_t* cache_seqlens,
                            int32_t* cu_seqlens_k, int32_t* page_table,
                            int64_t page_table_stride, int32_t* swa_page_table,
                            int64_t swa_page_table_stride, int32_t bs,
                            int32_t seqlen_offset, int32_t max_seq_pages,
                            int32_t page_size, void* stream, int32_t use_pdl);

/*
 * pa_build_metadata_full -- pa_build_metadata plus the other inputs and optional outputs
 * of the same module.  The [bs] index inputs (req_pool_indices, seq_lens, qlens; "int"
 * in the module's kernel signature) are int64 or int32 per index_bits (64 or 32).
 * cu_seqlens_q in the three modes above (qlens [bs] for PA_Q_MODE_CUMSUM,
 * cu_seqlens_q [bs+1] int32 for modes 1 and 2), and the
 * sliding-window translation of the step's output slots:
 *   for idx < swa_out_len:  idx < num_out_tokens -> loc = out_cache_loc[idx];
 *                                                   loc < 0 ? -1 : full_to_swa_mapping[loc]
 *                           otherwise            -> 0
 *   num_out_tokens = min(swa_out_len, out_cache_loc_len)
 * swa_out_cache_loc [swa_out_len] int64 (out) or NULL; it needs the mapping.
 * With use_pdl, qlens and out_cache_loc are inputs read before the wait too (the
 * same rule as pa_build_metadata's inputs).
 */
PA_API pa_status pa_build_metadata_full(
    const void* req_pool_indices, const void* seq_lens, int32_t index_bits,
    const int32_t* req_to_token, int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    const int64_t* out_cache_loc, int64_t out_cache_loc_len, const void* qlens,
    int32_t* cache_seqlens, int32_t* cu_seqlens_k, int32_t* cu_seqlens_q,
    int32_t* page_table, int64_t page_table_stride, int32_t* swa_page_table,
    int64_t swa_page_table_stride, int64_t* swa_out_cache_loc, int64_t swa_out_len,
    int32_t bs, int32_t seqlen_offset, int32_t max_seq_pages, int32_t page_size,
    int32_t q_mode, int32_t q_stride, void* stream, int32_t use_pdl);

/*
 * pa_decode_splitk -- the split-K paged-attention producer.
 *
 * lmdeploy PR #4861 "perf(cuda): use PDL for paged attention and V4 prefill"
 * (Changes: Split-K paged attention) names the producer that writes per-split
 * partials to scratch, signals its dependents before its final scratch stores, and
 * the reducer that waits immediately before reading them.  The attention is the
 * plain definition: for request b, query head h and kv head h / (Hq/Hkv), over the
 * tokens j < cache_seqlens[b] (token j lives in page page_table[b, j/page_size] at
 * row j % page_size),  x_j = sm_scale * q . K_j.
 *
 * Split s of request b covers token positions [s*L, min((s+1)*L, cache_seqlens[b]))
 * with L = page_size * ceil(max_seq_pages / num_splits) (one split length for the
 * whole batch, page aligned).  For every (b, h, s) it writes
 *   scratch_m   = max_j x_j                     (-inf for an empty split)
 *   scratch_l   = sum_j exp(x_j - scratch_m)    (0 for an empty split)
 *   scratch_acc = sum_j exp(x_j - scratch_m) V_j (not written for an empty split)
 *
 * Layouts (device pointers):
 *   q            [bs, num_q_heads, head_dim] bf16, 16-byte aligned
 *   k_cache, v_cache [num_pages, num_kv_heads, page_size, head_dim], bf16
 *                (PA_KV_BF16) or int8 codes (PA_KV_INT8), 16-byte aligned
 *   k_scale, v_scale [num_pages, num_kv_heads, page_size] fp32, 16-byte aligned;
 *                INT8 only (K = k_scale * code, V = v_scale * code); NULL for BF16
 *   page_table   [bs, page_table_stride] int32; cache_seqlens [bs] int32
 *   scratch_m, scratch_l [bs, num_q_heads, num_splits] fp32
 *   scratch_acc  [bs, num_q_heads, num_splits, head_dim] fp32
 * Supported: head_dim 128; page_size 16, 32, 64, 128; num_q_heads/num_kv_heads in
 * {1, 2, 4, 8, 16} (16 only with the tensor-core producer); otherwise
 * PA_ERR_UNSUPPORTED.  Which producer implementation runs is chosen with
 * pa_select_producer; both compute the same partials (to rounding).
 * With use_pdl, q is read before the kernel waits on the previous grid (the prologue
 * overlaps the metadata stage): the kernel launched just before must not write q.
 */
PA_API pa_status pa_decode_splitk(const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int32_t kv_dtype,
                           const int32_t* page_table, int64_t page_table_stride,
                           const int32_t* cache_seqlens, int32_t bs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           int64_t num_pages, int32_t max_seq_pages, int32_t num_splits,
                           float sm_scale, float* scratch_m, float* scratch_l,
                           float* scratch_acc, void* stream, int32_t use_pdl);

/*
 * pa_decode_splitk_multi -- the producer for several query tokens per request
 * (speculative target-verify / draft-extend steps, whose query lengths the metadata
 * module's cu_seqlens_q describes).  Query rows of request b are
 * q[cu_seqlens_q[b] .. cu_seqlens_q[b+1]) ([total_q, num_q_heads, head_dim] bf16), at most
 * max_q_len per request; they are the request's newest tokens, already in its cache,
 * so query i (0-based) attends causally to token positions j < n - q_len + i + 1,
 * n = cache_seqlens[b].  Splits, layouts and partial semantics are those of
 * pa_decode_splitk with one scratch row per query row: scratch_m/l
 * [total_q, num_q_heads, num_splits], scratch_acc [total_q, num_q_heads, num_splits,
 * head_dim]; pa_reduce with bs = total_q combines them.  cu_seqlens_q [bs+1] int32 is
 * read after the wait on the previous grid (it may be the metadata stage's output).
 * Tensor-core producer only: PA_ERR_UNSUPPORTED when (num_q_heads/num_kv_heads) *
 * max_q_len > 16 or the CUDA-core producer is selected.  A query whose causal range is
 * empty gets m = -inf in every split (out = 0, lse = -inf after pa_reduce).
 */
PA_API pa_status pa_decode_splitk_multi(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, int32_t kv_dtype, const int32_t* page_table, int64_t page_table_stride,
    const int32_t* cache_seqlens, const int32_t* cu_seqlens_q, int32_t bs, int32_t max_q_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int64_t num_pages, int32_t max_seq_pages, int32_t num_splits, float sm_scale,
    float* scratch_m, float* scratch_l, float* scratch_acc, void* stream, int32_t use_pdl);

/*
 * pa_decode_splitk_window -- the producer for sliding-window attention layers, reading
 * the sliding-window pool through the sliding-window page table that the metadata
 * module builds (sglang trtllm_mha_graph_metadata.py, module docstring: swa_page_table
 * = full_to_swa_mapping[token] // page_size, -1 where the slot is unmapped).  The pages
 * build that table but print no attention that reads it; this call is the plainest
 * reading:
 *   query i of request b (position pos = n - q_len + i, n = cache_seqlens[b]) attends the
 *   positions j with max(0, pos - sliding_window + 1) <= j <= pos whose table entry
 *   page_table[b, j / page_size] is >= 0; token j is row j % page_size of that page of
 *   the pool (k_cache / v_cache / scales laid out as for pa_decode_splitk).  Pages with a
 *   -1 entry are skipped: nothing is loaded from them and their tokens are not attended.
 * Query rows: one per request (row b) when cu_seqlens_q is NULL, else as for
 * pa_decode_splitk_multi (max_q_len queries at most per request).
 * Split partition: the splits cover the window rather than the whole context.  With
 * W = pa_window_pages(sliding_window, q_len_max, page_size, max_seq_pages) (q_len_max =
 * max_q_len, or 1 without cu_seqlens_q) and L = page_size * ceil(W / num_splits), split
 * s of request b holds positions [base + s L, base + (s+1) L), base = page_size *
 * floor(max(0, n - q_len - sliding_window + 1) / page_size) (the page of the request's
 * first visible position).  Scratch layouts and the empty-split convention are those of
 * pa_decode_splitk(_multi); pa_reduce combines them.
 * page_table here is the sliding-window table ([bs, page_table_stride] int32, entries
 * -1 or in [0, num_pages)) and num_pages the sliding-window pool's page count.
 * Errors: PA_ERR_INVALID for sliding_window < 1 and as pa_decode_splitk(_multi);
 * PA_ERR_UNSUPPORTED when the CUDA-core producer is selected, when
 * max_seq_pages * page_size > 2^29, or as pa_decode_splitk_multi for cu_seqlens_q.
 */
PA_API pa_status pa_decode_splitk_window(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, int32_t kv_dtype, const int32_t* page_table, int64_t page_table_stride,
    const int32_t* cache_seqlens, const int32_t* cu_seqlens_q, int32_t bs, int32_t max_q_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int64_t num_pages, int32_t max_seq_pages, int32_t sliding_window, int32_t num_splits,
    float sm_scale, float* scratch_m, float* scratch_l, float* scratch_acc, void* stream,
    int32_t use_pdl);

/*
 * Pages a sliding-window split partition spans: min(max_seq_pages,
 * floor((sliding_window + max_q_len - 2) / page_size) + 2), the most pages that the
 * sliding_window + max_q_len - 1 consecutive positions a request's queries can see may
 * touch.  0 for a non-positive argument.  pa_choose_splits(bs, num_kv_heads, this,
 * page_size, kv_dtype, 0) is the split count pa_decode_step_window picks.
 */
PA_API int32_t pa_window_pages(int32_t sliding_window, int32_t max_q_len, int32_t page_size,
                               int32_t max_seq_pages);

/*
 * pa_reduce -- the log-sum-exp reducer (the standard and quantized reducer paths of
 * lmdeploy PR #4861 read the same fp32 partials, so one reducer serves both KV types):
 *   M = max_s m_s;  L = sum_s l_s exp(m_s - M)
 *   out[b,h,:] = bf16_rne( sum_s acc_s exp(m_s - M) / L )
 *   lse[b,h]   = M + ln L   (natural log of the sum of exp of the scaled scores)
 * Splits with m_s = -inf are skipped without reading their acc.  A request with no
 * tokens gives out = 0 and lse = -inf.
 *   out [bs, num_q_heads, head_dim] bf16; lse [bs, num_q_heads] fp32 or NULL.
 * Supported: head_dim 128.
 */
PA_API pa_status pa_reduce(const float* scratch_m, const float* scratch_l, const float* scratch_acc,
                    int32_t bs, int32_t num_q_heads, int32_t head_dim, int32_t num_splits,
                    void* out, float* lse, void* stream, int32_t use_pdl);

/*
 * pa_decode_step -- metadata, producer and reducer in one call (three launches; the
 * second and third carry the PDL attribute when use_pdl is non-zero, the first
 * too, and it waits before writing anything).  Arguments are those of the three
 * functions above.  With use_pdl the step's inputs -- q and the metadata inputs --
 * are read before the step waits on the kernel launched before it (the metadata
 * kernel triggers its dependents on entry, so the producer's Q prologue can run while
 * that kernel finishes): that kernel must not write them after it triggers its
 * dependents (a kernel that never triggers early is always fine).  The split-K
 * scratch is carved from `workspace` (workspace_bytes >= pa_workspace_bytes(bs,
 * num_q_heads, head_dim, S)), where S is num_splits, or pa_choose_splits(bs,
 * num_kv_heads, max_seq_pages, page_size, kv_dtype, 0) when num_splits == 0.
 */
PA_API pa_status pa_decode_step(
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
    void* stream, int32_t use_pdl);

/*
 * pa_decode_step_host -- pa_decode_step for callers whose per-step inputs and outputs
 * live in host memory.  Enqueued on `stream`, in order: three host-to-device copies
 * (h_q -> q, h_req_pool_indices -> req_pool_indices, h_seq_lens -> seq_lens; q,
 * req_pool_indices and seq_lens are the caller's device buffers, overwritten here), the
 * three kernels of pa_decode_step, and two device-to-host copies (out -> h_out,
 * lse -> h_lse).  Returns without synchronising: the host outputs are valid once the
 * stream has completed.  h_* should be page-locked (cudaHostAlloc / pinned) for the
 * copies to be asynchronous; pageable memory works but the copies then block the host.
 * (pa_decode_step_host_packed does the same with one copy each way.)
 *   h_q    [bs, num_q_heads, head_dim] bf16     h_req_pool_indices, h_seq_lens [bs] int64
 *   h_out  [bs, num_q_heads, head_dim] bf16     h_lse [bs, num_q_heads] fp32 or NULL
 *                                               (NULL exactly when lse is NULL)
 * The remaining arguments are those of pa_decode_step.  Errors: PA_ERR_INVALID for a
 * NULL host or device buffer, and as pa_decode_step; a failed copy returns PA_ERR_CUDA.
 */
PA_API pa_status pa_decode_step_host(
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
    void* stream, int32_t use_pdl);

/*
 * pa_decode_step_host_packed -- pa_decode_step_host with the per-step inputs in one
 * buffer and the outputs in another, so a step makes one host-to-device and one
 * device-to-host copy (each copy has a fixed latency well above the transfer time of
 * these few hundred KB).  Layout, the same in host and device memory:
 *   inputs   q [bs, num_q_heads, head_dim] bf16, then req_pool_indices [bs] int64,
 *            then seq_lens [bs] int64, back to back: pa_packed_input_bytes() bytes
 *   outputs  out [bs, num_q_heads, head_dim] bf16, then lse [bs, num_q_heads] fp32,
 *            back to back: pa_packed_output_bytes() bytes
 * h_inputs / h_outputs are one host allocation each (page-locked for asynchronous
 * copies); inputs / outputs one device allocation each, 16-byte aligned.  Enqueued on
 * `stream`: h_inputs -> inputs, the three kernels of pa_decode_step reading q,
 * req_pool_indices and seq_lens from `inputs` and writing out and lse into `outputs`,
 * outputs -> h_outputs.  The remaining arguments are those of pa_decode_step.  Errors:
 * PA_ERR_INVALID for a NULL or misaligned buffer, and as pa_decode_step; a failed copy
 * returns PA_ERR_CUDA.
 */
PA_API size_t pa_packed_input_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim);
PA_API size_t pa_packed_output_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim);
PA_API pa_status pa_decode_step_host_packed(
    const void* h_inputs, void* inputs, void* h_outputs, void* outputs,
    const int32_t* req_to_token, int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* k_cache,
    const void* v_cache, const float* k_scale, const float* v_scale, int32_t kv_dtype,
    int32_t bs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int64_t num_pages, int32_t num_splits, float sm_scale, void* workspace,
    size_t workspace_bytes, void* stream, int32_t use_pdl);

/*
 * pa_decode_step_multi -- the decode step for several query tokens per request
 * (speculative target-verify / draft-extend steps): pa_build_metadata_full with the
 * query side of the metadata module (q_mode PA_Q_MODE_NONE: cu_seqlens_q is preset by
 * the caller; PA_Q_MODE_CUMSUM: cu_seqlens_q[1:] = cumsum(qlens) (qlens [bs] int64);
 * PA_Q_MODE_STRIDED: cu_seqlens_q[i] = i * q_stride), then pa_decode_splitk_multi over
 * those rows, then pa_reduce over the total_q rows.
 *   q [total_q, num_q_heads, head_dim] bf16, out [total_q, num_q_heads, head_dim] bf16,
 *   lse [total_q, num_q_heads] fp32 or NULL; total_q must equal cu_seqlens_q[bs] (the
 *   caller sized q by it); every request has at most max_q_len query rows.
 * The split-K scratch is carved from `workspace`, which must hold
 * pa_workspace_bytes(total_q, num_q_heads, head_dim, S), S = num_splits or
 * pa_choose_splits(bs, num_kv_heads, max_seq_pages, page_size, kv_dtype, 0).  The other
 * arguments are those of pa_decode_step.  Errors as the calls it makes; PA_ERR_INVALID
 * for a NULL cu_seqlens_q or max_q_len < 1.  total_q == 0 runs the metadata stage only.
 */
PA_API pa_status pa_decode_step_multi(
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
    float* lse, void* stream, int32_t use_pdl);

/*
 * pa_decode_step_window -- pa_decode_step for a sliding-window attention layer: the
 * metadata stage (full_to_swa_mapping and swa_page_table are required here), then
 * pa_decode_splitk_window over swa_page_table with one query per request, then
 * pa_reduce.  k_swa / v_swa / the scales and num_swa_pages describe the sliding-window
 * pool.  With num_splits == 0 the split count is
 * pa_choose_splits(bs, num_kv_heads, pa_window_pages(sliding_window, 1, page_size,
 * max_seq_pages), page_size, kv_dtype, 0), and the workspace must hold
 * pa_workspace_bytes(bs, num_q_heads, head_dim, that count).  Errors as the calls it makes.
 */
PA_API pa_status pa_decode_step_window(
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
    float* lse, void* stream, int32_t use_pdl);

/*
 * pa_decode_step_static_scratch -- pa_decode_step for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call; it is an addition of
 * this library.
 *
 * Some callers cannot call cudaMalloc where they run a decode step: runtimes whose
 * device memory is owned entirely by their own allocator or fixed at start-up (a
 * cudaMalloc behind the allocator's back takes memory it has already handed out, or
 * fails), code on a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable, and plain C hosts that link this library but have
 * no device allocator of their own.  This call takes the same arguments as
 * pa_decode_step except the workspace: the split-K scratch comes from an array of
 * PA_STATIC_SCRATCH_BYTES compiled into the library.  Inputs and outputs are still the
 * caller's.
 *   - Every GPU that loads the library holds that array until the process exits.
 *   - A step whose scratch, pa_workspace_bytes(bs, num_q_heads, head_dim, S), exceeds
 *     PA_STATIC_SCRATCH_BYTES returns PA_ERR_SCRATCH_LIMIT and launches nothing.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture.  A cudaDeviceReset destroys
 *     the array together with the context, and the kept address then names nothing:
 *     do not call the library on that device again afterwards.
 *   - All calls share the array and it keeps the last call's contents (nothing in it
 *     needs to start at zero).  Calls whose work overlaps on the GPU race on it: keep
 *     them in order on one stream.
 *   - It allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
#define PA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

PA_API pa_status pa_decode_step_static_scratch(
    const int64_t* req_pool_indices, const int64_t* seq_lens, const int32_t* req_to_token,
    int64_t req_to_token_rows, int64_t req_to_token_stride,
    const int64_t* full_to_swa_mapping, int64_t full_to_swa_mapping_len,
    int32_t seqlen_offset, int32_t max_seq_pages, int32_t* cache_seqlens,
    int32_t* cu_seqlens_k, int32_t* page_table, int64_t page_table_stride,
    int32_t* swa_page_table, int64_t swa_page_table_stride, const void* q,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    int32_t kv_dtype, int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t page_size, int64_t num_pages, int32_t num_splits,
    float sm_scale, void* out, float* lse, void* stream, int32_t use_pdl);

/* Bytes of workspace pa_decode_step needs: m, l and acc partials, each 256-byte aligned. */
PA_API size_t pa_workspace_bytes(int32_t bs, int32_t num_q_heads, int32_t head_dim,
                          int32_t num_splits);

/*
 * Split count heuristic, measured on GB300: a split holds about 2048 positions of the
 * longest request (bf16 and int8 KV alike), but there are at least 2.5 waves of
 * (request, kv head, split) blocks at three resident blocks per SM; each split holds at
 * least two 64-token chunks, its length is page-aligned, and no split count leaves the
 * longest request with an empty split.  kv_dtype is PA_KV_BF16 or PA_KV_INT8 (any other
 * value is read as bf16); sm_count <= 0 queries the current device.  Returns >= 1
 * (1 for degenerate sizes).
 */
PA_API int32_t pa_choose_splits(int32_t bs, int32_t num_kv_heads, int32_t max_seq_pages,
                                int32_t page_size, int32_t kv_dtype, int32_t sm_count);

/*
 * Choose the split-K producer implementation for later calls in this process
 * (PA_PRODUCER_AUTO, _FMA or _MMA); returns the previous choice.  An unknown value
 * changes nothing and returns the current choice.  Meant for A/B measurement.
 */
PA_API int32_t pa_select_producer(int32_t producer);

/*
 * Description of the last CUDA failure an entry point saw on the calling host thread
 * (the call that failed and the CUDA error), or "no CUDA error".  The string stays
 * valid until the next failing call on that thread.
 */
PA_API const char* pa_last_error_string(void);

/* Static description of a status code. */
PA_API const char* pa_status_string(pa_status status);

/*
 * Read (and, when reset != 0, clear) the current device's error word.  This call
 * synchronises the device; it is for tests and diagnostics, not the hot path.
 */
PA_API pa_status pa_read_error_flags(uint32_t* flags, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
