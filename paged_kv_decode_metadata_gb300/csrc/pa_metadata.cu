// Fused decode-step metadata update, one launch per step.
//
// Semantics: sglang "trtllm_mha_graph_metadata.py" (module docstring and the kernel
// update_trtllm_mha_graph_metadata_kernel): cache_seqlens, the int32 cu_seqlens_k
// scan, the page_table gather from req_to_token, the optional sliding-window page
// table through full_to_swa_mapping with the -1 sentinel, the optional cu_seqlens_q
// modes and the optional swa_out_cache_loc translation.
//
// Grid: blocks [0, bs) each own one request row (its cache_seqlens entry and its
// page-table row(s)); block bs runs the in-block scans; blocks after it translate
// swa_out_cache_loc in tiles of kThreads entries.  Every block triggers its
// dependents on entry, so the producer's blocks become resident and load Q while
// this grid still runs: the producer reads nothing of this kernel's outputs before
// its own griddepcontrol.wait, which blocks until this grid has completed and
// flushed.  Each block then reads its inputs (request rows, lengths, the gathered
// token slots and their sliding-window translations) and only then waits on the
// previous grid, before its first global write, so a PDL launch never overwrites a
// page table that a previous step's producer may still read.  Reading the inputs
// before the wait is the same contract as the producer's Q prologue: they must be
// complete when the kernel launched before this one triggers its dependents (always
// true of a kernel that does not trigger early).  (All of this grid's blocks are
// resident before the producer can launch, since a grid triggers only once every
// block has issued the trigger; the early producer blocks cannot hold SMs this grid
// still needs.)
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
// page-table columns per thread whose inputs are read before the wait (rows of at most
// kPre * kThreads pages are read entirely before it)
constexpr int kPre = 4;

// Index inputs ([bs] "int" in the source module) may be int64 or int32.
__device__ __forceinline__ int64_t load_index(const void* p, int64_t i, bool is64) {
  return is64 ? static_cast<const int64_t*>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t*>(p)[i]);
}

// Block-wide inclusive scan of one uint32 per thread (wrapping adds).  Returns the
// thread's inclusive prefix; *total receives the block total.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t up = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += up;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kThreads / 32 ? warp_sums[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t up = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += up;
    }
    if (lane < kThreads / 32) warp_sums[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[kThreads / 32 - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return v + before;
}

__global__ void __launch_bounds__(kThreads) metadata_kernel(const MetadataParams p) {
  PA_TS_FIRST(p.ts, 0, kTsEntry);
  trigger_dependents();

  const int tid = threadIdx.x;
  const int blk = blockIdx.x;

  if (blk < p.bs) {
    // ---- one request row -------------------------------------------------------
    // inputs first: the row, the length and the first kPre * kThreads token slots (and
    // their sliding-window slots); columns past those are read after the wait
    const int i = blk;
    int64_t row = load_index(p.req_pool_indices, i, p.idx64);
    const bool row_ok = row >= 0 && row < p.req_to_token_rows;
    if (!row_ok) row = 0;
    int64_t seq_len = 0;
    if (tid == 0) seq_len = load_index(p.seq_lens, i, p.idx64);
    const int32_t* row_in = p.req_to_token + row * p.req_to_token_stride;
    const bool swa = p.swa_page_table != nullptr;
    auto token_at = [&](int col) -> int32_t {
      return row_ok ? row_in[static_cast<int64_t>(col) * p.page_size] : 0;
    };
    // sliding-window slot of a token slot (-1: none); *bad when the slot is out of range
    auto swa_slot = [&](int32_t token, bool* bad) -> int64_t {
      if (token < 0) return -1;
      if (token < p.mapping_len) return p.full_to_swa_mapping[token];
      *bad = true;
      return -1;
    };
    int32_t tok[kPre];
    int64_t stok[kPre];
    bool slot_bad = false;
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const int col = tid + k * kThreads;
      tok[k] = col < p.max_seq_pages ? token_at(col) : 0;
    }
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const int col = tid + k * kThreads;
      stok[k] = swa && col < p.max_seq_pages ? swa_slot(tok[k], &slot_bad) : -1;
    }

    grid_dependency_wait();
    PA_TS_FIRST(p.ts, 0, kTsReady);
    if (!row_ok && tid == 0) record_error(p.err, kErrPoolRowOutOfRange);
    if (tid == 0) {
      const uint64_t sum = static_cast<uint64_t>(seq_len) +
                           static_cast<uint64_t>(static_cast<int64_t>(p.seqlen_offset));
      p.cache_seqlens[i] = static_cast<int32_t>(static_cast<uint32_t>(sum));
    }
    int32_t* row_out = p.page_table + static_cast<int64_t>(i) * p.page_table_stride;
    int32_t* swa_out = swa ? p.swa_page_table + static_cast<int64_t>(i) * p.swa_page_table_stride
                           : nullptr;
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const int col = tid + k * kThreads;
      if (col < p.max_seq_pages) {
        row_out[col] = tok[k] / p.page_size;
        if (swa) swa_out[col] = stok[k] < 0 ? -1 : static_cast<int32_t>(stok[k] / p.page_size);
      }
    }
    for (int col = tid + kPre * kThreads; col < p.max_seq_pages; col += kThreads) {
      const int32_t token = token_at(col);
      row_out[col] = token / p.page_size;
      if (swa) {
        const int64_t s = swa_slot(token, &slot_bad);
        swa_out[col] = s < 0 ? -1 : static_cast<int32_t>(s / p.page_size);
      }
    }
    if (slot_bad) record_error(p.err, kErrSlotOutOfRange);
    PA_TS_LAST(p.ts, 0);
    return;
  }

  if (blk == p.bs) {
    // ---- scans: cu_seqlens_k, and cu_seqlens_q in the computed modes -------------
    // the first tile of lengths is read before the wait, later tiles after it
    const uint32_t k0 = tid < p.bs ? static_cast<uint32_t>(load_index(p.seq_lens, tid, p.idx64)) : 0u;
    const uint32_t q0 =
        p.q_mode == 1 && tid < p.bs ? static_cast<uint32_t>(load_index(p.qlens, tid, p.idx64)) : 0u;
    grid_dependency_wait();
    PA_TS_FIRST(p.ts, 0, kTsReady);
    __shared__ uint32_t warp_sums[kThreads / 32];
    uint32_t carry = 0;
    for (int base = 0; base < p.bs; base += kThreads) {
      const int j = base + tid;
      const uint32_t len =
          base == 0 ? k0 : j < p.bs ? static_cast<uint32_t>(load_index(p.seq_lens, j, p.idx64)) : 0u;
      const uint32_t v = j < p.bs ? len + static_cast<uint32_t>(p.seqlen_offset) : 0u;
      uint32_t total;
      const uint32_t incl = block_inclusive_scan(v, warp_sums, &total);
      if (j < p.bs) p.cu_seqlens_k[j + 1] = static_cast<int32_t>(incl + carry);
      carry += total;
    }
    if (tid == 0) p.cu_seqlens_k[0] = 0;
    if (p.q_mode == 1) {
      carry = 0;
      for (int base = 0; base < p.bs; base += kThreads) {
        const int j = base + tid;
        const uint32_t v =
            base == 0 ? q0 : j < p.bs ? static_cast<uint32_t>(load_index(p.qlens, j, p.idx64)) : 0u;
        uint32_t total;
        const uint32_t incl = block_inclusive_scan(v, warp_sums, &total);
        if (j < p.bs) p.cu_seqlens_q[j + 1] = static_cast<int32_t>(incl + carry);
        carry += total;
      }
      if (tid == 0) p.cu_seqlens_q[0] = 0;
    } else if (p.q_mode == 2) {
      for (int j = tid; j < p.bs; j += kThreads) {
        p.cu_seqlens_q[j + 1] =
            static_cast<int32_t>(static_cast<uint32_t>(j + 1) * static_cast<uint32_t>(p.q_stride));
      }
      if (tid == 0) p.cu_seqlens_q[0] = 0;
    }
    PA_TS_LAST(p.ts, 0);
    return;
  }

  // ---- swa_out_cache_loc tile ------------------------------------------------------
  const int64_t idx = static_cast<int64_t>(blk - p.bs - 1) * kThreads + tid;
  int64_t value = 0;
  bool bad = false;
  if (idx < p.num_out_tokens) {
    const int64_t loc = p.out_cache_loc[idx];
    if (loc < 0) {
      value = -1;
    } else if (loc < p.mapping_len) {
      value = p.full_to_swa_mapping[loc];
    } else {
      bad = true;
      value = -1;
    }
  }
  grid_dependency_wait();
  PA_TS_FIRST(p.ts, 0, kTsReady);
  if (bad) record_error(p.err, kErrSlotOutOfRange);
  if (idx < p.swa_out_len) p.swa_out_cache_loc[idx] = value;
  PA_TS_LAST(p.ts, 0);
}

}  // namespace

cudaError_t launch_metadata(const MetadataParams& p, cudaStream_t stream, bool use_pdl) {
  const int64_t out_blocks =
      p.swa_out_cache_loc != nullptr ? (p.swa_out_len + kThreads - 1) / kThreads : 0;
  const dim3 grid(static_cast<unsigned>(p.bs + 1 + out_blocks));
  return launch_kernel(metadata_kernel, grid, dim3(kThreads), 0, stream, use_pdl, p);
}

}  // namespace pa
