// Device helpers shared by the decode-step kernels (sm_103a).
//
// * Programmatic Dependent Launch: griddepcontrol.wait / launch_dependents, the PTX
//   forms of cudaGridDependencySynchronize / cudaTriggerProgrammaticLaunchCompletion
//   (vLLM PR #50230 report, implementation step 2: wait and trigger in the kernel
//   body, cudaLaunchKernelEx with cudaLaunchAttributeProgrammaticStreamSerialization
//   at the launch site).
// * mbarrier + cp.async.bulk: one-dimensional TMA copies of contiguous KV rows into
//   shared memory, completed on a transaction-count barrier.
// * Bounded waits: every spin on an mbarrier gives up after a fixed time, records
//   an error bit and lets the kernel return, so a lost copy cannot hang the GPU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Bits of the library's device-side error word (see pa_read_error_flags).
enum : unsigned int {
  kErrPageOutOfRange = 1u << 0,     // page_table entry outside [0, num_pages)
  kErrPoolRowOutOfRange = 1u << 1,  // req_pool_indices entry outside the table
  kErrSlotOutOfRange = 1u << 2,     // token slot outside full_to_swa_mapping / a table row
  kErrWaitTimeout = 1u << 3,        // an mbarrier wait gave up
  kErrSeqLenOutOfRange = 1u << 4,   // cache_seqlens entry < 0 or beyond the page table
};

// ~2 s: far longer than any copy this library issues takes on a healthy GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void trigger_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make the barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
    }
    if (global_timer_ns() - start > kWaitLimitNs) return false;
  }
}

// L2 policy: KV rows are read exactly once per step, so they are marked evict-first
// and leave the L2 to the small, re-read tensors (page table, scratch, Q).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// One-dimensional bulk copy global -> shared, completing on `bar`.  `bytes` must be a
// multiple of 16 and both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Stage timestamps for measuring launch gaps (builds with -DPA_TIMESTAMPS only; the
// production build compiles these to nothing).  Stage k (0 metadata, 1 producer,
// 2 reducer) owns slots 3k: earliest block entry, 3k+1: earliest pass of
// griddepcontrol.wait, 3k+2: latest warp finish, all %globaltimer nanoseconds.
enum : int { kTsEntry = 0, kTsReady = 1, kTsExit = 2 };
#ifdef PA_TIMESTAMPS
#define PA_TS_FIRST(ts, stage, what)                                                      \
  do {                                                                                   \
    if ((ts) != nullptr && threadIdx.x == 0)                                             \
      atomicMin((ts) + 3 * (stage) + (what), ::pa::global_timer_ns());                   \
  } while (0)
#define PA_TS_LAST(ts, stage)                                                             \
  do {                                                                                   \
    if ((ts) != nullptr && (threadIdx.x & 31) == 0)                                      \
      atomicMax((ts) + 3 * (stage) + ::pa::kTsExit, ::pa::global_timer_ns());            \
  } while (0)
#else
#define PA_TS_FIRST(ts, stage, what) ((void)0)
#define PA_TS_LAST(ts, stage) ((void)0)
#endif

__device__ __forceinline__ void record_error(unsigned int* err, unsigned int bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// bf16x2 word -> two floats (exact: bf16 is the upper half of a binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four signed int8 codes in a word -> floats, exactly.  Each byte is biased to
// unsigned, placed as the low mantissa byte of 2^23 (0x4B000000), and the bias
// 2^23 + 128 is subtracted again.
__device__ __forceinline__ void s8x4_to_float(uint32_t w, float& f0, float& f1, float& f2,
                                              float& f3) {
  const uint32_t u = w ^ 0x80808080u;
  constexpr float kBias = 8388736.0f;  // 2^23 + 128
  f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - kBias;
  f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - kBias;
  f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - kBias;
  f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - kBias;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// ---------------------------------------------------------------------------------
// Host side: launch with or without the programmatic-stream-serialisation attribute.
// ---------------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool use_pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pa
