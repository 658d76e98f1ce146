// Log-sum-exp reducer of the split-K decode attention.
//
// lmdeploy PR #4861 (Changes: Split-K paged attention): the reducer is launched
// with PDL and waits immediately before it reads the producer's scratch.  The
// combination is the standard one: M = max_s m_s, L = sum_s l_s e^(m_s - M),
// out = sum_s acc_s e^(m_s - M) / L, lse = M + ln L.
//
// One warp per (request, query head) row; a lane owns 4 of the 128 channels, so a
// split's accumulator row is one coalesced 512-byte read.  Split weights are kept
// in shared memory (one slot per split per warp).  Empty splits (m = -inf) are
// skipped without touching their accumulator.
#include <math_constants.h>

#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__global__ void __launch_bounds__(kThreads) reduce_kernel(const ReduceParams p) {
  extern __shared__ float weights[];  // [kWarps][num_splits]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int S = p.num_splits;
  float* w = weights + warp * S;

  PA_TS_FIRST(p.ts, 2, kTsEntry);
  grid_dependency_wait();  // the producer's partials are complete and visible
  PA_TS_FIRST(p.ts, 2, kTsReady);
  if (row >= p.num_rows) {
    PA_TS_LAST(p.ts, 2);
    return;
  }

  const float* m = p.m + row * S;
  const float* l = p.l + row * S;
  float mx = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, m[s]);
  mx = warp_max(mx);

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + row * 128 + lane * 4;
  if (mx == -CUDART_INF_F) {  // no tokens at all
    trigger_dependents();
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    if (p.lse != nullptr && lane == 0) p.lse[row] = -CUDART_INF_F;
    PA_TS_LAST(p.ts, 2);
    return;
  }

  float total = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float ms = m[s];
    const float ws = ms == -CUDART_INF_F ? 0.f : expf(ms - mx);
    w[s] = ws;
    if (ws != 0.f) total += ws * l[s];
  }
  total = warp_sum(total);
  __syncwarp();

  // Batches of 8 independent row loads; an empty split's row is loaded (it lies inside
  // the scratch buffer) but never used, its contents may be anything.
  const float4* acc = reinterpret_cast<const float4*>(p.acc + row * S * 128) + lane;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += 8) {
    float4 a[8];
    float ws[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int s = min(s0 + k, S - 1);
      ws[k] = s0 + k < S ? w[s] : 0.f;
      a[k] = acc[s * 32];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (ws[k] != 0.f) {
        o.x = fmaf(ws[k], a[k].x, o.x);
        o.y = fmaf(ws[k], a[k].y, o.y);
        o.z = fmaf(ws[k], a[k].z, o.z);
        o.w = fmaf(ws[k], a[k].w, o.w);
      }
    }
  }
  trigger_dependents();  // last scratch read done

  const float inv = 1.f / total;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * inv, o.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z * inv, o.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&lo);
  packed.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out) = packed;
  if (p.lse != nullptr && lane == 0) p.lse[row] = mx + logf(total);
  PA_TS_LAST(p.ts, 2);
}

}  // namespace

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream, bool use_pdl) {
  const size_t smem = static_cast<size_t>(kWarps) * p.num_splits * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>((p.num_rows + kWarps - 1) / kWarps));
  return launch_kernel(reduce_kernel, grid, dim3(kThreads), smem, stream, use_pdl, p);
}

}  // namespace pa
