// Log-sum-exp reducer of the split-K decode attention.
//
// lmdeploy PR #4861 (Changes: Split-K paged attention): the reducer is launched
// with PDL and waits immediately before it reads the producer's scratch.  The
// combination is the standard one: M = max_s m_s, L = sum_s l_s e^(m_s - M),
// out = sum_s acc_s e^(m_s - M) / L, lse = M + ln L.
//
// One to eight warps per (request, query head) row; a lane owns 4 of the 128
// channels, so a split's accumulator row is one coalesced 512-byte read.  Split
// weights are kept in shared memory (one slot per split per warp).  Empty splits
// (m = -inf) get weight 0; their accumulator rows may be loaded but never contribute.
#include <math_constants.h>

#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;  // accumulator rows in flight per lane

// WPR warps share one (request, query head) row; warp `sub` combines splits
// sub*spw .. sub*spw + spw - 1.  Every warp loads its accumulator rows before it knows
// the split weights (the loads do not depend on them), so a row costs about one
// round trip to memory however many splits it has.
template <int WPR>
__global__ void __launch_bounds__(kThreads) reduce_kernel(const ReduceParams p) {
  extern __shared__ float smem[];  // [kWarps][S] weights, then [kWarps][32] float4 partials
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = warp % WPR;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kWarps / WPR) + warp / WPR;
  const int S = p.num_splits;
  const int spw = (S + WPR - 1) / WPR;
  const int s_begin = min(sub * spw, S), s_end = min(s_begin + spw, S);
  float* w = smem + warp * S;
  float4* part = reinterpret_cast<float4*>(smem + kWarps * S);
  const bool active = row < p.num_rows;

  PA_TS_FIRST(p.ts, 2, kTsEntry);
  grid_dependency_wait();  // the producer's partials are complete and visible
  PA_TS_FIRST(p.ts, 2, kTsReady);

  const int64_t r = active ? row : 0;
  const float4* acc = reinterpret_cast<const float4*>(p.acc + r * S * 128) + lane;
  float4 a[kBatch];
  const int first_n = min(kBatch, s_end - s_begin);
#pragma unroll
  for (int k = 0; k < kBatch; ++k) {
    a[k] = k < first_n ? acc[(s_begin + k) * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* m = p.m + r * S;
  const float* l = p.l + r * S;
  // the split maxima and sums of a lane's first (usually only) split slot are loaded
  // together, so the sums cost no second round trip after the maximum is known
  const float m0 = lane < S ? m[lane] : -CUDART_INF_F;
  const float l0 = lane < S ? l[lane] : 0.f;
  float mx = m0;
  for (int s = lane + 32; s < S; s += 32) mx = fmaxf(mx, m[s]);
  mx = warp_max(mx);
  float total = 0.f;
  if (mx != -CUDART_INF_F) {
    for (int s = lane; s < S; s += 32) {
      const float ms = s == lane ? m0 : m[s];
      const float ls = s == lane ? l0 : l[s];
      const float ws = ms == -CUDART_INF_F ? 0.f : expf(ms - mx);
      w[s] = ws;
      if (ws != 0.f) total += ws * ls;
    }
    total = warp_sum(total);
  }
  __syncwarp();

  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mx != -CUDART_INF_F) {
    for (int s0 = s_begin; s0 < s_end; s0 += kBatch) {
      if (s0 != s_begin) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int s = min(s0 + k, S - 1);
          a[k] = acc[s * 32];
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float ws = s0 + k < s_end ? w[s0 + k] : 0.f;  // empty split: weight 0, unused
        if (ws != 0.f) {
          o.x = fmaf(ws, a[k].x, o.x);
          o.y = fmaf(ws, a[k].y, o.y);
          o.z = fmaf(ws, a[k].z, o.z);
          o.w = fmaf(ws, a[k].w, o.w);
        }
      }
    }
  }
  trigger_dependents();  // last scratch read done

  if constexpr (WPR > 1) {
    part[warp * 32 + lane] = o;
    __syncthreads();
    if (sub != 0) {
      PA_TS_LAST(p.ts, 2);
      return;
    }
#pragma unroll
    for (int k = 1; k < WPR; ++k) {
      const float4 v = part[(warp + k) * 32 + lane];
      o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
    }
  }
  if (!active) {
    PA_TS_LAST(p.ts, 2);
    return;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + row * 128 + lane * 4;
  if (mx == -CUDART_INF_F) {  // no tokens at all
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    if (p.lse != nullptr && lane == 0) p.lse[row] = -CUDART_INF_F;
    PA_TS_LAST(p.ts, 2);
    return;
  }
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

template <int WPR>
cudaError_t launch_reduce_wpr(const ReduceParams& p, cudaStream_t stream, bool use_pdl) {
  const size_t smem = static_cast<size_t>(kWarps) * p.num_splits * sizeof(float) +
                      static_cast<size_t>(kWarps) * 32 * sizeof(float4);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(reduce_kernel<WPR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  constexpr int kRowsPerCta = kWarps / WPR;
  const dim3 grid(static_cast<unsigned>((p.num_rows + kRowsPerCta - 1) / kRowsPerCta));
  return launch_kernel(reduce_kernel<WPR>, grid, dim3(kThreads), smem, stream, use_pdl, p);
}

}  // namespace

// Warps per row: enough that a warp combines at most 4 splits (up to 8 warps), so a
// batch-1 step with many splits pays one memory round trip, not S / 8 of them.
cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream, bool use_pdl) {
  const int S = p.num_splits;
  if (S > 16) return launch_reduce_wpr<8>(p, stream, use_pdl);
  if (S > 8) return launch_reduce_wpr<4>(p, stream, use_pdl);
  if (S > 4) return launch_reduce_wpr<2>(p, stream, use_pdl);
  return launch_reduce_wpr<1>(p, stream, use_pdl);
}

}  // namespace pa
