// Split-K paged-attention producer for decode (one query token per request).
//
// The producer/reducer split and the PDL placement follow lmdeploy PR #4861
// "perf(cuda): use PDL for paged attention and V4 prefill" (Changes: Split-K paged
// attention): the producer writes per-split partials (running max, sum of
// exponentials, unnormalised accumulator) to scratch and signals its dependents
// before its final scratch stores.  The attention arithmetic is the textbook
// definition, softmax(q K^T * sm_scale) V with grouped KV heads.
//
// GB300 mapping
//   * One CTA per (split, kv head, request), 128 threads.  All G = Hq/Hkv query heads
//     of a kv head share one pass over its K/V rows, so every KV byte is read once.
//   * KV pages are [num_pages, Hkv, page_size, 128]: the rows of one (page, kv head)
//     are contiguous, so a 64-token chunk is one (or, for pages < 64 tokens, a few)
//     1-D bulk TMA copies (cp.async.bulk) per tensor, landing in a STAGES-deep
//     shared-memory ring completed on mbarriers.  KV is loaded with an L2
//     evict-first policy: it is streamed exactly once per step.
//   * QK^T: a lane owns E consecutive channels of the query rows (held in registers,
//     pre-scaled by sm_scale*log2 e) and of each K row; LPR = 128/E lanes cover a
//     row.  Partial dot products of TB tokens x G heads are combined by a butterfly
//     reduce-scatter across the LPR lanes (one value per lane at the end, V-1
//     shuffles for V values).
//   * Online softmax in base 2 per chunk: warp w owns heads w, w+4; it takes the
//     chunk maximum, rescales its running sum and publishes exp2 weights and the
//     rescale factor through shared memory.
//   * PV: a lane accumulates E channels x G heads for the tokens of its row group;
//     the row groups are summed once at the end of the split.
//   * int8 KV: codes are widened exactly to fp32; the per-token K scale multiplies
//     the finished dot product and the V scale folds into the softmax weight, so
//     both scales cost one multiply per (token, head).
//   * CUDA cores do the arithmetic.  For bf16 with G = 4 a step needs about four
//     FMAs per KV element, well inside the FP32 rate at full HBM bandwidth.
#pragma once

#include <math_constants.h>

#include <atomic>
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <bool kQuant, int G, int P, int STAGES>
struct SplitKConfig {
  static constexpr int D = 128;
  static constexpr int CHUNK = 64;
  static constexpr int THREADS = 128;
  static constexpr int E = (G <= 4) ? 8 : 4;        // channels per lane
  static constexpr int LPR = D / E;                 // lanes per K/V row
  static constexpr int RG = THREADS / LPR;          // row groups per CTA
  static constexpr int TPR = CHUNK / RG;            // tokens per row group per chunk
  static constexpr int TB_RAW = LPR / G;
  static constexpr int TB = TB_RAW < TPR ? TB_RAW : TPR;  // tokens per butterfly batch
  static constexpr int NB = TPR / TB;               // batches per chunk
  static constexpr int V = TB * G;                  // values per butterfly
  static constexpr int ESZ = kQuant ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int KV_BYTES = CHUNK * ROW_BYTES;
  static constexpr int SCALE_BYTES = kQuant ? CHUNK * 4 : 0;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES + 2 * SCALE_BYTES;
  static constexpr int PAGES_PER_CHUNK = P >= CHUNK ? 1 : CHUNK / P;
  static constexpr int MAX_SPLIT_PAGES = 256;
  static constexpr int OFF_SCORES = STAGES * STAGE_BYTES;          // [G][CHUNK] f32
  static constexpr int OFF_P = OFF_SCORES + G * CHUNK * 4;         // [CHUNK][G] f32
  static constexpr int OFF_ALPHA = OFF_P + CHUNK * G * 4;          // [G] f32 (32 slots)
  static constexpr int OFF_PAGES = OFF_ALPHA + 32 * 4;             // [MAX_SPLIT_PAGES] i32
  static constexpr int OFF_BARS = OFF_PAGES + MAX_SPLIT_PAGES * 4; // [STAGES] u64
  static constexpr int SMEM = OFF_BARS + STAGES * 8;
  static constexpr int RED_BYTES = RG * G * D * 4;
  static constexpr int HEADS_PER_WARP = (G + 3) / 4;
  static_assert(V <= LPR, "butterfly needs at most one value per lane");
  static_assert(TPR % TB == 0, "row-group tokens must split into batches");
  static_assert(RED_BYTES <= STAGES * STAGE_BYTES, "reduction buffer reuses the ring");
  static_assert((LPR & (LPR - 1)) == 0 && (V & (V - 1)) == 0, "powers of two");
};

// Butterfly reduce-scatter of CNT values over the lanes selected by masks M, M/2..1.
// Afterwards v[0] holds the sum over those lanes of value index
// (r >> (log2(2M) - log2(CNT))), where r is the lane's index within its row.
template <int CNT, int M>
struct Butterfly {
  __device__ __forceinline__ static void run(float* v, int r) {
    if constexpr (M >= 1) {
      if constexpr (CNT > 1) {
        constexpr int H = CNT / 2;
        const bool upper = (r & M) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
        }
        Butterfly<H, M / 2>::run(v, r);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
        Butterfly<1, M / 2>::run(v, r);
      }
    }
  }
};

template <int N>
__device__ __forceinline__ constexpr int ilog2() {
  return N <= 1 ? 0 : 1 + ilog2<N / 2>();
}

// Load E channels of a K/V row at byte offset `off` of a stage and widen to fp32.
template <bool kQuant, int E>
__device__ __forceinline__ void load_row(const unsigned char* base, float (&f)[E]) {
  if constexpr (!kQuant && E == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(base);
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  } else if constexpr (!kQuant && E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(base);
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  } else if constexpr (kQuant && E == 8) {
    const uint2 w = *reinterpret_cast<const uint2*>(base);
    s8x4_to_float(w.x, f[0], f[1], f[2], f[3]);
    s8x4_to_float(w.y, f[4], f[5], f[6], f[7]);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(base);
    s8x4_to_float(w, f[0], f[1], f[2], f[3]);
  }
}

template <bool kQuant, int G, int P, int STAGES, int MINB>
__global__ void __launch_bounds__(128, MINB) splitk_kernel(const SplitKParams prm) {
  using C = SplitKConfig<kQuant, G, P, STAGES>;
  constexpr int D = C::D, CHUNK = C::CHUNK, E = C::E, LPR = C::LPR, TPR = C::TPR;
  constexpr int TB = C::TB, NB = C::NB, V = C::V;
  extern __shared__ __align__(128) unsigned char smem[];

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rg = tid / LPR, r = tid % LPR;
  const int num_splits = prm.num_splits;
  PA_TS_FIRST(prm.ts, 1, kTsEntry);

  // ---- prologue that does not depend on the metadata stage: the query rows -------
  float qf[G][E];
  {
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(prm.q) +
                                (static_cast<int64_t>(b) * prm.num_q_heads + kvh * G) * D + r * E;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      load_row<false, E>(reinterpret_cast<const unsigned char*>(qrow + h * D), qf[h]);
#pragma unroll
      for (int e = 0; e < E; ++e) qf[h][e] *= prm.q_scale;
    }
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }

  // ---- everything below reads what the metadata stage wrote ----------------------
  grid_dependency_wait();
  PA_TS_FIRST(prm.ts, 1, kTsReady);

  int n = prm.cache_seqlens[b];
  const int cap = prm.max_seq_pages * P;
  if (n < 0 || n > cap) {
    if (tid == 0 && split == 0 && kvh == 0) record_error(prm.err, kErrSeqLenOutOfRange);
    n = n < 0 ? 0 : cap;
  }
  const int n_pages = (n + P - 1) / P;
  const int p_begin = split * prm.pages_per_split;
  const int p_end = min(p_begin + prm.pages_per_split, n_pages);
  const int tok_begin = p_begin * P;
  const int n_tok = min(p_end * P, n) - tok_begin;
  const int64_t slot0 =
      (static_cast<int64_t>(b) * prm.num_q_heads + kvh * G) * num_splits + split;

  if (n_tok <= 0) {
    trigger_dependents();
    if (tid < G) {
      prm.m_out[slot0 + static_cast<int64_t>(tid) * num_splits] = -CUDART_INF_F;
      prm.l_out[slot0 + static_cast<int64_t>(tid) * num_splits] = 0.f;
    }
    PA_TS_LAST(prm.ts, 1);
    return;
  }

  // Page indices of this split, bounds-checked once, cached in shared memory.
  const int n_split_pages = p_end - p_begin;
  int32_t* pages_s = reinterpret_cast<int32_t*>(smem + C::OFF_PAGES);
  const int32_t* pt_row = prm.page_table + static_cast<int64_t>(b) * prm.page_table_stride + p_begin;
  for (int i = tid; i < min(n_split_pages, C::MAX_SPLIT_PAGES); i += C::THREADS) {
    int32_t pg = pt_row[i];
    if (pg < 0 || pg >= prm.num_pages) {
      record_error(prm.err, kErrPageOutOfRange);
      pg = 0;
    }
    pages_s[i] = pg;
  }
  __syncthreads();

  const int n_chunks = (n_tok + CHUNK - 1) / CHUNK;
  const unsigned char* kbase = static_cast<const unsigned char*>(prm.k_cache);
  const unsigned char* vbase = static_cast<const unsigned char*>(prm.v_cache);
  const int64_t hkv = prm.num_kv_heads;

  auto page_at = [&](int i) -> int64_t {
    if (i < C::MAX_SPLIT_PAGES) return pages_s[i];
    int32_t pg = pt_row[i];
    if (pg < 0 || pg >= prm.num_pages) {
      record_error(prm.err, kErrPageOutOfRange);
      pg = 0;
    }
    return pg;
  };

  // Issue the copies of chunk c into its stage (thread 0 only).
  uint64_t policy = 0;
  if (tid == 0) policy = l2_evict_first_policy();
  auto issue = [&](int c) {
    const int stage = c % STAGES;
    unsigned char* st = smem + stage * C::STAGE_BYTES;
    const int ctok = c * CHUNK;  // token offset inside the split
    if constexpr (P >= CHUNK) {
      const int64_t pg = page_at(ctok / P);
      const int64_t row = (pg * hkv + kvh) * P + (ctok % P);
      mbar_arrive_expect_tx(&bars[stage], C::STAGE_BYTES);
      bulk_copy_g2s(st, kbase + row * C::ROW_BYTES, C::KV_BYTES, &bars[stage], policy);
      bulk_copy_g2s(st + C::KV_BYTES, vbase + row * C::ROW_BYTES, C::KV_BYTES, &bars[stage],
                    policy);
      if constexpr (kQuant) {
        bulk_copy_g2s(st + 2 * C::KV_BYTES, prm.k_scale + row, C::SCALE_BYTES, &bars[stage],
                      policy);
        bulk_copy_g2s(st + 2 * C::KV_BYTES + C::SCALE_BYTES, prm.v_scale + row,
                      C::SCALE_BYTES, &bars[stage], policy);
      }
    } else {
      const int first = ctok / P;
      const int np = min(C::PAGES_PER_CHUNK, n_split_pages - first);
      constexpr int kPageKV = P * C::ROW_BYTES;
      constexpr int kPageScale = kQuant ? P * 4 : 0;
      mbar_arrive_expect_tx(&bars[stage], np * (2 * kPageKV + 2 * kPageScale));
      for (int k = 0; k < np; ++k) {
        const int64_t pg = page_at(first + k);
        const int64_t row = (pg * hkv + kvh) * P;
        bulk_copy_g2s(st + k * kPageKV, kbase + row * C::ROW_BYTES, kPageKV, &bars[stage],
                      policy);
        bulk_copy_g2s(st + C::KV_BYTES + k * kPageKV, vbase + row * C::ROW_BYTES, kPageKV,
                      &bars[stage], policy);
        if constexpr (kQuant) {
          bulk_copy_g2s(st + 2 * C::KV_BYTES + k * kPageScale, prm.k_scale + row, kPageScale,
                        &bars[stage], policy);
          bulk_copy_g2s(st + 2 * C::KV_BYTES + C::SCALE_BYTES + k * kPageScale,
                        prm.v_scale + row, kPageScale, &bars[stage], policy);
        }
      }
    }
  };

  int issued = 0;
  if (tid == 0) {
    for (; issued < min(STAGES, n_chunks); ++issued) issue(issued);
  }

  float* scores = reinterpret_cast<float*>(smem + C::OFF_SCORES);  // [G][CHUNK]
  float* p_s = reinterpret_cast<float*>(smem + C::OFF_P);          // [CHUNK][G]
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);

  float acc[G][E];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  float m_run[C::HEADS_PER_WARP], l_run[C::HEADS_PER_WARP];
#pragma unroll
  for (int j = 0; j < C::HEADS_PER_WARP; ++j) {
    m_run[j] = -CUDART_INF_F;
    l_run[j] = 0.f;
  }

  bool failed = false;
  int consumed = 0;
  for (int c = 0; c < n_chunks; ++c) {
    const int stage = c % STAGES;
    const uint32_t parity = static_cast<uint32_t>(c / STAGES) & 1u;
    const int valid = min(CHUNK, n_tok - c * CHUNK);
    const bool ready = mbar_wait_bounded(&bars[stage], parity);
    const unsigned char* kst = smem + stage * C::STAGE_BYTES;
    const unsigned char* vst = kst + C::KV_BYTES;

    // ---- scores of this chunk: s[h][t] = log2(e) * sm_scale * q_h . k_t ------------
#pragma unroll
    for (int bt = 0; bt < NB; ++bt) {
      float part[V];
#pragma unroll
      for (int j = 0; j < TB; ++j) {
        const int t = rg * TPR + bt * TB + j;
        float kf[E];
        load_row<kQuant, E>(kst + t * C::ROW_BYTES + r * E * C::ESZ, kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float d = qf[h][0] * kf[0];
#pragma unroll
          for (int e = 1; e < E; ++e) d = fmaf(qf[h][e], kf[e], d);
          part[j * G + h] = d;
        }
      }
      Butterfly<V, LPR / 2>::run(part, r);
      constexpr int kShift = ilog2<LPR>() - ilog2<V>();
      if ((r & ((1 << kShift) - 1)) == 0) {
        const int idx = r >> kShift;
        const int t = rg * TPR + bt * TB + idx / G;
        const int h = idx % G;
        float s = part[0];
        if constexpr (kQuant) s *= reinterpret_cast<const float*>(kst + 2 * C::KV_BYTES)[t];
        scores[h * CHUNK + t] = t < valid ? s : -CUDART_INF_F;
      }
    }

    // barrier A: scores complete; every thread is done with chunk c-1's stage.
    if (__syncthreads_or(!ready)) {
      failed = true;
      consumed = c;
      break;
    }
    if (tid == 0 && issued < n_chunks && issued < c + STAGES) {
      issue(issued);
      ++issued;
    }

    // ---- online softmax per head (base 2) -------------------------------------------
#pragma unroll
    for (int j = 0; j < C::HEADS_PER_WARP; ++j) {
      const int h = warp + 4 * j;
      if (h < G) {
        const float s0 = scores[h * CHUNK + lane];
        const float s1 = scores[h * CHUNK + lane + 32];
        const float m_new = fmaxf(m_run[j], warp_max(fmaxf(s0, s1)));
        float alpha = 1.f, p0 = 0.f, p1 = 0.f;
        if (m_new != -CUDART_INF_F) {
          alpha = exp2f(m_run[j] - m_new);
          p0 = exp2f(s0 - m_new);
          p1 = exp2f(s1 - m_new);
        }
        l_run[j] = l_run[j] * alpha + warp_sum(p0 + p1);
        m_run[j] = m_new;
        if constexpr (kQuant) {
          const float* vsc = reinterpret_cast<const float*>(kst + 2 * C::KV_BYTES + C::SCALE_BYTES);
          p0 *= vsc[lane];
          p1 *= vsc[lane + 32];
        }
        p_s[lane * G + h] = p0;
        p_s[(lane + 32) * G + h] = p1;
        if (lane == 0) alpha_s[h] = alpha;
      }
    }
    __syncthreads();  // barrier B: weights and rescale factors published

    // ---- PV -----------------------------------------------------------------------
    {
      float a[G];
      bool rescale = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        a[h] = alpha_s[h];
        rescale |= a[h] != 1.f;
      }
      if (rescale) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[h][e] *= a[h];
      }
      const int t0 = rg * TPR;
      const int my_n = max(0, min(TPR, valid - t0));
#pragma unroll 2
      for (int i = 0; i < my_n; ++i) {
        const int t = t0 + i;
        float vf[E];
        load_row<kQuant, E>(vst + t * C::ROW_BYTES + r * E * C::ESZ, vf);
        float pw[G];
        if constexpr (G == 8) {
          const float4 x = reinterpret_cast<const float4*>(p_s + t * G)[0];
          const float4 y = reinterpret_cast<const float4*>(p_s + t * G)[1];
          pw[0] = x.x; pw[1] = x.y; pw[2] = x.z; pw[3] = x.w;
          pw[4] = y.x; pw[5] = y.y; pw[6] = y.z; pw[7] = y.w;
        } else if constexpr (G == 4) {
          const float4 x = *reinterpret_cast<const float4*>(p_s + t * G);
          pw[0] = x.x; pw[1] = x.y; pw[2] = x.z; pw[3] = x.w;
        } else if constexpr (G == 2) {
          const float2 x = *reinterpret_cast<const float2*>(p_s + t * G);
          pw[0] = x.x; pw[1] = x.y;
        } else {
          pw[0] = p_s[t];
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[h][e] = fmaf(pw[h], vf[e], acc[h][e]);
      }
    }
  }

  if (failed) {
    // Drain the copies still in flight so no TMA write lands after the CTA exits.
    if (tid == 0) {
      record_error(prm.err, kErrWaitTimeout);
      for (int c = consumed; c < issued; ++c) {
        mbar_wait_bounded(&bars[c % STAGES], static_cast<uint32_t>(c / STAGES) & 1u);
      }
    }
    __syncthreads();
    return;
  }

  // All KV reads of this CTA are done: let the reducer launch (its own wait still
  // blocks until this grid has completed), then store the partials.
  trigger_dependents();

  __syncthreads();  // every thread is done with the ring; reuse it for the reduction
  float* red = reinterpret_cast<float*>(smem);  // [RG][G][D]
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float* dst = red + (rg * G + h) * D + r * E;
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      *reinterpret_cast<float4*>(dst + e) = make_float4(acc[h][e], acc[h][e + 1], acc[h][e + 2], acc[h][e + 3]);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D / 4; idx += C::THREADS) {
    const int h = (idx * 4) / D, d = (idx * 4) % D;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < C::RG; ++g) {
      const float4 x = *reinterpret_cast<const float4*>(red + (g * G + h) * D + d);
      sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
    }
    *reinterpret_cast<float4*>(prm.acc_out + (slot0 + static_cast<int64_t>(h) * num_splits) * D + d) = sum;
  }
#pragma unroll
  for (int j = 0; j < C::HEADS_PER_WARP; ++j) {
    const int h = warp + 4 * j;
    if (h < G && lane == 0) {
      const int64_t slot = slot0 + static_cast<int64_t>(h) * num_splits;
      prm.m_out[slot] = m_run[j] * 0.69314718055994530942f;  // back to natural-log units
      prm.l_out[slot] = l_run[j];
    }
  }
  PA_TS_LAST(prm.ts, 1);
}

// Host launch of one instantiation.  The dynamic shared-memory limit is raised once
// per device (the attribute is per device context).
template <bool kQuant, int G, int P, int STAGES, int MINB>
cudaError_t launch_splitk_one(const SplitKParams& p, dim3 grid, cudaStream_t stream,
                              bool use_pdl) {
  using C = SplitKConfig<kQuant, G, P, STAGES>;
  void (*kernel)(const SplitKParams) = splitk_kernel<kQuant, G, P, STAGES, MINB>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return launch_kernel(kernel, grid, dim3(C::THREADS), static_cast<size_t>(C::SMEM), stream,
                       use_pdl, p);
}

// Host launcher for one KV type: picks the (G, page_size) instantiation.
template <bool kQuant, int STAGES, int MINB>
cudaError_t launch_splitk_impl(const SplitKParams& p, int bs, int group, int page_size,
                               cudaStream_t stream, bool use_pdl) {
  const dim3 grid(static_cast<unsigned>(p.num_splits), static_cast<unsigned>(p.num_kv_heads),
                  static_cast<unsigned>(bs));
#define PA_SPLITK_CASE(GG, PP)                                                            \
  if (group == GG && page_size == PP) {                                                   \
    return launch_splitk_one<kQuant, GG, PP, STAGES, MINB>(p, grid, stream, use_pdl);     \
  }
#define PA_SPLITK_PAGES(GG) \
  PA_SPLITK_CASE(GG, 16) PA_SPLITK_CASE(GG, 32) PA_SPLITK_CASE(GG, 64) PA_SPLITK_CASE(GG, 128)
  PA_SPLITK_PAGES(1)
  PA_SPLITK_PAGES(2)
  PA_SPLITK_PAGES(4)
  PA_SPLITK_PAGES(8)
#undef PA_SPLITK_PAGES
#undef PA_SPLITK_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
