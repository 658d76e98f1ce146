// Split-K paged-attention producer on the tensor cores (warp-level mma.sync).
//
// Same contract as the CUDA-core producer in pa_splitk.cuh (lmdeploy PR #4861,
// "perf(cuda): use PDL for paged attention and V4 prefill", Changes: Split-K paged
// attention): per split it writes the running max, the sum of exponentials and the
// unnormalised accumulator, and signals its dependents before those final stores.
//
// Why tensor cores here: the G = Hq/Hkv query heads of a kv head turn QK^T and PV into
// small dense contractions (G x 128 by 128 x tokens, and G x tokens by tokens x 128).
// On CUDA cores every KV element costs G FMAs plus a widening conversion; at full HBM
// rate that saturates the issue slots (G = 8 int8) or leaves the kernel latency bound
// (G = 4 bf16).  One m16n8k16 MMA does 2048 multiply-adds per warp instruction.
//
// GB300 mapping
//   * CTA = 4 consumer warps (4 * NG for small grids) + 1 producer warp.  The producer
//     warp's lane 0 streams 64-token chunks with 4-D TMA tiled copies
//     (cp.async.bulk.tensor) of the [num_pages, Hkv, page_size, 128] pools into a
//     STAGES-deep ring; full/empty
//     mbarriers hand stages back and forth, so there is no CTA-wide barrier per chunk.
//     128-byte swizzle makes every ldmatrix / 16-byte shared load conflict free.
//     Grids of at most one block per SM take a deeper ring at one CTA per SM.
//   * Consumer warps come in groups of four; warp w of a group owns tokens [16w, 16w+16)
//     of each of its group's chunks and keeps its own online-softmax state for its
//     tokens; the warps' states are merged once at the end of the split (the same
//     log-sum-exp combination the reducer applies across splits).  One group consumes
//     every chunk; grids of at most one block per SM use several groups, each taking
//     every NG-th chunk, so a short split's chunks are worked on at once.  The weights
//     of a column are relative to a reference maximum that moves only when a score
//     passes it by more than 2^kMaxSlack (log2 units), so most slices need one warp
//     vote instead of a shuffle reduction and a rescale.
//   * Persistent form (kPersist; large int8 grids): one CTA per resident slot claims
//     (request, kv head, split) items from a largest-first work list, and the ring keeps
//     cycling across items.
//   * Transposed orientation: S^T = K Q^T with M = 16 tokens, N = 8 columns (a column is
//     a query head, or a (query, head) pair with several queries per request), K = 16
//     channels; then O^T += V^T P^T with M = 16 channels, K = 16 tokens, and P^T taken
//     from the S^T fragments with movmatrix.trans.  Q^T fragments stay in registers for
//     the whole split.
//   * bf16 KV: K fragments come from ldmatrix, V^T fragments from ldmatrix.trans.
//   * int8 KV: codes widened exactly to fp16 in registers (a byte placed in the
//     mantissa of 1024: one XOR per 4 bytes, one byte permute per fp16 pair) and fed to
//     fp16 MMAs.  K: 16-byte shared loads, with the contraction order over channels
//     permuted so that each lane reads 16 contiguous bytes (QK^T does not depend on
//     that order).  V: ldmatrix.trans hands each lane two tokens of one channel, the
//     pair an A register of V^T holds.  Both K and V codes come out biased by +1152: the
//     resulting 1152 * sum(q) per column is taken out of the fp32 score (the odd QK^T
//     accumulator starts at its negative), and the V codes get the bias subtracted in
//     fp16 (exact) before the PV product.  Q is scaled per column by a power of two into
//     fp16's range (bf16 values stay exact; the factor returns in the fp32 score
//     scale).  The K scale multiplies the fp32 score; the V scale folds into the fp16
//     softmax weight, prescaled per warp by a power of two so that no significant
//     weight is an fp16 subnormal.
//   * Sliding window (kWindow): the splits cover each request's window, positions below
//     a column's window start are masked, and pages with a -1 table entry are neither
//     loaded nor attended.
//   * Scores are scaled in fp32 (sm_scale * log2 e), never by rounding Q.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <atomic>
#include <climits>
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace mma {

constexpr int kChunk = 64;
// Consumer warps come in groups of four; a group shares the 64 tokens of a chunk (16
// each).  One group (NG = 1) consumes every chunk; with NG groups, group g consumes the
// chunks c with c % NG == g, so NG chunks are worked on at once (small grids).
constexpr int kGroupWarps = 4;
template <int NG>
constexpr int threads_of() { return (NG * kGroupWarps + 1) * 32; }
constexpr int kMaxSplitPages = 256;
// The persistent form (one CTA per resident slot walking a work list) takes batches of
// at most this many requests.
constexpr int kMaxPersistRequests = 128;
// Work-claim counters of the persistent form: [claimed items, CTAs done] per slot.  A
// launch takes the next slot (host side, round robin); its last CTA to finish sets the
// slot back to zero, so the slot is ready for its next launch.  Launches of one stream
// never overlap their claims (each waits for the previous producer to complete), so
// only more than kWorkSlots producers in flight on different streams could collide.
constexpr int kWorkSlots = 64;
static __device__ unsigned int g_work_claims[kWorkSlots][2];
static std::atomic<unsigned int> g_next_work_slot{0};
// Online-softmax slack (log2 units): the reference maximum of a column moves only when a
// score exceeds it by more than this, so softmax weights stay below 2^8.
#ifndef PA_MAX_SLACK
#define PA_MAX_SLACK 8
#endif
constexpr float kMaxSlack = PA_MAX_SLACK;
// Full 16-token slices of a one-query, full-context split skip the per-score masks.
#ifndef PA_MASK_FAST
#define PA_MASK_FAST 1
#endif
// 1: the PV weights enter as two MMA operands, the weight rounded to the operand type
// and its rounding residual rounded again (bf16: ~2^-16 relative, fp16: ~2^-22), which
// keeps the output error well inside the output's own rounding; 0: one operand.
#ifndef PA_P_SPLIT
#define PA_P_SPLIT 1
#endif

template <bool kQuant, int STAGES, int NW>
struct Layout {
  static constexpr int KV_BYTES = kQuant ? kChunk * 128 : kChunk * 256;  // per tensor per chunk
  static constexpr int SCALE_BYTES = kQuant ? kChunk * 4 : 0;
  static constexpr int STAGE_RAW = 2 * KV_BYTES + 2 * SCALE_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;   // 1024-aligned tiles
  static constexpr int OFF_PAGES = STAGES * STAGE_BYTES;
  static constexpr int OFF_FULL = OFF_PAGES + kMaxSplitPages * 4;
  static constexpr int OFF_EMPTY = OFF_FULL + STAGES * 8;
  static constexpr int OFF_ML = OFF_EMPTY + STAGES * 8;      // [NW warps][16 columns][3]
  static constexpr int OFF_MISC = OFF_ML + NW * 16 * 3 * 4;  // abort, issued, done
  static constexpr int OFF_SKIP = OFF_MISC + 16;  // per stage: mask of its skipped pages
  // persistent form: per-request length, full and partial split counts, the requests
  // ranked by partial-split size, prefix of full splits (+1), two counts
  // persistent form: per stage, the work-list position of the item whose first chunk
  // the stage holds (-1: no more work)
  static constexpr int OFF_DESC = OFF_SKIP + (STAGES * 4 + 15) / 16 * 16;
  static constexpr int OFF_SCHED = OFF_DESC + (STAGES * 4 + 15) / 16 * 16;
  static constexpr int SCHED_INTS = 5 * kMaxPersistRequests + 3;
  static constexpr int SMEM = OFF_SCHED + (SCHED_INTS * 4 + 15) / 16 * 16 + 1024;  // + align slack
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool kF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Transpose an 8x8 matrix of 16-bit values held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <int NW>
__device__ __forceinline__ void consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// Two bf16/fp16 values packed low-first.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two int8 codes (already XORed with 0x80, i.e. code + 128 as unsigned bytes) picked by
// `selector` -> fp16x2 holding code + 1152 each: the byte becomes the low mantissa byte
// of 1024 (0x64xx), exact.
__device__ __forceinline__ uint32_t biased_bytes_to_f16x2(uint32_t x, uint32_t selector) {
  return __byte_perm(x, 0x64646464u, selector);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-row tile written by
// TMA with 128-byte swizzle (the tile starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32: relative error ~2^-22,
// results below 2^-126 flush to 0, 2^-inf = 0): the softmax weights of the inner loop.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Power of two 2^e with e clamped to [-100, 100] (exact; built from the exponent bits).
__device__ __forceinline__ float pow2_clamped(int e) {
  e = max(-100, min(100, e));
  return __int_as_float((e + 127) << 23);
}

// Exponent E of a finite x > 0 (x = m * 2^E, 1 <= m < 2); subnormals read as -127.
__device__ __forceinline__ int float_exponent(float x) {
  return ((__float_as_int(x) >> 23) & 0xff) - 127;
}

// B operand of S^T = K Q^T.  Column n of the N dimension is query i = n / G of the
// request (row q_begin + i) and query head kvh * G + n % G; columns n >= q_len * G are
// zero.  b0 = Q[col][k 2tig, 2tig+1], b1 = Q[col][k 2tig+8, +9] of k-step j, for
// column n = 8 * nt + gid.  qf[nt][e]: the fp32 factor that turns column 8nt + 2tig + e
// of the MMA result into a base-2 score (q_scale, times the column's Q prescale below).
// int8 path (kF16): fp16 Q in the permuted contraction order (k-step j, lane tig ->
// channels 32*tig + 4*j + {0..3}).  Each column is first scaled by a power of two that
// puts its largest |q| in [2^14, 2^15) (exact for bf16 values, and no |q| can overflow
// fp16's 65504); qf undoes it.  kbias: the K codes enter the MMA biased by +1152 (the
// widening skips the subtract), so each score carries 1152 * sum_d q[col][d];
// kbias[nt][e] is that offset from the same fp16 Q values.  The whole warp calls this.
template <bool kF16, int kNT>
__device__ __forceinline__ void load_q_fragments(const SplitKParams& prm, int q_begin, int q_len,
                                                 int kvh, int G, int gid, int tig,
                                                 uint32_t (&qb)[kNT][8][2],
                                                 float (&kbias)[kNT][2], float (&qf)[kNT][2]) {
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int col = 8 * nt + gid;
    const int qi = col / G;
    const int head = kvh * G + (col - qi * G);
    const bool live = col < q_len * G;
    const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(prm.q) +
                              (static_cast<int64_t>(q_begin + qi) * prm.num_q_heads + head) * 128;
    if constexpr (kF16) {
      // a lane's 32 channels are 64 contiguous bytes of the row (rows are 256 bytes and
      // Q is 16-byte aligned): four 16-byte loads
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 r = live ? reinterpret_cast<const uint4*>(qr + 32 * tig)[k]
                             : make_uint4(0u, 0u, 0u, 0u);
        w[4 * k] = r.x;
        w[4 * k + 1] = r.y;
        w[4 * k + 2] = r.z;
        w[4 * k + 3] = r.w;
      }
      float v[8][4];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t pair = w[2 * j + (u >> 1)];  // channels 4j + u, low half first
          v[j][u] = __uint_as_float((u & 1) ? (pair & 0xffff0000u) : (pair << 16));
          amax = fmaxf(amax, fabsf(v[j][u]));
        }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));  // over the 128 channels
      const int e = amax > 0.f ? 14 - float_exponent(amax) : 0;
      const float up = pow2_clamped(e);
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qb[nt][j][0] = pack_f16(v[j][0] * up, v[j][1] * up);
        qb[nt][j][1] = pack_f16(v[j][2] * up, v[j][3] * up);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qb[nt][j][0]));
        const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&qb[nt][j][1]));
        part += (a.x + a.y) + (c.x + c.y);
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);  // sum over the column's 128 channels
      const float down = prm.q_scale * pow2_clamped(-e);
#pragma unroll
      for (int ee = 0; ee < 2; ++ee) {
        kbias[nt][ee] = 1152.f * __shfl_sync(0xffffffffu, part, (2 * tig + ee) * 4);
        qf[nt][ee] = __shfl_sync(0xffffffffu, down, (2 * tig + ee) * 4);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t lo = 0, hi = 0;
        if (live) {
          const int d = 16 * j + 2 * tig;
          lo = *reinterpret_cast<const uint32_t*>(qr + d);
          hi = *reinterpret_cast<const uint32_t*>(qr + d + 8);
        }
        qb[nt][j][0] = lo;
        qb[nt][j][1] = hi;
      }
      kbias[nt][0] = kbias[nt][1] = 0.f;
      qf[nt][0] = qf[nt][1] = prm.q_scale;
    }
  }
}

// Scratch slot of column `col` (query col / G, head col % G of kv head kvh) for `split`.
__device__ __forceinline__ int64_t column_slot(int q_begin, int col, int G, int kvh,
                                               int num_q_heads, int S, int split) {
  const int qi = col / G;
  return ((static_cast<int64_t>(q_begin) + qi) * num_q_heads + kvh * G + (col - qi * G)) * S +
         split;
}

// kWindow: the sliding-window variant (prm.window > 0); without it every window test
// folds away at compile time.
// kPersist: the persistent form.  The grid is one CTA per resident slot; each CTA walks
// a list of (request, kv head, split) items, built in shared memory from the request
// lengths: the splits with a full page range first (all the same size), then the
// partial last splits of each request, largest first; a CTA claims the next item from
// an atomic counter whenever its TMA warp is free to issue one, so the slots finish
// together however the lengths are spread.  The ring keeps cycling across items, so
// the TMA warp copies the next item's first chunks while the consumers finish the
// current one (a fresh block would wait ~2 us for its first data).  One consumer group,
// one query per request, at most kMaxPersistRequests requests.
template <bool kQuant, int P, int STAGES, int MINB, int kNT, bool kWindow, int NG,
          bool kPersist>
__global__ void __launch_bounds__(threads_of<NG>(), MINB)
    splitk_mma_kernel(const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const SplitKParams prm) {
  static_assert(STAGES % NG == 0, "every group owns whole stages");
  static_assert(!kPersist || NG == 1, "the persistent form has one consumer group");
  constexpr int kConsumerWarps = NG * kGroupWarps;
  constexpr int kThreads = threads_of<NG>();
  using L = Layout<kQuant, STAGES, kConsumerWarps>;
  // output merge buffer: [consumer warps][8 * kNT columns][kRedStride] fp32 (128
  // channels; the 4-float pad puts the columns a warp stores at once in different
  // banks); the persistent form merges in the stage of the item's last chunk (held
  // until then)
  constexpr int kRedStride = 132;
  constexpr int kRedBytes = kConsumerWarps * 8 * kNT * kRedStride * 4;
  static_assert(kRedBytes <= STAGES * L::STAGE_BYTES, "merge buffer reuses the ring");
  static_assert(!kPersist || kRedBytes <= L::STAGE_BYTES, "merge buffer fits one stage");
  constexpr bool kF16 = kQuant;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_addr(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int G = prm.num_q_heads / prm.num_kv_heads;
  const int S = prm.num_splits;
  const bool is_consumer = warp < kConsumerWarps;
  PA_TS_FIRST(prm.ts, 1, kTsEntry);

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::OFF_EMPTY);
  int32_t* pages_s = reinterpret_cast<int32_t*>(smem + L::OFF_PAGES);
  float* ml_s = reinterpret_cast<float*>(smem + L::OFF_ML);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC);
  // chunks the TMA warp has issued (or skipped), and whether it has stopped issuing:
  // the failure path drains exactly the copies that were issued
  volatile int* issued_s = abort_flag + 1;
  volatile int* producer_done = abort_flag + 2;
  uint32_t* skip_s = reinterpret_cast<uint32_t*>(smem + L::OFF_SKIP);
  // Wait (bounded) for the copies of the first `issued` chunks to land: per stage, the
  // phase of its last issued chunk (earlier phases of that stage completed before the
  // stage was refilled, so that phase is the only one that can be pending).
  auto drain_issued = [&](int issued) {
    for (int st = 0; st < STAGES && st < issued; ++st) {
      const int last = st + (issued - 1 - st) / STAGES * STAGES;
      if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>(last / STAGES) & 1u)) break;
    }
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroupWarps);
    }
    *abort_flag = 0;
    *issued_s = 0;
    *producer_done = 0;
    fence_barrier_init();
  }
  __syncthreads();  // barriers initialised; no global load has been issued yet

  // ---- consumers: Q^T fragments in registers, independent of the metadata stage -----
  // (with several queries per request their rows come from cu_seqlens_q, a metadata
  // output, and the persistent form learns its items from the lengths, so Q is loaded
  // after the wait instead).  The TMA warp does not wait for this: it goes straight to
  // the split's length and page indices and starts copying.
  const bool multi = prm.cu_seqlens_q != nullptr;
  uint32_t qb[kNT][8][2];
  float kbias[kNT][2], qf[kNT][2];
  if (!kPersist && !multi && is_consumer)
    load_q_fragments<kF16, kNT>(prm, blockIdx.z, 1, blockIdx.y, G, gid, tig, qb, kbias, qf);

  // ---- everything below reads what the metadata stage wrote -------------------------
  grid_dependency_wait();
#ifdef PA_TIMESTAMPS
  if (prm.ts != nullptr && tid == kConsumerWarps * 32)
    atomicMin(prm.ts + 3 * 1 + kTsReady, global_timer_ns());
#endif
  const int window = kWindow ? prm.window : 0;
  const int cap = prm.max_seq_pages * P;
  const int pps = prm.pages_per_split;
  const int Hkv = prm.num_kv_heads;

  // ---- persistent form: the work list ------------------------------------------------
  int* n_s = reinterpret_cast<int*>(smem + L::OFF_SCHED);  // clamped request lengths
  int* full_s = n_s + kMaxPersistRequests;                  // splits with a full range
  int* part_s = full_s + kMaxPersistRequests;               // pages of the partial split
  int* part_list = part_s + kMaxPersistRequests;            // requests by partial size
  int* pref_s = part_list + kMaxPersistRequests;            // exclusive prefix of full_s
  int* cnt_s = pref_s + kMaxPersistRequests + 1;            // [full splits, partials]
  int total_items = 1;
  if constexpr (kPersist) {
    const int bs = prm.bs;
    for (int r = tid; r < bs; r += kThreads) {
      int n = prm.cache_seqlens[r];
      if (n < 0 || n > cap) {
        if (blockIdx.x == 0) record_error(prm.err, kErrSeqLenOutOfRange);
        n = n < 0 ? 0 : cap;
      }
      // the split partition of a request: from its first visible page (window) or page 0
      const int base = window > 0 ? max(0, n - window) / P : 0;
      const int pages = max(0, (n + P - 1) / P - base);
      const int fulls = min(pages / pps, S);
      n_s[r] = n;
      full_s[r] = fulls;
      part_s[r] = fulls < S ? pages - fulls * pps : 0;
    }
    __syncthreads();
    if (warp == 0) {
      int carry = 0, partials = 0;
      for (int r0 = 0; r0 < bs; r0 += 32) {
        const int r = r0 + lane;
        const int v = r < bs ? full_s[r] : 0;
        int incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int up = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += up;
        }
        if (r < bs) pref_s[r] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
        partials += __popc(__ballot_sync(0xffffffffu, r < bs && part_s[r] > 0));
      }
      if (lane == 0) {
        pref_s[bs] = carry;
        cnt_s[0] = carry;
        cnt_s[1] = partials;
      }
    }
    // rank of each partial split: larger first, ties by request index
    for (int r = tid; r < bs; r += kThreads) {
      const int pr = part_s[r];
      if (pr > 0) {
        int rank = 0;
        for (int q = 0; q < bs; ++q) {
          const int pq = part_s[q];
          rank += (pq > pr || (pq == pr && q < r)) ? 1 : 0;
        }
        part_list[rank] = r;
      }
    }
    __syncthreads();
    total_items = (cnt_s[0] + cnt_s[1]) * Hkv;
  }
  // Item at position `pos` of the persistent form's work list: the splits with a full
  // page range (kv head fastest), then the partial splits by size, largest first.
  auto decode_item = [&](int pos, int& b_, int& kvh_, int& split_) {
    const int full_items = cnt_s[0] * Hkv;
    if (pos < full_items) {
      const int f = pos / Hkv;
      kvh_ = pos - f * Hkv;
      int lo = 0, hi = prm.bs;  // the request whose full splits hold the f-th one
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref_s[mid] <= f) lo = mid; else hi = mid;
      }
      b_ = lo;
      split_ = f - pref_s[lo];
    } else {
      const int k2 = pos - full_items;
      const int rank = k2 / Hkv;
      kvh_ = k2 - rank * Hkv;
      b_ = part_list[rank];
      split_ = full_s[b_];
    }
  };
  // Persistent form: items are claimed one at a time by the TMA warp from this launch's
  // counter (the work list is largest first, so free CTAs take the largest items left);
  // the position of each item travels to the consumers in the descriptor of the stage
  // that holds its first chunk.
  unsigned int* claims = kPersist ? g_work_claims[prm.work_slot] : nullptr;
  int32_t* desc_s = reinterpret_cast<int32_t*>(smem + L::OFF_DESC);
  // TMA warp lane 0, once per CTA: this CTA claims nothing more; the last CTA to get
  // here sets the launch's counters back to zero for the slot's next launch (also when
  // the CTA stops early, so a failed launch leaves its slot clean)
  auto finish_claims = [&]() {
    __threadfence();
    if (atomicAdd(claims + 1, 1u) == gridDim.x - 1) {
      claims[0] = 0;
      claims[1] = 0;
      __threadfence();
    }
  };

  // ring position: chunks this thread's role has issued (TMA warp) or consumed so far
  int gc = 0;
  bool failed = false, triggered = false;
  for (int round = 0;; ++round) {
  int b, kvh, split;
  int item_pos = 0;  // persistent form: the item's position in the work list
  if constexpr (kPersist) {
    int pos = -1;
    if (!is_consumer) {  // claim the next item of the work list
      if (lane == 0 && !*abort_flag) pos = static_cast<int>(atomicAdd(claims, 1u));
      pos = __shfl_sync(0xffffffffu, pos, 0);
      if (pos < 0 || pos >= total_items) break;
    } else {  // learn it from the descriptor of the stage holding its first chunk
      const int stage0 = gc % STAGES;
      if (!mbar_wait_bounded(&full[stage0], static_cast<uint32_t>(gc / STAGES) & 1u) &&
          lane == 0) {
        record_error(prm.err, kErrWaitTimeout);
        *abort_flag = 1;
      }
      consumer_barrier<kConsumerWarps>();  // every consumer warp takes the same path
      if (*abort_flag) {
        failed = true;
        break;
      }
      pos = desc_s[stage0];
      if (pos < 0) break;  // no more work
    }
    decode_item(pos, b, kvh, split);
    item_pos = pos;
    // the consumers load this item's Q rows once its first chunk has landed: bring them
    // into L2 now, while the ring still holds the previous item
    if (!is_consumer && lane < 2 * G)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(prm.q) +
                   (static_cast<int64_t>(b) * prm.num_q_heads + kvh * G) * 256 + lane * 128));
  } else {
    if (round > 0) break;
    b = blockIdx.z;
    kvh = blockIdx.y;
    split = blockIdx.x;
  }

  int q_begin = b, q_len = 1;
  if (multi) {
    q_begin = prm.cu_seqlens_q[b];
    q_len = prm.cu_seqlens_q[b + 1] - q_begin;
    if (q_len < 0 || q_len > prm.max_q_len) {
      if (tid == 0 && split == 0 && kvh == 0) record_error(prm.err, kErrSeqLenOutOfRange);
      q_len = q_len < 0 ? 0 : prm.max_q_len;
    }
    if (is_consumer)
      load_q_fragments<kF16, kNT>(prm, q_begin, q_len, kvh, G, gid, tig, qb, kbias, qf);
  } else if (kPersist && is_consumer) {
    load_q_fragments<kF16, kNT>(prm, b, 1, kvh, G, gid, tig, qb, kbias, qf);
  }
  const int ncols = q_len * G;  // (query, head) columns of this request and kv head

  // Without a window the split's page indices and the request length are independent
  // loads: the TMA warp issues both before either is used (page indices are
  // bounds-checked where they are used).  With a window the split starts at the page of
  // the request's first visible position, which depends on the length.  Only the TMA
  // warp reads the page indices.
  int p_begin = split * pps;
  const int32_t* pt_row = prm.page_table + static_cast<int64_t>(b) * prm.page_table_stride;
  auto cache_page_indices = [&]() {
    pt_row += p_begin;
    const int pages_cap =
        min(min(prm.pages_per_split, prm.max_seq_pages - p_begin), kMaxSplitPages);
    for (int i = lane; i < pages_cap; i += 32) pages_s[i] = pt_row[i];
  };
  if (window == 0 && !is_consumer) cache_page_indices();
  int n;
  if constexpr (kPersist) {
    n = n_s[b];
  } else {
    n = prm.cache_seqlens[b];
    if (n < 0 || n > cap) {
      if (tid == 0 && split == 0 && kvh == 0) record_error(prm.err, kErrSeqLenOutOfRange);
      n = n < 0 ? 0 : cap;
    }
  }
  if (window > 0) {
    p_begin += max(0, n - q_len - window + 1) / P;
    if (!is_consumer) cache_page_indices();
  }
  const int n_pages = (n + P - 1) / P;
  const int p_end = min(p_begin + prm.pages_per_split, n_pages);
  const int tok_begin = p_begin * P;
  const int n_tok = min(p_end * P, n) - tok_begin;

  if (n_tok <= 0) {  // (never an item of the persistent form's work list)
    trigger_dependents();
    if (tid < ncols) {
      const int64_t slot = column_slot(q_begin, tid, G, kvh, prm.num_q_heads, S, split);
      prm.m_out[slot] = -CUDART_INF_F;
      prm.l_out[slot] = 0.f;
    }
    PA_TS_LAST(prm.ts, 1);
    return;
  }

  const int n_split_pages = p_end - p_begin;
  if (!is_consumer) __syncwarp();  // the TMA warp's page indices, cached by its lanes

  const int n_chunks = (n_tok + kChunk - 1) / kChunk;

  // ======================= producer warp: TMA issue loop ============================
  if (!is_consumer) {
#ifdef PA_TIMESTAMPS
    // failure-detection test of the instrumented build: nothing is issued, so every
    // consumer wait gives up after its time limit and the kernel reports it
    if (prm.hold_loads) {
      if (lane == 0) {
        if constexpr (kPersist) finish_claims();
        *producer_done = 1;
      }
      trigger_dependents();
      return;
    }
#endif
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      for (int c = 0; c < n_chunks; ++c) {
        const int g = gc + c;  // ring position of this chunk
        const int stage = g % STAGES;
        if (g >= STAGES) {
          const uint32_t parity = static_cast<uint32_t>(g / STAGES - 1) & 1u;
          if (!mbar_wait_bounded(&empty[stage], parity) || *abort_flag) {
            record_error(prm.err, kErrWaitTimeout);
            *abort_flag = 1;
            break;
          }
        }
        *issued_s = g + 1;
        // the first chunk's stage carries the item to the consumers (published by the
        // arrive on its full barrier below, read after their wait on it)
        if (kPersist && c == 0) desc_s[stage] = item_pos;
        const uint32_t kdst = smem_base + stage * L::STAGE_BYTES;
        const uint32_t vdst = kdst + L::KV_BYTES;
        const int ctok = c * kChunk;
        // -1: a page the sliding-window pool does not hold (window mode only); its
        // tokens are skipped and nothing is loaded for it
        auto page_at = [&](int i) -> int {
          int32_t pg = i < kMaxSplitPages ? pages_s[i] : pt_row[i];
          if (pg < 0 && window > 0) return -1;
          if (pg < 0 || pg >= prm.num_pages) {
            record_error(prm.err, kErrPageOutOfRange);
            pg = 0;
          }
          return pg;
        };
        if constexpr (P >= kChunk) {
          const int pg = page_at(ctok / P);
          const int row = ctok % P;
          // the mask is published by the arrive below (release) and read after the
          // consumers' wait on the same barrier (acquire)
          if constexpr (kWindow) {
            skip_s[stage] = pg < 0 ? 1u : 0u;
            if (pg < 0) {
              mbar_arrive(&full[stage]);
              continue;
            }
          }
          mbar_arrive_expect_tx(&full[stage], 2 * L::KV_BYTES + 2 * L::SCALE_BYTES);
          if constexpr (kQuant) {
            tma_load_4d(kdst, &map_k, 0, row, kvh, pg, &full[stage], policy);
            tma_load_4d(vdst, &map_v, 0, row, kvh, pg, &full[stage], policy);
            const int64_t srow = (static_cast<int64_t>(pg) * prm.num_kv_heads + kvh) * P + row;
            unsigned char* st = smem + stage * L::STAGE_BYTES;
            bulk_copy_g2s(st + 2 * L::KV_BYTES, prm.k_scale + srow, L::SCALE_BYTES, &full[stage],
                          policy);
            bulk_copy_g2s(st + 2 * L::KV_BYTES + L::SCALE_BYTES, prm.v_scale + srow,
                          L::SCALE_BYTES, &full[stage], policy);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_4d(kdst + h * 8192, &map_k, 64 * h, row, kvh, pg, &full[stage], policy);
              tma_load_4d(vdst + h * 8192, &map_v, 64 * h, row, kvh, pg, &full[stage], policy);
            }
          }
        } else {
          constexpr int kPages = kChunk / P;
          const int first = ctok / P;
          const int np = min(kPages, n_split_pages - first);
          constexpr int kPageRows = P * 128;  // bytes of one page's rows in a 128-B-row tile
          int pgs[kPages];
          uint32_t skip = 0;
          int loaded = 0;
#pragma unroll
          for (int k = 0; k < kPages; ++k) {
            pgs[k] = k < np ? page_at(first + k) : -1;
            if (k < np && pgs[k] < 0) skip |= 1u << k;
            loaded += pgs[k] >= 0 ? 1 : 0;
          }
          if constexpr (kWindow) skip_s[stage] = skip;
          if (loaded == 0) {
            mbar_arrive(&full[stage]);
            continue;
          }
          mbar_arrive_expect_tx(&full[stage],
                                loaded * (kQuant ? 2 * (P * 128 + P * 4) : 2 * P * 256));
#pragma unroll
          for (int k = 0; k < kPages; ++k) {
            const int pg = pgs[k];
            if (pg < 0) continue;
            if constexpr (kQuant) {
              tma_load_4d(kdst + k * kPageRows, &map_k, 0, 0, kvh, pg, &full[stage], policy);
              tma_load_4d(vdst + k * kPageRows, &map_v, 0, 0, kvh, pg, &full[stage], policy);
              const int64_t srow = (static_cast<int64_t>(pg) * prm.num_kv_heads + kvh) * P;
              unsigned char* st = smem + stage * L::STAGE_BYTES;
              bulk_copy_g2s(st + 2 * L::KV_BYTES + k * P * 4, prm.k_scale + srow, P * 4,
                            &full[stage], policy);
              bulk_copy_g2s(st + 2 * L::KV_BYTES + L::SCALE_BYTES + k * P * 4,
                            prm.v_scale + srow, P * 4, &full[stage], policy);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                tma_load_4d(kdst + h * 8192 + k * kPageRows, &map_k, 64 * h, 0, kvh, pg,
                            &full[stage], policy);
                tma_load_4d(vdst + h * 8192 + k * kPageRows, &map_v, 64 * h, 0, kvh, pg,
                            &full[stage], policy);
              }
            }
          }
        }
      }
    }
    __syncwarp();  // lane 0 is done with this item's page indices
    gc += n_chunks;
    if (*abort_flag) break;
    continue;
  }

  // ======================= consumer warps =============================================
  // O^T[channel][head] fragments: M-tile i covers 16 channels, n-tile nt 8 heads.
  float o[kNT][8][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int i = 0; i < 8; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
  // int8: the fp16 PV weights are p * v_scale * vmul, with vmul a warp-uniform power of
  // two that puts the largest V scale seen so far in [64, 128): weights stay below
  // 2^kMaxSlack * 128 (no fp16 overflow) and every weight within 2^-20 of the largest
  // one is a normal fp16 number (no subnormal rounding).  o is in those units;
  // vmul only shrinks (exact rescale) when a larger scale appears; it starts at 2^100,
  // so the first slice with a nonzero scale sets it.
  float vmul = 0x1p100f;
  // softmax state of heads 8*nt + 2*tig + e (identical in the 8 lanes sharing tig)
  // m_run: the reference maximum the weights are relative to (warp-uniform per column);
  // t_max: this thread's true maximum of its own scores, reduced once per split.
  // ref: m_run, or 0 while a column has no score yet (its scores are all -inf then)
  // thr: m_run + kMaxSlack, the score above which the reference moves
  float m_run[kNT][2], l_part[kNT][2], t_max[kNT][2], ref[kNT][2], thr[kNT][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
    thr[nt][0] = thr[nt][1] = -CUDART_INF_F;
    t_max[nt][0] = t_max[nt][1] = -CUDART_INF_F;
    l_part[nt][0] = l_part[nt][1] = 0.f;
    ref[nt][0] = ref[nt][1] = 0.f;
  }
  const int group = warp / kGroupWarps;
  const int t0 = (warp % kGroupWarps) * 16;  // this warp's tokens inside its group's chunks
  // Causal limit of this thread's columns, in token positions of the split: query i of a
  // request with q_len queries sees positions < n - q_len + i + 1 (its own token is the
  // request's (q_len - i)-th newest).  One query per request: the whole context.
  int lim[kNT][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 8 * nt + 2 * tig + e;
      lim[nt][e] = col < ncols ? n - q_len + col / G + 1 - tok_begin : 0;
    }
  // With a window, a column sees positions >= lim - window (its query's `window` newest
  // positions); the largest such bound over the request's columns (its newest query,
  // lim = n - tok_begin), relative to the split.
  const int lo_hi = window > 0 ? n - window - tok_begin : INT_MIN;

  for (int c = group; c < n_chunks; c += NG) {
    const int g = gc + c;  // ring position of this chunk
    const int stage = g % STAGES;
    // (a TMA warp that stopped issuing leaves this wait to run out; the consumers do
    // not poll the abort flag on every chunk)
    if (!mbar_wait_bounded(&full[stage], static_cast<uint32_t>(g / STAGES) & 1u)) {
      if (lane == 0) {
        record_error(prm.err, kErrWaitTimeout);
        *abort_flag = 1;
      }
      failed = true;
      break;
    }
    const int valid = min(kChunk, n_tok - c * kChunk);
    unsigned char* st = smem + stage * L::STAGE_BYTES;
    const uint32_t kst = smem_base + stage * L::STAGE_BYTES;
    const uint32_t vst = kst + L::KV_BYTES;
    const bool partial = valid < t0 + 16;
    // a warp's 16 tokens lie on one page (P >= 16); a skipped page was not loaded
    const bool skipped = window > 0 && ((skip_s[stage] >> (t0 / P)) & 1u);
    const bool active = t0 < valid && !skipped;
    // positions below a column's window start occur only in the first slices
    const bool check_lo = c * kChunk + t0 < lo_hi;

    if (active) {
      // Rows of this warp's slice past the context: their V bytes are not ours to trust
      // (stale ring contents or cache slots past the request), so zero them before PV
      // (bf16: 0 * NaN would poison the output).  int8 needs none of it: every byte
      // widens to a finite fp16 number and those rows have weight 0.
      if (!kQuant && partial) {
        for (int r = max(valid, t0) + (lane >> 3); r < t0 + 16; r += 4) {
          uint4* row = reinterpret_cast<uint4*>(st + L::KV_BYTES + r * 128);
          row[lane & 7] = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (!kQuant) {
            uint4* row2 = reinterpret_cast<uint4*>(st + L::KV_BYTES + 8192 + r * 128);
            row2[lane & 7] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        __syncwarp();
      }

      // ---- S^T = K Q^T for tokens t0..t0+15 (M = 16 tokens, N = 8 heads per n-tile) --
      // two accumulators (even / odd k-steps) halve the dependent MMA chain; int8 with
      // one n-tile: the odd one starts at -kbias, which takes the +1152 of the K codes
      // back out (two n-tiles subtract it afterwards, which keeps the register count down)
      constexpr bool kBiasInAcc = kQuant && kNT == 1;
      float acc[2][kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[0][nt][i] = 0.f;
          acc[1][nt][i] = kBiasInAcc ? -kbias[nt][i & 1] : 0.f;
        }
      if constexpr (!kQuant) {
        const int mi = lane >> 3;
        const int row = t0 + (lane & 7) + 8 * (mi & 1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int chunk = 2 * j + (mi >> 1);  // 16-byte chunk of the 256-byte row
          const uint32_t addr = kst + (chunk >> 3) * 8192 + swz(row, chunk & 7);
          uint32_t a[4];
          ldsm_x4(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) mma16816<false>(acc[j & 1][nt], a, qb[nt][j][0], qb[nt][j][1]);
        }
      } else {
        const uint4 r0a = *reinterpret_cast<const uint4*>(st + swz(t0 + gid, 2 * tig));
        const uint4 r0b = *reinterpret_cast<const uint4*>(st + swz(t0 + gid, 2 * tig + 1));
        const uint4 r1a = *reinterpret_cast<const uint4*>(st + swz(t0 + gid + 8, 2 * tig));
        const uint4 r1b = *reinterpret_cast<const uint4*>(st + swz(t0 + gid + 8, 2 * tig + 1));
        const uint32_t w0[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
        const uint32_t w1[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t x0 = w0[j] ^ 0x80808080u, x1 = w1[j] ^ 0x80808080u;
          uint32_t a[4];
          // 1024 + (code + 128) = code + 1152, exact in fp16; the +1152 is removed
          // from the score through kbias (the odd accumulator's start)
          a[0] = __byte_perm(x0, 0x64646464u, 0x4140);  // token gid,     channels +0, +1
          a[1] = __byte_perm(x1, 0x64646464u, 0x4140);  // token gid + 8
          a[2] = __byte_perm(x0, 0x64646464u, 0x4342);  // token gid,     channels +2, +3
          a[3] = __byte_perm(x1, 0x64646464u, 0x4342);  // token gid + 8
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) mma16816<true>(acc[j & 1][nt], a, qb[nt][j][0], qb[nt][j][1]);
        }
      }

      // ---- online softmax (base 2) per head over this warp's 16 tokens ---------------
      const float* kscale = reinterpret_cast<const float*>(st + 2 * L::KV_BYTES);
      const float* vscale = kscale + kChunk;
      const int tok_a = t0 + gid, tok_b = t0 + gid + 8;
      float ks_a = 1.f, ks_b = 1.f, vs_a = 0.f, vs_b = 0.f;
      if constexpr (kQuant) {
        ks_a = kscale[tok_a];
        ks_b = kscale[tok_b];
        vs_a = tok_a < valid ? vscale[tok_a] : 0.f;
        vs_b = tok_b < valid ? vscale[tok_b] : 0.f;
        const float vhi = fmaxf(vs_a, vs_b);
        if (__any_sync(0xffffffffu, vhi * vmul >= 128.f)) {
          float vmax = vhi;  // over the warp's 16 tokens
#pragma unroll
          for (int m = 4; m <= 16; m <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, m));
          if (vmax > 0.f) {
            const float vmul_new = pow2_clamped(6 - float_exponent(vmax));
            if (vmul_new < vmul) {
              const float r = vmul_new / vmul;  // a power of two: exact
#pragma unroll
              for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                  for (int r4 = 0; r4 < 4; ++r4) o[nt][i][r4] *= r;
            }
            if (vmul_new < vmul) vmul = vmul_new;
          }
        }
        vs_a *= vmul;
        vs_b *= vmul;
      }
      uint32_t pb[kNT][2], pl[kNT][2];  // weights (B operand) and their residuals
      // every score of a full slice of a one-query split without a window is visible
      // (columns past the request's heads carry zero queries and are never written)
      const bool need_mask = !PA_MASK_FAST || partial || multi || check_lo;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        float x[4];  // (token a, head e0), (a, e1), (b, e0), (b, e1)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v = (acc[0][nt][i] + acc[1][nt][i]);
          if constexpr (kQuant && !kBiasInAcc) v -= kbias[nt][i & 1];
          v *= qf[nt][i & 1];
          if constexpr (kQuant) v *= (i < 2 ? ks_a : ks_b);
          x[i] = v;
        }
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int pos = c * kChunk + (i < 2 ? tok_a : tok_b);  // position in the split
            bool seen = (i < 2 ? tok_a : tok_b) < valid && pos < lim[nt][i & 1];
            if (check_lo) seen = seen && pos >= lim[nt][i & 1] - window;
            x[i] = seen ? x[i] : -CUDART_INF_F;
          }
        }
        // Reference maximum per column, moved only when a score exceeds it by more than
        // 2^kMaxSlack (one vote instead of a shuffle reduction and a rescale per slice);
        // weights stay <= 2^kMaxSlack and (m, l, acc) stay consistent for any reference.
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
        t_max[nt][0] = fmaxf(t_max[nt][0], mx0);
        t_max[nt][1] = fmaxf(t_max[nt][1], mx1);
        float alpha[2] = {1.f, 1.f}, p[4];
        // (two n-tiles: recomputed, which keeps the register count down)
        const bool grow = kNT == 1 ? mx0 > thr[nt][0] || mx1 > thr[nt][1]
                                   : mx0 > m_run[nt][0] + kMaxSlack || mx1 > m_run[nt][1] + kMaxSlack;
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int m = 4; m <= 16; m <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float m_new = fmaxf(m_run[nt][e], e == 0 ? mx0 : mx1);
            if (m_new != -CUDART_INF_F) {
              alpha[e] = fast_exp2(m_run[nt][e] - m_new);
              m_run[nt][e] = m_new;
              ref[nt][e] = m_new;
              thr[nt][e] = m_new + kMaxSlack;
            }
          }
          if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              o[nt][i][0] *= alpha[0];
              o[nt][i][1] *= alpha[1];
              o[nt][i][2] *= alpha[0];
              o[nt][i][3] *= alpha[1];
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[e] = fast_exp2(x[e] - ref[nt][e]);
          p[2 + e] = fast_exp2(x[2 + e] - ref[nt][e]);
          l_part[nt][e] = l_part[nt][e] * alpha[e] + (p[e] + p[2 + e]);
        }
        // P^T as the B operand of O^T += V^T P^T: transpose the two 8x8 (token, head)
        // blocks in registers.
        uint32_t xa, xb;
        uint32_t ra = 0u, rb = 0u;
        if constexpr (kQuant) {
          const float w0 = p[0] * vs_a, w1 = p[1] * vs_a, w2 = p[2] * vs_b, w3 = p[3] * vs_b;
          xa = pack_f16(w0, w1);
          xb = pack_f16(w2, w3);
          if constexpr (PA_P_SPLIT) {
            const float2 ha = __half22float2(*reinterpret_cast<const __half2*>(&xa));
            const float2 hb = __half22float2(*reinterpret_cast<const __half2*>(&xb));
            ra = pack_f16(w0 - ha.x, w1 - ha.y);
            rb = pack_f16(w2 - hb.x, w3 - hb.y);
          }
        } else {
          xa = pack_bf16(p[0], p[1]);
          xb = pack_bf16(p[2], p[3]);
          if constexpr (PA_P_SPLIT) {
            ra = pack_bf16(p[0] - bf16_lo(xa), p[1] - bf16_hi(xa));
            rb = pack_bf16(p[2] - bf16_lo(xb), p[3] - bf16_hi(xb));
          }
        }
        pb[nt][0] = movmatrix_trans(xa);
        pb[nt][1] = movmatrix_trans(xb);
        if constexpr (PA_P_SPLIT) {
          pl[nt][0] = movmatrix_trans(ra);
          pl[nt][1] = movmatrix_trans(rb);
        }
      }

      // ---- O^T += V^T P^T (M = 16 channels per tile, K = 16 tokens) ----------------------
      if constexpr (kQuant) {
        // ldmatrix.trans of (8 tokens x 16 bytes) matrices: lane (gid, tig) receives the
        // bytes of channels 16i + 2gid, +1 for tokens 2tig, 2tig + 1 of the matrix, so one
        // byte permute per fp16x2 gives an A register of V^T (two tokens of one channel).
        // M-tile i row gid is channel 16i + 2gid, row gid + 8 is channel 16i + 2gid + 1.
        // Matrices per x4 load: tokens t0..+7 / t0+8..+15 of chunk 2ii, then of 2ii + 1.
        const int mrow = t0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          uint32_t x[4];
          ldsm_x4_trans(vst + swz(mrow, 2 * ii + (lane >> 4)), x[0], x[1], x[2], x[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t xa = x[2 * h] ^ 0x80808080u, xb = x[2 * h + 1] ^ 0x80808080u;
            uint32_t a[4] = {biased_bytes_to_f16x2(xa, 0x4240), biased_bytes_to_f16x2(xa, 0x4341),
                             biased_bytes_to_f16x2(xb, 0x4240), biased_bytes_to_f16x2(xb, 0x4341)};
            // exact codes: the +1152 comes off in fp16 (an integer below 2048)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&a[u]),
                                        __floats2half2_rn(1152.f, 1152.f));
              a[u] = *reinterpret_cast<const uint32_t*>(&v);
            }
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              mma16816<true>(o[nt][2 * ii + h], a, pb[nt][0], pb[nt][1]);
              if constexpr (PA_P_SPLIT) mma16816<true>(o[nt][2 * ii + h], a, pl[nt][0], pl[nt][1]);
            }
          }
        }
      } else {
        const int mi = lane >> 3;
        const int row = t0 + (lane & 7) + 8 * (mi >> 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // channels 16i .. 16i + 15
          const int chunk = 2 * i + (mi & 1);
          const uint32_t addr = vst + (chunk >> 3) * 8192 + swz(row, chunk & 7);
          uint32_t a[4];
          ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            mma16816<false>(o[nt][i], a, pb[nt][0], pb[nt][1]);
            if constexpr (PA_P_SPLIT) mma16816<false>(o[nt][i], a, pl[nt][0], pl[nt][1]);
          }
        }
      }
    }
    // this warp is done with the stage; zeroing stores (generic proxy) must be ordered
    // before the TMA (async proxy) refills the buffer
    if (!kQuant && active && partial) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    // (the persistent form keeps the item's last stage for the merge below)
    if (lane == 0 && !(kPersist && c == n_chunks - 1)) mbar_arrive(&empty[stage]);
  }

  if (!kPersist) {  // (the persistent form signals once its CTA has no item left)
    trigger_dependents();
    triggered = true;
  }

  // ---- merge the consumer warps' softmax states, write the split's partials --------
  // Per column: M = the split's true maximum (over warps of the lane-reduced t_max);
  // warp w's weights are relative to its reference m_w <= M, so its sum and output
  // are scaled by 2^(m_w - M).
  float l_head[kNT][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l_part[nt][e], t = t_max[nt][e];
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        v += __shfl_xor_sync(0xffffffffu, v, m);
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, m));
      }
      l_head[nt][e] = v;
      t_max[nt][e] = t;
    }
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int head = 8 * nt + 2 * tig + e;
        ml_s[(warp * 16 + head) * 3 + 0] = m_run[nt][e];
        ml_s[(warp * 16 + head) * 3 + 1] = l_head[nt][e];
        ml_s[(warp * 16 + head) * 3 + 2] = t_max[nt][e];
      }
  }
  consumer_barrier<kConsumerWarps>();
  if (failed || *abort_flag) {
    // Drain what the TMA warp issued so no copy lands after the CTA exits.  It may
    // first sit out its own bounded wait on a stage the consumers never released.
    if (tid == 0) {
      const unsigned long long start = global_timer_ns();
      while (*producer_done == 0 && global_timer_ns() - start < 2 * kWaitLimitNs) {
      }
      if (*producer_done != 0) {
        __threadfence_block();
        drain_issued(*issued_s);
      }
    }
    return;
  }
  // [warps][8 * kNT columns][kRedStride]: the ring (its start, or the held stage)
  const int held_stage = (gc + n_chunks - 1) % STAGES;
  float* red = reinterpret_cast<float*>(kPersist ? smem + held_stage * L::STAGE_BYTES : smem);
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int head = 8 * nt + 2 * tig + e;  // column
      if (head < ncols) {
        float mrow = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mrow = fmaxf(mrow, ml_s[(w * 16 + head) * 3 + 2]);
        float scale = m_run[nt][e] == -CUDART_INF_F ? 0.f : exp2f(m_run[nt][e] - mrow);
        if constexpr (kQuant) scale /= vmul;  // vmul: a power of two
        float* dst = red + (warp * 8 * kNT + head) * kRedStride;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float v0 = o[nt][i][e], v1 = o[nt][i][2 + e];
          if constexpr (kQuant) {  // channels 16i + 2gid and the next one: one 8-byte store
            *reinterpret_cast<float2*>(dst + 16 * i + 2 * gid) = make_float2(v0 * scale, v1 * scale);
          } else {  // channels 16i + gid and 16i + gid + 8
            dst[16 * i + gid] = v0 * scale;
            dst[16 * i + gid + 8] = v1 * scale;
          }
        }
      }
    }
  consumer_barrier<kConsumerWarps>();
  for (int idx = tid; idx < ncols * 32; idx += kConsumerWarps * 32) {
    const int head = idx >> 5, d = (idx & 31) * 4;  // column, channel
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(red + (w * 8 * kNT + head) * kRedStride + d);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    *reinterpret_cast<float4*>(
        prm.acc_out + column_slot(q_begin, head, G, kvh, prm.num_q_heads, S, split) * 128 + d) = sum;
  }
  if (tid < ncols) {
    float mrow = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mrow = fmaxf(mrow, ml_s[(w * 16 + tid) * 3 + 2]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = ml_s[(w * 16 + tid) * 3];
      if (mw != -CUDART_INF_F) lsum += ml_s[(w * 16 + tid) * 3 + 1] * exp2f(mw - mrow);
    }
    const int64_t slot = column_slot(q_begin, tid, G, kvh, prm.num_q_heads, S, split);
    prm.m_out[slot] = mrow * 0.69314718055994530942f;
    prm.l_out[slot] = lsum;
  }
  if constexpr (kPersist) {
    // every consumer has read the merge buffer and ml_s: hand the held stage back (the
    // merge stores are generic-proxy writes the next TMA copy must be ordered after)
    consumer_barrier<kConsumerWarps>();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive(&empty[held_stage]);
  }
  gc += n_chunks;
  }  // item loop

  if (!is_consumer) {
    if (lane == 0) {
      if constexpr (kPersist) {
        // no item left: a stage with descriptor -1 tells the consumers
        if (!*abort_flag) {
          const int stage = gc % STAGES;
          if (gc >= STAGES &&
              (!mbar_wait_bounded(&empty[stage], static_cast<uint32_t>(gc / STAGES - 1) & 1u) ||
               *abort_flag)) {
            record_error(prm.err, kErrWaitTimeout);
            *abort_flag = 1;
          } else {
            desc_s[stage] = -1;
            mbar_arrive(&full[stage]);
          }
        }
        finish_claims();
      }
      // stopped early: the consumers have given up, so nothing else waits for these
      if (*abort_flag) drain_issued(*issued_s);
      __threadfence_block();
      *producer_done = 1;
    }
    trigger_dependents();
    return;
  }
  if (kPersist && failed) {
    // Drain what the TMA warp issued so no copy lands after the CTA exits (it may first
    // sit out its own bounded wait on a stage the consumers never released).
    if (tid == 0) {
      const unsigned long long start = global_timer_ns();
      while (*producer_done == 0 && global_timer_ns() - start < 2 * kWaitLimitNs) {
      }
      if (*producer_done != 0) {
        __threadfence_block();
        drain_issued(*issued_s);
      }
    }
    return;
  }
  if constexpr (kPersist) {
    // splits past a request's last page range: no tokens (m = -inf, l = 0); the
    // (request, kv head) pairs are shared out over the CTAs
    for (int pair = blockIdx.x; pair < prm.bs * Hkv; pair += gridDim.x) {
      const int rb = pair / Hkv, rk = pair - rb * Hkv;
      const int first = full_s[rb] + (part_s[rb] > 0 ? 1 : 0);
      for (int t = tid; t < (S - first) * G; t += kConsumerWarps * 32) {
        const int sp = first + t / G;
        const int64_t slot = column_slot(rb, t % G, G, rk, prm.num_q_heads, S, sp);
        prm.m_out[slot] = -CUDART_INF_F;
        prm.l_out[slot] = 0.f;
      }
    }
  }
  if (!triggered) trigger_dependents();
  PA_TS_LAST(prm.ts, 1);
}

// ---- host side ------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      return nullptr;
    }
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f);
  }
  return f;
}

// Tensor map over a [num_pages, Hkv, P, 128] pool: box of 64 (bf16) or 128 (int8)
// channels by min(P, 64) rows of one (page, kv head), 128-byte swizzle.
inline cudaError_t encode_pool_map(CUtensorMap* map, const void* pool, bool quant, int64_t num_pages,
                                   int num_kv_heads, int page_size) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t esz = quant ? 1 : 2;
  const cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(page_size),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {128 * esz, 128 * esz * page_size,
                                 128 * esz * page_size * num_kv_heads};
  const cuuint32_t box[4] = {quant ? 128u : 64u,
                             static_cast<cuuint32_t>(page_size < kChunk ? page_size : kChunk), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = encode(map, quant ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            4, const_cast<void*>(pool), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kQuant, int P, int STAGES, int MINB, int kNT, bool kWindow, int NG = 1,
          bool kPersist = false>
cudaError_t launch_mma_one(const SplitKParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                           dim3 grid, cudaStream_t stream, bool use_pdl) {
  using L = Layout<kQuant, STAGES, NG * kGroupWarps>;
  constexpr int kThreads = threads_of<NG>();
  void (*kernel)(const CUtensorMap, const CUtensorMap, const SplitKParams) =
      splitk_mma_kernel<kQuant, P, STAGES, MINB, kNT, kWindow, NG, kPersist>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return fail_at(e, "shared-memory attribute");
    configured.fetch_or(bit);
  }
  return fail_at(launch_kernel(kernel, grid, dim3(kThreads), static_cast<size_t>(L::SMEM), stream,
                               use_pdl, mk, mv, p),
                 "cudaLaunchKernelEx");
}

// (STAGES, MINB) for G <= 8 (one n-tile of heads) and for G = 16 (two n-tiles, more
// registers per thread).
// STAGES_DEEP > 0: grids of at most p.sm_count blocks with one n-tile use STAGES_DEEP
// stages, GROUPS_DEEP consumer groups (chunks worked on at once) and one CTA per SM.
// PERSIST: grids of at least two blocks per resident slot (one n-tile, one query per
// request, at most kMaxPersistRequests requests) run the persistent form, one CTA per
// slot.
template <bool kQuant, int STAGES1, int MINB1, int STAGES2, int MINB2, int STAGES_DEEP,
          bool kWindow, int GROUPS_DEEP = 1, bool PERSIST = false>
cudaError_t launch_mma_impl(const SplitKParams& p, int bs, int group, int page_size,
                            cudaStream_t stream, bool use_pdl) {
  CUtensorMap mk, mv;
  cudaError_t e = encode_pool_map(&mk, p.k_cache, kQuant, p.num_pages, p.num_kv_heads, page_size);
  if (e != cudaSuccess) return fail_at(e, "tensor map encode (K)");
  e = encode_pool_map(&mv, p.v_cache, kQuant, p.num_pages, p.num_kv_heads, page_size);
  if (e != cudaSuccess) return fail_at(e, "tensor map encode (V)");
  const dim3 grid(static_cast<unsigned>(p.num_splits), static_cast<unsigned>(p.num_kv_heads),
                  static_cast<unsigned>(bs));
  const bool two_tiles = group * (p.cu_seqlens_q != nullptr ? p.max_q_len : 1) > 8;
  const int64_t blocks = static_cast<int64_t>(grid.x) * grid.y * grid.z;
  const bool deep = STAGES_DEEP > 0 && !two_tiles && blocks <= p.sm_count;
  const int64_t slots = static_cast<int64_t>(p.sm_count) * MINB1;
  const bool persist = PERSIST && !two_tiles && !deep && p.cu_seqlens_q == nullptr &&
                       bs <= kMaxPersistRequests && slots > 0 && blocks >= 2 * slots &&
                       !p.no_persist;
  const dim3 persist_grid(static_cast<unsigned>(persist ? slots : 1));
#define PA_MMA_CASE(PP)                                                                        \
  if (page_size == PP) {                                                                       \
    if constexpr (STAGES_DEEP > 0) {                                                           \
      if (deep)                                                                                \
        return launch_mma_one<kQuant, PP, (STAGES_DEEP > 0 ? STAGES_DEEP : GROUPS_DEEP), 1, 1, \
                              kWindow, GROUPS_DEEP>(p, mk, mv, grid, stream, use_pdl);           \
    }                                                                                          \
    if constexpr (PERSIST) {                                                                   \
      if (persist) {                                                                           \
        SplitKParams pp = p;                                                                   \
        pp.work_slot = static_cast<int32_t>(g_next_work_slot.fetch_add(1) % kWorkSlots);       \
        return launch_mma_one<kQuant, PP, STAGES1, MINB1, 1, kWindow, 1, true>(                \
            pp, mk, mv, persist_grid, stream, use_pdl);                                        \
      }                                                                                        \
    }                                                                                          \
    return two_tiles                                                                           \
               ? launch_mma_one<kQuant, PP, STAGES2, MINB2, 2, kWindow>(p, mk, mv, grid, stream,  \
                                                                         use_pdl)               \
               : launch_mma_one<kQuant, PP, STAGES1, MINB1, 1, kWindow>(p, mk, mv, grid, stream,  \
                                                                         use_pdl);              \
  }
  PA_MMA_CASE(16)
  PA_MMA_CASE(32)
  PA_MMA_CASE(64)
  PA_MMA_CASE(128)
#undef PA_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mma
}  // namespace pa
