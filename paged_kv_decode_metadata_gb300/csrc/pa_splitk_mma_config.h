// Pipeline depth (STAGES) and resident CTAs per SM (MINB) of the tensor-core split-K
// producer, per KV type; suffix 1: G <= 8 query heads per KV head (one n-tile of
// columns), suffix 2: up to 16 columns (two n-tiles, twice the output fragments).
#pragma once

// G <= 8: two 32 KiB stages (K + V of a 64-token chunk) per CTA, three CTAs per SM.
// G = 16: three stages, two CTAs per SM (twice the output fragments per thread).
#ifndef PA_MMA_BF16_STAGES1
#define PA_MMA_BF16_STAGES1 2
#endif
#ifndef PA_MMA_BF16_MINB1
#define PA_MMA_BF16_MINB1 3
#endif
#ifndef PA_MMA_BF16_STAGES2
#define PA_MMA_BF16_STAGES2 3
#endif
#ifndef PA_MMA_BF16_MINB2
#define PA_MMA_BF16_MINB2 2
#endif

// G <= 8: four 17 KiB stages (codes and scales of a 64-token chunk) per CTA, three CTAs
// per SM.  G = 16: six stages, two CTAs per SM.
#ifndef PA_MMA_INT8_STAGES1
#define PA_MMA_INT8_STAGES1 4
#endif
#ifndef PA_MMA_INT8_MINB1
#define PA_MMA_INT8_MINB1 3
#endif
#ifndef PA_MMA_INT8_STAGES2
#define PA_MMA_INT8_STAGES2 6
#endif
#ifndef PA_MMA_INT8_MINB2
#define PA_MMA_INT8_MINB2 2
#endif

// Grids of at most one block per SM (batch-1 steps): a deep ring instead, one CTA per SM,
// so every chunk of a short split is in flight from the start (the split is latency
// bound, not bandwidth bound).  bf16: four 32 KiB stages; int8: eight 17 KiB stages.
#ifndef PA_MMA_SMALL_GRID_DEEP
#define PA_MMA_SMALL_GRID_DEEP 1
#endif
#ifndef PA_MMA_BF16_STAGES_DEEP
#define PA_MMA_BF16_STAGES_DEEP 4
#endif
#ifndef PA_MMA_INT8_STAGES_DEEP
#define PA_MMA_INT8_STAGES_DEEP 8
#endif
// Consumer groups of four warps in that configuration: each takes every GROUPS-th chunk
// (its own stages of the ring), so GROUPS chunks of a short split are worked on at once.
#ifndef PA_MMA_BF16_GROUPS_DEEP
#define PA_MMA_BF16_GROUPS_DEEP 2
#endif
#ifndef PA_MMA_INT8_GROUPS_DEEP
#define PA_MMA_INT8_GROUPS_DEEP 2
#endif

// Grids of at least two blocks per resident slot run the persistent form (one CTA per
// slot claiming items of a largest-first work list, the next item's copies overlapping
// the current item).  Measured on GB300 it pays where the consumers' arithmetic, not
// the copies, bounds the kernel and the batch is ragged: the int8 full-context
// producer (bs64 ragged: 180.8 -> 174.5 us alone, step 181.7 -> 177.8 us).  bf16 and
// sliding-window steps ran 2-4% slower with it (their blocks' starts already hide
// behind the other resident blocks), so they keep one block per item.
#ifndef PA_MMA_BF16_PERSIST
#define PA_MMA_BF16_PERSIST 0
#endif
#ifndef PA_MMA_INT8_PERSIST
#define PA_MMA_INT8_PERSIST 1
#endif
#ifndef PA_MMA_WINDOW_PERSIST
#define PA_MMA_WINDOW_PERSIST 0
#endif
