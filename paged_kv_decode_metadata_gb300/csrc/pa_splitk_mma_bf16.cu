// bf16 KV instantiations of the tensor-core split-K producer.
#include "pa_splitk_mma.cuh"

namespace pa {

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

cudaError_t launch_splitk_mma_bf16(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<false, PA_MMA_BF16_STAGES1, PA_MMA_BF16_MINB1, PA_MMA_BF16_STAGES2,
                              PA_MMA_BF16_MINB2>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
