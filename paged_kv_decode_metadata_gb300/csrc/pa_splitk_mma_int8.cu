// int8 KV instantiations of the tensor-core split-K producer.
#include "pa_splitk_mma.cuh"

namespace pa {

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

cudaError_t launch_splitk_mma_int8(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<true, PA_MMA_INT8_STAGES1, PA_MMA_INT8_MINB1, PA_MMA_INT8_STAGES2,
                              PA_MMA_INT8_MINB2>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
