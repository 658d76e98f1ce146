// bf16 KV instantiations of the tensor-core split-K producer.
#include "pa_splitk_mma.cuh"
#include "pa_splitk_mma_config.h"

namespace pa {

cudaError_t launch_splitk_mma_bf16(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<false, PA_MMA_BF16_STAGES1, PA_MMA_BF16_MINB1, PA_MMA_BF16_STAGES2,
                              PA_MMA_BF16_MINB2,
                              PA_MMA_SMALL_GRID_DEEP ? PA_MMA_BF16_STAGES_DEEP : 0, false,
                              PA_MMA_BF16_GROUPS_DEEP, PA_MMA_BF16_PERSIST>(
      p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
