// int8 KV instantiations of the tensor-core split-K producer, sliding-window variant
// (its own translation unit, so it compiles beside the full-context one).
#include "pa_splitk_mma.cuh"
#include "pa_splitk_mma_config.h"

namespace pa {

cudaError_t launch_splitk_mma_window_int8(const SplitKParams& p, int bs, int group,
                                          int page_size, cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<true, PA_MMA_INT8_STAGES1, PA_MMA_INT8_MINB1, PA_MMA_INT8_STAGES2,
                              PA_MMA_INT8_MINB2,
                              PA_MMA_SMALL_GRID_DEEP ? PA_MMA_INT8_STAGES_DEEP : 0, true,
                              PA_MMA_INT8_GROUPS_DEEP, PA_MMA_WINDOW_PERSIST>(
      p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
