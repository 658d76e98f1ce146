// int8 KV instantiations of the tensor-core split-K producer.
#include "pa_splitk_mma.cuh"

namespace pa {

// Six 17 KiB stages per CTA (codes and scales of a 64-token chunk), two CTAs per SM:
// the int8 widening needs more registers than three CTAs per SM leave.
cudaError_t launch_splitk_mma_int8(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<true, 6, 2>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
