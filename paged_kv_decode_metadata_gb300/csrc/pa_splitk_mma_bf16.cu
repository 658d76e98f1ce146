// bf16 KV instantiations of the tensor-core split-K producer.
#include "pa_splitk_mma.cuh"

namespace pa {

// Three 32 KiB stages per CTA (K + V of a 64-token chunk), two CTAs per SM.
cudaError_t launch_splitk_mma_bf16(const SplitKParams& p, int bs, int group, int page_size,
                                   cudaStream_t stream, bool use_pdl) {
  return mma::launch_mma_impl<false, 3, 2>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
