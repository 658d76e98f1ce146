// bf16 KV instantiations of the split-K producer.
#include "pa_splitk.cuh"

namespace pa {

// Three 32 KiB stages (K + V of a 64-token chunk) per CTA, two CTAs per SM.
cudaError_t launch_splitk_bf16(const SplitKParams& p, int bs, int group, int page_size,
                               cudaStream_t stream, bool use_pdl) {
  return launch_splitk_impl<false, 3, 2>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
