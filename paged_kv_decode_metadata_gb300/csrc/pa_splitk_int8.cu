// int8 KV (per-token-per-head fp32 scales) instantiations of the split-K producer.
#include "pa_splitk.cuh"

namespace pa {

// Four 16.5 KiB stages (K + V codes and scales of a 64-token chunk), three CTAs per SM.
cudaError_t launch_splitk_int8(const SplitKParams& p, int bs, int group, int page_size,
                               cudaStream_t stream, bool use_pdl) {
  return launch_splitk_impl<true, 4, 3>(p, bs, group, page_size, stream, use_pdl);
}

}  // namespace pa
