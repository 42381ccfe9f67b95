// prefill.cu -- instantiations of the prefill-chunk kernel (prefill_kernel.cuh) with 128-row tiles.
#include "prefill_launch.cuh"

namespace pa {

cudaError_t launch_prefill(int bf16, int head_dim, int group, const PrefillParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st) {
    return launch_prefill_any<false>(bf16, head_dim, group, p, tmK, tmV, st);
}

}  // namespace pa
