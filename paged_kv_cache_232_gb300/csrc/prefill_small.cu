// prefill_small.cu -- instantiations of the prefill-chunk kernel whose units with at most 64
// rows (query tokens x group heads) run M = 64 tiles (pa_prefill_chunk_small_m).
#include "prefill_launch.cuh"

namespace pa {

cudaError_t launch_prefill_small(int bf16, int head_dim, int group, const PrefillParams& p, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, cudaStream_t st) {
    return launch_prefill_any<true>(bf16, head_dim, group, p, tmK, tmV, st);
}

}  // namespace pa
