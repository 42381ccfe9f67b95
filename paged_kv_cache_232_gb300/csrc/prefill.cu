// prefill.cu -- prefill-chunk attention on the tcgen05 tensor cores (in progress).
#include "pa_launch.h"

namespace pa {

cudaError_t launch_prefill(int, int, int, const PrefillParams&, const CUtensorMap&, const CUtensorMap&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace pa
