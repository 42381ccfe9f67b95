// decode_write.cu -- the dynamic split-K grid's instantiations that also write the step's new
// K/V rows (pa_decode_write), in a translation unit of their own so that they compile beside
// decode.cu's.
#include "decode.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int G, bool BF16>
cudaError_t launch_dyn_write(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                             cudaStream_t st) {
    using C = DecodeCfg<D, G, BF16>;
    auto kern = decode_kernel_dyn<D, G, BF16, true>;
    static std::atomic<unsigned long long> s_flag{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kern), C::D_SMEM_BYTES, s_flag);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, (unsigned)grid, C::THREADS, (size_t)C::D_SMEM_BYTES, st, p, tmK, tmV);
}

#define PA_DYN_WRITE(D, G, BF16)                                                                               \
    template cudaError_t launch_dyn_write<D, G, BF16>(const DecodeParams&, const CUtensorMap&, const CUtensorMap&, \
                                                      int, cudaStream_t);
PA_DYN_WRITE(64, 1, false)
PA_DYN_WRITE(64, 1, true)
PA_DYN_WRITE(64, 2, false)
PA_DYN_WRITE(64, 2, true)
PA_DYN_WRITE(128, 1, false)
PA_DYN_WRITE(128, 1, true)
PA_DYN_WRITE(128, 2, false)
PA_DYN_WRITE(128, 2, true)
PA_DYN_WRITE(256, 1, false)
PA_DYN_WRITE(256, 1, true)
PA_DYN_WRITE(256, 2, false)
PA_DYN_WRITE(256, 2, true)
#undef PA_DYN_WRITE

}  // namespace pa
