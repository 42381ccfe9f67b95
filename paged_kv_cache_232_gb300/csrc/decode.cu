// decode.cu -- instantiations and launchers of the decode kernels (see decode.cuh).
#include "pa_launch.h"

namespace pa {

template <int D, int G, bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                                   bool with_reduce, cudaStream_t st) {
    using C = DecodeCfg<D, G, BF16>;
    auto kern = decode_kernel<D, G, BF16>;
    static std::atomic<unsigned long long> s_done{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, s_done);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(p, tmK, tmV);
    e = cudaGetLastError();
    if (e != cudaSuccess || !with_reduce) return e;
    const size_t red_smem = (size_t)(((p.max_parts + 3) & ~3) + 8 * D) * sizeof(float);
    auto rk = splitk_reduce_kernel<D, BF16>;
    if (red_smem > 227 * 1024) return cudaErrorInvalidValue;
    if (red_smem > 48 * 1024) {
        // set once to the per-CTA maximum, so that no later (larger) piece count needs it again
        static std::atomic<unsigned long long> s_red_done{0};
        e = smem_limit_once(reinterpret_cast<const void*>(rk), 227 * 1024, s_red_done);
        if (e != cudaSuccess) return e;
    }
    rk<<<p.num_seqs * p.n_q_heads, 256, red_smem, st>>>(p);
    return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t by_group(int group, const DecodeParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                            bool r, cudaStream_t st) {
    switch (group) {
        case 1: return launch_decode_t<D, 1, BF16>(p, k, v, grid, r, st);
        case 2: return launch_decode_t<D, 2, BF16>(p, k, v, grid, r, st);
        case 4: return launch_decode_t<D, 4, BF16>(p, k, v, grid, r, st);
        case 8: return launch_decode_t<D, 8, BF16>(p, k, v, grid, r, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(int bf16, int head_dim, int group, const DecodeParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int grid, bool with_reduce, cudaStream_t st) {
    if (head_dim == 128)
        return bf16 ? by_group<128, true>(group, p, tmK, tmV, grid, with_reduce, st)
                    : by_group<128, false>(group, p, tmK, tmV, grid, with_reduce, st);
    if (head_dim == 64)
        return bf16 ? by_group<64, true>(group, p, tmK, tmV, grid, with_reduce, st)
                    : by_group<64, false>(group, p, tmK, tmV, grid, with_reduce, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
