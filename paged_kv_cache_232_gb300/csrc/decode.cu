// decode.cu -- instantiations and launchers of the decode kernels (see decode.cuh).
#include "pa_launch.h"

namespace pa {

// per kernel instantiation: the devices whose shared-memory limit for it has been raised
template <int D, int G, bool BF16, bool PERSIST>
static std::atomic<unsigned long long>& smem_flag() {
    static std::atomic<unsigned long long> f{0};
    return f;
}

// CTAs of the instantiation resident per SM (registers, shared memory, launch bounds),
// queried once per device and cached.
template <int D, int G, bool BF16>
static int resident_t() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int r = cache[dev & 63].load(std::memory_order_acquire);
    if (r > 0) return r;
    using C = DecodeCfg<D, G, BF16>;
    auto kern = decode_kernel<D, G, BF16>;
    if (smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, smem_flag<D, G, BF16, false>()) !=
        cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kern, C::THREADS, C::SMEM_BYTES) != cudaSuccess || r < 1)
        return 0;
    cache[dev & 63].store(r, std::memory_order_release);
    return r;
}

template <int D, int G, bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                                   bool with_reduce, cudaStream_t st) {
    using C = DecodeCfg<D, G, BF16>;
    cudaError_t e;
    // always a programmatic dependent launch: its grid is set up while the previous kernel of the
    // stream drains (a KV write signals at its start), and its CTAs wait (griddepcontrol.wait)
    // before reading anything; after a shared-prefix pass they wait only at their merge
    auto launch = [&](auto kern, int smem) -> cudaError_t {
        return launch_dependent(kern, (unsigned)grid, C::THREADS, (size_t)smem, st, p, tmK, tmV);
    };
    if (p.dyn) {
        // group sizes 1 and 2 only (at 4 the piece loop spills and the static grid is faster)
        if constexpr (G <= 2) {
            static_assert(C::DYN_SMAX == kDynTailMaxSeqs, "tail-piece batch limit");
            if (p.new_k) {
                // pa_decode_write: the instantiation that writes the step's rows (decode_write.cu)
                e = launch_dyn_write<D, G, BF16>(p, tmK, tmV, grid, st);
            } else {
                auto kern = decode_kernel_dyn<D, G, BF16>;
                static std::atomic<unsigned long long> s_dyn{0};
                e = smem_limit_once(reinterpret_cast<const void*>(kern), C::D_SMEM_BYTES, s_dyn);
                if (e != cudaSuccess) return e;
                e = launch(kern, C::D_SMEM_BYTES);
            }
        } else {
            return cudaErrorInvalidValue;
        }
    } else if (p.persist) {
        // group sizes 1 and 2 only: larger groups run out of registers in the unit loop
        if constexpr (G <= 2) {
            auto kern = decode_kernel_persistent<D, G, BF16>;
            e = smem_limit_once(reinterpret_cast<const void*>(kern), C::P_SMEM_BYTES, smem_flag<D, G, BF16, true>());
            if (e != cudaSuccess) return e;
            e = launch(kern, C::P_SMEM_BYTES);
        } else {
            return cudaErrorInvalidValue;
        }
    } else {
        auto kern = decode_kernel<D, G, BF16>;
        e = smem_limit_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, smem_flag<D, G, BF16, false>());
        if (e != cudaSuccess) return e;
        e = launch(kern, C::SMEM_BYTES);
    }
    if (e != cudaSuccess || !with_reduce) return e;
    // a programmatic dependent launch: the merge grid is set up while the piece kernel drains and
    // waits for it (griddepcontrol.wait) before reading the partials
    const int rows = p.num_seqs * p.n_q_heads;
    constexpr int per_cta = 8;  // rows (warps) per CTA
    return launch_dependent(splitk_merge_kernel<D, BF16>, (unsigned)((rows + per_cta - 1) / per_cta), 32 * per_cta, 0,
                            st, p);
}

template <int D, bool BF16>
static cudaError_t by_group(int group, const DecodeParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                            bool r, cudaStream_t st) {
    switch (group) {
        case 1: return launch_decode_t<D, 1, BF16>(p, k, v, grid, r, st);
        case 2: return launch_decode_t<D, 2, BF16>(p, k, v, grid, r, st);
        case 4: return launch_decode_t<D, 4, BF16>(p, k, v, grid, r, st);
        case 8:
            if constexpr (D != 256) return launch_decode_t<D, 8, BF16>(p, k, v, grid, r, st);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int D, bool BF16>
static int resident_by_group(int group) {
    switch (group) {
        case 1: return resident_t<D, 1, BF16>();
        case 2: return resident_t<D, 2, BF16>();
        case 4: return resident_t<D, 4, BF16>();
        case 8:
            if constexpr (D != 256) return resident_t<D, 8, BF16>();
            return 0;
        default: return 0;
    }
}

// CTAs of the dynamic split-K kernel resident per SM (0 on a CUDA error), queried once per device.
template <int D, int G, bool BF16>
static int dyn_resident_t() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int r = cache[dev & 63].load(std::memory_order_acquire);
    if (r > 0) return r;
    using C = DecodeCfg<D, G, BF16>;
    auto kern = decode_kernel_dyn<D, G, BF16>;
    static std::atomic<unsigned long long> s_dyn_q{0};
    if (smem_limit_once(reinterpret_cast<const void*>(kern), C::D_SMEM_BYTES, s_dyn_q) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kern, C::THREADS, C::D_SMEM_BYTES) != cudaSuccess || r < 1)
        return 0;
    cache[dev & 63].store(r, std::memory_order_release);
    return r;
}

template <int D, bool BF16>
static int dyn_resident_by_group(int group) {
    switch (group) {
        case 1: return dyn_resident_t<D, 1, BF16>();
        case 2: return dyn_resident_t<D, 2, BF16>();
        default: return 0;  // the dynamic grid runs group sizes 1 and 2 only
    }
}

int decode_dyn_resident_ctas(int bf16, int head_dim, int group) {
    if (head_dim == 256) return bf16 ? dyn_resident_by_group<256, true>(group) : dyn_resident_by_group<256, false>(group);
    if (head_dim == 128) return bf16 ? dyn_resident_by_group<128, true>(group) : dyn_resident_by_group<128, false>(group);
    if (head_dim == 64) return bf16 ? dyn_resident_by_group<64, true>(group) : dyn_resident_by_group<64, false>(group);
    return 0;
}

int decode_resident_ctas(int bf16, int head_dim, int group) {
    if (head_dim == 256) return bf16 ? resident_by_group<256, true>(group) : resident_by_group<256, false>(group);
    if (head_dim == 128) return bf16 ? resident_by_group<128, true>(group) : resident_by_group<128, false>(group);
    if (head_dim == 64) return bf16 ? resident_by_group<64, true>(group) : resident_by_group<64, false>(group);
    return 0;
}

cudaError_t launch_decode(int bf16, int head_dim, int group, const DecodeParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int grid, bool with_reduce, cudaStream_t st) {
    if (head_dim == 256)
        return bf16 ? by_group<256, true>(group, p, tmK, tmV, grid, with_reduce, st)
                    : by_group<256, false>(group, p, tmK, tmV, grid, with_reduce, st);
    if (head_dim == 128)
        return bf16 ? by_group<128, true>(group, p, tmK, tmV, grid, with_reduce, st)
                    : by_group<128, false>(group, p, tmK, tmV, grid, with_reduce, st);
    if (head_dim == 64)
        return bf16 ? by_group<64, true>(group, p, tmK, tmV, grid, with_reduce, st)
                    : by_group<64, false>(group, p, tmK, tmV, grid, with_reduce, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
