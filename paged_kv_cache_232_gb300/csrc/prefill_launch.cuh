// prefill_launch.cuh -- the prefill-chunk kernel's launcher, shared by its two instantiation
// units (prefill.cu: 128-row tiles; prefill_small.cu: M = 64 tiles for units that fit).
#pragma once
#include "prefill_kernel.cuh"

namespace pa {

template <int G, bool BF16, int D, bool SMALL>
static cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    cudaStream_t st) {
    auto kern = prefill_kernel<G, BF16, D, false, SMALL>;
    static std::atomic<unsigned long long> s_done{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kern), pf::Layout<D>::SMEM_BYTES, s_done);
    if (e != cudaSuccess) return e;
    // one CTA per pair of 128-row query tiles of a (chunk, KV head)
    constexpr int NQ = pf::Layout<D>::NQ;
    const int units = (p.tiles_per_chunk + NQ - 1) / NQ;
    PrefillParams q = p;
    q.tiles_per_chunk = units;
    const int ncost = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2) / pf::BN + 2;
    const long sched_words = 2L * p.num_chunks + 1 + ncost + 3 + pf::THREADS / 32;
    q.lpt = (sched_words * 4 <= pf::SCHED_BYTES) ? 1 : 0;
    const int grid = units * p.num_chunks * p.n_kv_heads;
    return launch_dependent(kern, (unsigned)grid, pf::THREADS, pf::Layout<D>::SMEM_BYTES, st, q, tmK, tmV);
}

template <bool BF16, int D, bool SMALL>
static cudaError_t by_group(int group, const PrefillParams& p, const CUtensorMap& k, const CUtensorMap& v,
                            cudaStream_t st) {
    switch (group) {
        case 1: return launch_prefill_t<1, BF16, D, SMALL>(p, k, v, st);
        case 2: return launch_prefill_t<2, BF16, D, SMALL>(p, k, v, st);
        case 4: return launch_prefill_t<4, BF16, D, SMALL>(p, k, v, st);
        case 8:
            if constexpr (D != 256) return launch_prefill_t<8, BF16, D, SMALL>(p, k, v, st);
            return cudaErrorNotSupported;
        default: return cudaErrorInvalidValue;
    }
}

template <bool SMALL>
static cudaError_t launch_prefill_any(int bf16, int head_dim, int group, const PrefillParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, cudaStream_t st) {
    if (head_dim == 256)
        return bf16 ? by_group<true, 256, SMALL>(group, p, tmK, tmV, st) : by_group<false, 256, SMALL>(group, p, tmK, tmV, st);
    if (head_dim == 128)
        return bf16 ? by_group<true, 128, SMALL>(group, p, tmK, tmV, st) : by_group<false, 128, SMALL>(group, p, tmK, tmV, st);
    if (head_dim == 64)
        return bf16 ? by_group<true, 64, SMALL>(group, p, tmK, tmV, st) : by_group<false, 64, SMALL>(group, p, tmK, tmV, st);
    return cudaErrorNotSupported;
}

}  // namespace pa
