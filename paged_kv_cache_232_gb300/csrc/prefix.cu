// prefix.cu -- instantiations and launcher of the shared-prefix pass of a decode batch: the
// prefill kernel (prefill_kernel.cuh) in shared-prefix mode.
//
// When the sequences of a decode batch share their first prefix_tokens tokens (the same
// physical blocks at the head of every block table: mini_engine, "Features", hash-based prefix
// caching), the prefix part of their attention is one dense contraction per KV head -- rows =
// the sequences' G query heads, keys = the prefix tokens -- which the tcgen05 prefill kernel
// runs once per KV head instead of every sequence streaming the same blocks again.  Each CTA
// takes a pair of 128-row query tiles, one KV head and one piece of the prefix, and writes
// per-row partials (m, l, o) that the suffix decode merges.
#include "prefill_kernel.cuh"

namespace pa {

template <int G, bool BF16, int D>
static cudaError_t launch_prefix_t(const PrefillParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                   cudaStream_t st) {
    auto kern = prefill_kernel<G, BF16, D, true>;
    static std::atomic<unsigned long long> s_done{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(kern), pf::Layout<D>::SMEM_BYTES, s_done);
    if (e != cudaSuccess) return e;
    constexpr int NQ = pf::Layout<D>::NQ;
    PrefillParams q = p;
    q.tiles_per_chunk = (p.tiles_per_chunk + NQ - 1) / NQ;  // CTA units (query-tile pairs) per KV head
    q.lpt = 0;
    const long grid = (long)q.tiles_per_chunk * p.n_kv_heads * p.pf_parts;
    if (grid <= 0 || grid > 0x7fffffffL) return cudaErrorInvalidValue;
    return launch_dependent(kern, (unsigned)grid, pf::THREADS, pf::Layout<D>::SMEM_BYTES, st, q, tmK, tmV);
}

template <bool BF16, int D>
static cudaError_t by_group(int group, const PrefillParams& p, const CUtensorMap& k, const CUtensorMap& v,
                            cudaStream_t st) {
    switch (group) {
        case 1: return launch_prefix_t<1, BF16, D>(p, k, v, st);
        case 2: return launch_prefix_t<2, BF16, D>(p, k, v, st);
        case 4: return launch_prefix_t<4, BF16, D>(p, k, v, st);
        case 8:
            if constexpr (D != 256) return launch_prefix_t<8, BF16, D>(p, k, v, st);
            return cudaErrorNotSupported;
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prefix(int bf16, int head_dim, int group, const PrefillParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t st) {
    if (head_dim == 256)
        return bf16 ? by_group<true, 256>(group, p, tmK, tmV, st) : by_group<false, 256>(group, p, tmK, tmV, st);
    if (head_dim == 128)
        return bf16 ? by_group<true, 128>(group, p, tmK, tmV, st) : by_group<false, 128>(group, p, tmK, tmV, st);
    if (head_dim == 64)
        return bf16 ? by_group<true, 64>(group, p, tmK, tmV, st) : by_group<false, 64>(group, p, tmK, tmV, st);
    return cudaErrorNotSupported;
}

}  // namespace pa
