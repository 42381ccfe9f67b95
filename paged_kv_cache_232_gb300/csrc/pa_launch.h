// pa_launch.h -- host-side interface between the C ABI (api.cu) and the translation units
// that instantiate the kernels.  Internal to libpagedattn.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode.cuh"

namespace pa {

// Launch the decode piece kernel for (dtype, head_dim, group) on `grid` CTAs; when
// params.part_tokens > 0 and any sequence has more than one piece, also launch the reduce.
cudaError_t launch_decode(int bf16, int head_dim, int group, const DecodeParams& params, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int grid, bool with_reduce, cudaStream_t stream);

struct PrefillParams {
    void* out;                  // [total_q, Hq, D]
    const void* q;              // [total_q, Hq, D]
    const int32_t* block_tables;
    const int32_t* query_start_loc;
    const int32_t* seq_lens;
    unsigned* err;
    int num_chunks, n_q_heads, n_kv_heads, max_blocks_per_seq, num_blocks;
    int tiles_per_chunk;        // query tiles (or CTA units) per (chunk, kv head)
    int lpt;                    // 1: CTAs take units longest-first (schedule fits in shared memory)
    float qk_scale_log2;
};

cudaError_t launch_prefill(int bf16, int head_dim, int group, const PrefillParams& params, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t stream);

}  // namespace pa
