// pa_launch.h -- host-side interface between the C ABI (api.cu) and the translation units
// that instantiate the kernels.  Internal to libpagedattn.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include "decode.cuh"

namespace pa {

// Raise a kernel's dynamic shared-memory limit once per device: the attribute persists, and
// not touching it again keeps the launch path free of host calls other than the launch itself
// (what a CUDA-graph capture of a decode or prefill step needs).  `done` is one bit per device,
// owned by the launcher of that kernel instantiation.
inline cudaError_t smem_limit_once(const void* func, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}


// Launch `kern` as a programmatic dependent of the previous kernel in the stream: its grid may be
// set up while that kernel drains; the kernel itself executes griddepcontrol.wait before reading
// anything the previous kernel may write (a no-op when that kernel never signalled early).
template <typename Kern, typename... Args>
inline cudaError_t launch_dependent(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                                    Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The dynamic split-K grid that also writes pa_decode_write's rows (decode_kernel_dyn with
// WRITE; instantiated in decode_write.cu for group sizes 1 and 2 and head_dim 64, 128 and 256).
template <int D, int G, bool BF16>
cudaError_t launch_dyn_write(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                             cudaStream_t st);

// Launch the decode piece kernel for (dtype, head_dim, group) on `grid` CTAs; when
// params.part_tokens > 0 and any sequence has more than one piece, also launch the reduce.
// Bytes of the decode kernel's ring for head_dim (64, 128 or 256).
inline int decode_ring_bytes(int head_dim) {
    return head_dim == 256   ? DecodeCfg<256, 1, true>::RING_BYTES
           : head_dim == 128 ? DecodeCfg<128, 1, true>::RING_BYTES
                             : DecodeCfg<64, 1, true>::RING_BYTES;
}

// Units one CTA of the persistent decode grid can run.
inline int decode_list_max() { return DecodeCfg<128, 1, true>::LIST_MAX; }


// CTAs of the decode kernel for (dtype, head_dim, group) that fit on one SM (0 on a CUDA error);
// queried once per device, so a call inside a stream capture makes no CUDA call.
int decode_resident_ctas(int bf16, int head_dim, int group);
// Batches of up to this many sequences get the dynamic split-K grid's tail pieces (its
// per-sequence counts live in shared memory).
constexpr int kDynTailMaxSeqs = 256;
// The same for the dynamic split-K kernel (decode_kernel_dyn).
int decode_dyn_resident_ctas(int bf16, int head_dim, int group);

cudaError_t launch_decode(int bf16, int head_dim, int group, const DecodeParams& params, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int grid, bool with_reduce, cudaStream_t stream);

struct PrefillParams {
    void* out;                  // [total_q, Hq, hd]
    const void* q;              // [total_q, Hq, hd]
    const int32_t* block_tables;
    const int32_t* query_start_loc;
    const int32_t* seq_lens;
    unsigned* err;
    int num_chunks, n_q_heads, n_kv_heads, max_blocks_per_seq, num_blocks;
    int tiles_per_chunk;        // query tiles (or CTA units) per (chunk, kv head)
    int max_q_len;              // host-side bound of the chunks' query lengths (sizes the grid)
    int cpb_log2;               // log2 of the 16-token chunks per cache block; -1: blocks of 8 tokens
    int lpt;                    // 1: CTAs take units longest-first (schedule fits in shared memory)
    float qk_scale_log2;
    int hd;                     // head_dim of q, out and the cache (<= D; columns hd .. D-1 are zero)
    // shared-prefix mode (launch_prefix): the query rows are the decode sequences (q [num_seqs,
    // Hq, hd]), the keys the prefix's tokens [0, prefix_tokens) read through row 0 of
    // block_tables, cut into pieces of piece_tokens; sequence s sees keys t < context_lens[s].
    // Each (sequence, head, piece) gets a partial: pf_m (base-2 log of the weights' reference),
    // pf_l (sum of the weights) and pf_o (the normalised output, kernel head_dim columns).
    const int32_t* context_lens;
    float* pf_m;                // [num_seqs * Hq][pf_parts]
    float* pf_l;                // [num_seqs * Hq][pf_parts]
    float* pf_o;                // [num_seqs * Hq][pf_parts][D]
    int num_seqs, prefix_tokens, piece_tokens, pf_parts;
};

cudaError_t launch_prefill(int bf16, int head_dim, int group, const PrefillParams& params, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t stream);
// The same launch with M = 64 tiles for the units whose rows (query tokens x group heads) fit in 64.
cudaError_t launch_prefill_small(int bf16, int head_dim, int group, const PrefillParams& params,
                                 const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t stream);

// The shared-prefix pass (prefill kernel in shared-prefix mode): grid of query-tile pairs x KV
// heads x prefix pieces.  Its CTAs let a programmatic dependent launch (the suffix decode) start
// at once.
cudaError_t launch_prefix(int bf16, int head_dim, int group, const PrefillParams& params, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t stream);

}  // namespace pa
