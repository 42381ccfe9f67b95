// decode_static_scratch.cu -- split-K decode for callers that cannot allocate device memory.
//
// pa_decode_splitk needs a scratch buffer for its per-piece (max, exp-sum, output) partials,
// and normally the caller allocates it.  Some callers cannot: code that runs inside a host
// framework which owns every device allocation (a raw cudaMalloc would bypass its pool and
// its accounting), code on a latency-critical path where an allocation's implicit device
// synchronisation is not acceptable, and code running under a capture mode in which
// cudaMalloc is not permitted.  pa_decode_splitk_static gives them the same computation with
// the scratch taken from a fixed array that lives in this library's device image.
//
// The array is a file-scope __device__ object: every GPU that loads the library holds
// PA_STATIC_SCRATCH_BYTES of device memory for it until the process exits.  Host code cannot
// use the array's name as a device address (on the host it names a stand-in object), so the
// entry point looks up the real address with cudaGetSymbolAddress once per device and passes
// that pointer down.
#include <cuda_runtime.h>

#include <mutex>

#include "pagedattn.h"

namespace {

static __device__ __align__(256) unsigned char g_splitk_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitk_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_splitk_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int max_context_len, int num_seqs,
                                       int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                       int64_t num_blocks, float scale, int dtype, int partition_tokens,
                                       void* stream) {
    // the partials these sizes need, in the layout pa_decode_workspace_size describes
    const size_t need = pa_decode_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len, partition_tokens);
    if (need > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (num_seqs > 0 && need > 0) {
        const int st = scratch_address(&scratch);
        if (st != PA_OK) return st;
    }
    return pa_decode_splitk(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            max_context_len, num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks,
                            scale, dtype, partition_tokens, scratch, scratch ? (size_t)PA_STATIC_SCRATCH_BYTES : 0,
                            stream);
}
