// kv_write.cuh -- KV-cache write (mini_engine, "Custom CUDA kernels": a kernel that puts each
// new K/V row into its slot of the paged pool with 16-byte vector copies and leaves padded rows
// out; miniserve, "Engine": slot = block_id * block_size + offset).
//
// A cache row for one slot, [n_kv_heads, head_dim], is contiguous in the
// [num_blocks, block_size, n_kv_heads, head_dim] layout, so the write is a row scatter:
// thread t of a CTA owns 16-byte chunks t, t + blockDim.x, ... of the (K row ++ V row) pair
// (one chunk when the pair has at most 512 of them, as at 8 KV heads x 128), and each CTA walks
// U rows at a time so every thread has U independent 16-byte loads in flight before its
// stores.  Bit-exact: no arithmetic touches the data.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kKvWriteRowsPerIter = 4;

__global__ void kv_write_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value, uint4* k_cache,
                                uint4* v_cache, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                                int row_vecs, int64_t num_slots, unsigned* err) {
    constexpr int U = kKvWriteRowsPerIter;
    const int t = threadIdx.x;
    // the next kernel of the step (the decode, launched as a programmatic dependent) may start its
    // launch now; it waits (griddepcontrol.wait) for this grid to complete before reading the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t r0 = (int64_t)blockIdx.x * U; r0 < num_tokens; r0 += (int64_t)gridDim.x * U) {
        int64_t slot[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = r0 + u;
            slot[u] = (r < num_tokens) ? __ldg(slot_mapping + r) : -1;
            if (slot[u] < -1 || slot[u] >= num_slots) {
                if (t == 0) flag_error(err, PA_DEVERR_SLOT);
                slot[u] = -1;
            }
        }
        for (int k = t; k < 2 * row_vecs; k += blockDim.x) {
            const bool is_v = k >= row_vecs;
            const int c = is_v ? k - row_vecs : k;
            const uint4* src = (is_v ? value : key) + c;
            uint4* dst = (is_v ? v_cache : k_cache) + c;
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (slot[u] >= 0) v[u] = ldg_nc_128(src + (r0 + u) * row_vecs);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (slot[u] >= 0) dst[slot[u] * row_vecs] = v[u];
        }
    }
}

}  // namespace pa
