// rope_write.cuh -- KV-cache write with rotary position embedding applied on the way, and the
// query rows rotated in place (mini_engine, "Roadmap": a planned kernel that applies the rotary
// embedding inside the KV-cache write; "Features": the Qwen3 decoder's RoPE; miniserve, "Engine": per forward, the qkv
// projection and RoPE, then the KV write at slot = block_id * block_size + offset).
//
// Rotation (rotate-half pairing): dims i and i + D/2 of a row at position m turn by the angle
// m f_i, with cos / sin read from a float32 table row [cos(m f_0..), sin(m f_0..)].  Work per
// token row: Hq * D/16 query pairs, Hkv * D/16 key pairs and Hkv * D/8 value chunks, one per
// thread.  A pair is the 16-byte chunk of dims [8c, 8c+8) with the chunk of dims [8c + D/2,
// 8c + D/2 + 8): both halves of eight rotations, so no thread needs another's data.  The
// rotation runs in fp32 and each result is rounded once to the 16-bit format (nearest even).
#pragma once

#include "pa_device.cuh"

namespace pa {


__device__ __forceinline__ float4 ldg_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Rotate the eight pairs (lo[e], hi[e]) by the table's cos / sin at offsets c8 .. c8+7.
template <bool BF16>
__device__ __forceinline__ void rope8(uint4& lo, uint4& hi, const float* cs_row, int c8, int half) {
    using F = F16x2<BF16>;
    const float4 ca = ldg_f4(cs_row + c8), cb = ldg_f4(cs_row + c8 + 4);
    const float4 sa = ldg_f4(cs_row + half + c8), sb = ldg_f4(cs_row + half + c8 + 4);
    const float c[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
    const float s[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    uint32_t l[4] = {lo.x, lo.y, lo.z, lo.w}, h[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 a = F::unpack(l[k]), b = F::unpack(h[k]);
        const float y0 = fmaf(a.x, c[2 * k], -(b.x * s[2 * k]));
        const float y1 = fmaf(a.y, c[2 * k + 1], -(b.y * s[2 * k + 1]));
        const float z0 = fmaf(b.x, c[2 * k], a.x * s[2 * k]);
        const float z1 = fmaf(b.y, c[2 * k + 1], a.y * s[2 * k + 1]);
        l[k] = F::pack_rn(y0, y1);
        h[k] = F::pack_rn(z0, z1);
    }
    lo = make_uint4(l[0], l[1], l[2], l[3]);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
}

// R: rows whose loads each thread has in flight at once (2 at bandwidth scale, 1 for small batches,
// where more CTAs matter more)
template <bool BF16, int D, int R>
__global__ void rope_write_kernel(uint4* q, const uint4* __restrict__ key, const uint4* __restrict__ value,
                                  uint4* k_cache, uint4* v_cache, const int64_t* __restrict__ slot_mapping,
                                  const int64_t* __restrict__ positions, const float* __restrict__ cos_sin,
                                  int64_t num_tokens, int n_q_heads, int n_kv_heads, int64_t num_slots,
                                  int64_t max_position, unsigned* err) {
    constexpr int VEC = D / 8;     // 16-byte chunks per head row
    constexpr int PAIRS = D / 16;  // rotation chunk pairs per head row (= chunk distance of D/2)
    const int nq = q ? n_q_heads * PAIRS : 0, nk = n_kv_heads * PAIRS, nv = n_kv_heads * VEC;
    const int units = nq + nk + nv;
    // the next kernel of the step (the decode, launched as a programmatic dependent) may start its
    // launch now; it waits (griddepcontrol.wait) for this grid to complete before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t r0 = (int64_t)blockIdx.x * R; r0 < num_tokens; r0 += (int64_t)gridDim.x * R) {
        int64_t pos[R], slot[R];
        bool live[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int64_t r = r0 + i;
            live[i] = r < num_tokens;
            pos[i] = live[i] ? __ldg(positions + r) : 0;
            slot[i] = live[i] ? __ldg(slot_mapping + r) : -1;
            if (live[i] && (pos[i] < 0 || pos[i] >= max_position)) {  // the row is left untouched
                if (threadIdx.x == 0) flag_error(err, PA_DEVERR_POSITION);
                live[i] = false;
            }
            if (live[i] && (slot[i] < -1 || slot[i] >= num_slots)) {
                if (threadIdx.x == 0) flag_error(err, PA_DEVERR_SLOT);
                slot[i] = -1;
            }
        }
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            // the unit: a query pair, a key pair or a value chunk of head h, chunk c
            const int kind = u < nq ? 0 : (u < nq + nk ? 1 : 2);
            const int uu = kind == 0 ? u : (kind == 1 ? u - nq : u - nq - nk);
            const int h = kind == 2 ? uu / VEC : uu / PAIRS;
            const int c = kind == 2 ? uu % VEC : uu % PAIRS;
            bool act[R];
            uint4 lo[R], hi[R];
#pragma unroll
            for (int i = 0; i < R; ++i) {  // every row's loads before any arithmetic
                const int64_t r = r0 + i;
                act[i] = live[i] && (kind == 0 || slot[i] >= 0);
                if (!act[i]) continue;
                if (kind == 0) {  // read and written back by this thread only
                    const uint4* row = q + (r * n_q_heads + h) * VEC;
                    lo[i] = row[c];
                    hi[i] = row[c + PAIRS];
                } else if (kind == 1) {
                    const uint4* row = key + (r * n_kv_heads + h) * VEC;
                    lo[i] = ldg_nc_128(row + c);
                    hi[i] = ldg_nc_128(row + c + PAIRS);
                } else {
                    lo[i] = ldg_nc_128(value + (r * n_kv_heads + h) * VEC + c);
                }
            }
#pragma unroll
            for (int i = 0; i < R; ++i) {
                if (!act[i]) continue;
                const int64_t r = r0 + i;
                if (kind == 2) {
                    v_cache[(slot[i] * n_kv_heads + h) * VEC + c] = lo[i];
                    continue;
                }
                rope8<BF16>(lo[i], hi[i], cos_sin + pos[i] * D, 8 * c, D / 2);
                uint4* dst = kind == 0 ? q + (r * n_q_heads + h) * VEC : k_cache + (slot[i] * n_kv_heads + h) * VEC;
                dst[c] = lo[i];
                dst[c + PAIRS] = hi[i];
            }
        }
    }
}

}  // namespace pa
