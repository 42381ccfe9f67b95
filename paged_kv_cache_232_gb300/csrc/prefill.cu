// prefill.cu -- prefill-chunk attention over the paged cache on the tcgen05 tensor cores.
//
// What is computed (mini_engine, "Custom CUDA kernels", paged prefill attention; miniserve,
// "Engine", bottom-right causal mask): for chunk c with q_len query rows and kv length kv_len
// (cached context ctx = kv_len - q_len, plus the chunk's own tokens, already in the cache),
// query row j of head h attends to keys t <= ctx + j of KV head h / G:
//     out[j, h] = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m),  s_t = scale * q[j, h] . K_t.
//
// GB300 design:
//  * One CTA per 128-row query tile of one (chunk, KV head).  The tile packs 128 / G query
//    tokens x the G heads of the group, so each K/V tile feeds all G heads (GQA sharing) and
//    the MMA M dimension is always a full 128.
//  * Warp 4 gathers K and V tiles of 128 keys (8 paged blocks) with one 4-D TMA load per
//    block and 64-column slab, 128-byte swizzled, into two-stage rings.  Block ids come from
//    the chunk's block-table row; blocks past the sequence load zeros (out-of-range block
//    coordinate).
//  * Warp 5 owns 512 TMEM columns and issues the MMAs (one elected lane):
//      S_i = Q K_i^T  (M=128, N=128, K=16 x 8; Q and K K-major)  into one of two S buffers,
//      O  += P_i V_i  (M=128, N=128, K=16 x 8; P K-major, V MN-major)  into the O columns.
//    S_{i+1} is issued before waiting for P_i, so QK of the next tile overlaps the softmax.
//  * Warps 0-3 (thread = query row = TMEM lane) read S rows from TMEM, apply the causal mask
//    (only on tiles that reach past the tile's smallest row limit), and run an online softmax
//    in base 2 with a lazily updated reference max: O and l are rescaled only when the row
//    max grows by more than 2^8, otherwise probabilities up to 2^8 are kept (exact in fp32;
//    the final O / l uses the same reference).  The PV operand must be 16-bit like V, but
//    one 16-bit P costs up to 2^-9 relative per weight -- too much next to the bf16 output
//    rounding for a 2e-3 bound -- so P is split as P_hi = round(p), P_lo = round(p - P_hi)
//    (about 16 significant bits together) and O accumulates P_hi V + P_lo V in fp32.  Both
//    halves go to shared memory in the K-major swizzled layout.
//  * Every mbarrier wait has a time limit; on expiry the kernel flags PA_DEVERR_TIMEOUT, all
//    roles leave their loops, and the TMEM columns are released before exit.
#include "pa_launch.h"
#include "tcgen05.cuh"

namespace pa {
namespace pf {

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per tile
constexpr int D = 128;                  // head_dim
constexpr int SLAB = BN * 128;          // 128 rows x 128 bytes: one 64-column slab
constexpr int TILE = 2 * SLAB;          // a [128 x 128] 16-bit tile
constexpr int Q_OFF = 0;
constexpr int K_OFF = TILE;             // two stages
constexpr int V_OFF = 3 * TILE;         // two stages
constexpr int P_OFF = 5 * TILE;         // P split in two: P_hi, then P_lo
constexpr int BAR_OFF = 7 * TILE;
enum Bar { Q_FULL = 0, K_FULL = 1, K_EMPTY = 3, V_FULL = 5, V_EMPTY = 7, S_FULL = 9, S_EMPTY = 11, P_FULL = 13,
           PV_DONE = 14, NUM_BARS = 15 };
constexpr int TMEM_SLOT_OFF = BAR_OFF + 16 * 8;
constexpr int SMEM_BYTES = TMEM_SLOT_OFF + 16 + 1024;  // + alignment slack
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;         // S buffers at columns 0 and 128
constexpr float RESCALE_LOG2 = 8.f;

}  // namespace pf

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

template <int G, bool BF16>
__global__ void __launch_bounds__(pf::THREADS, 1)
prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using namespace pf;
    using F = F16x2<BF16>;
    constexpr int TQ = BM / G;  // query tokens per tile
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + Q_OFF, sK = sbase + K_OFF, sV = sbase + V_OFF, sP = sbase + P_OFF;
    const uint32_t bars = sbase + BAR_OFF;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + TMEM_SLOT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tiles with the most keys (largest query offset) are scheduled first
    const int per_tile = p.num_chunks * p.n_kv_heads;
    const int tile = p.tiles_per_chunk - 1 - (int)(blockIdx.x / per_tile);
    const int rem = blockIdx.x % per_tile;
    const int c = rem / p.n_kv_heads, g = rem % p.n_kv_heads;

    const int q0 = __ldg(p.query_start_loc + c);
    const int q_len = __ldg(p.query_start_loc + c + 1) - q0;
    const int kv_len = __ldg(p.seq_lens + c);
    if (q_len < 0 || kv_len < q_len || kv_len > p.max_blocks_per_seq * 16) {
        if (tile == 0 && g == 0 && threadIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
        return;
    }
    const int j0 = tile * TQ;
    if (j0 >= q_len) return;  // whole CTA: this tile is past the chunk
    const int ctx = kv_len - q_len;
    const int j_last = min(j0 + TQ, q_len) - 1;
    const int n_keys = ctx + j_last + 1;
    const int n_kt = (n_keys + BN - 1) / BN;
    const int nblk_seq = (kv_len + 15) / 16;

    if (threadIdx.x == 0) {
        mbar_init(bars + 8 * Q_FULL, BM);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bars + 8 * (K_FULL + s), 1);
            mbar_init(bars + 8 * (K_EMPTY + s), 1);
            mbar_init(bars + 8 * (V_FULL + s), 1);
            mbar_init(bars + 8 * (V_EMPTY + s), 1);
            mbar_init(bars + 8 * (S_FULL + s), 1);
            mbar_init(bars + 8 * (S_EMPTY + s), BM);
        }
        mbar_init(bars + 8 * P_FULL, BM);
        mbar_init(bars + 8 * PV_DONE, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tc::alloc(smem_addr(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // ------------------------------------------------------------ softmax warps
        const int r = threadIdx.x;                 // query row of the tile == TMEM lane
        const int jr = j0 + r / G;
        const int hr = g * G + (r % G);
        const bool row_valid = jr < q_len;
        const int lim = row_valid ? ctx + jr : -1;  // keys t <= lim are visible
        const int lim_min = ctx + j0;               // smallest limit among the tile's rows
        {
            const uint16_t* src = static_cast<const uint16_t*>(p.q) + ((size_t)(q0 + jr) * p.n_q_heads + hr) * D;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint4 v = row_valid ? ldg_nc_128(src + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
                sts128(sQ + (ch >> 3) * SLAB + swz128(r, ch & 7), v);
            }
            tc::fence_async_smem();
            mbar_arrive(bars + 8 * Q_FULL);
        }
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float sc = p.qk_scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < n_kt; ++i) {
            const int sb = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * (S_FULL + sb), (i >> 1) & 1, p.err))) { ok = false; break; }
            tc::fence_after();
            float s[BN];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t raw[32];
                tc::ld32(trow + sb * BN + 32 * q, raw);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) s[32 * q + e] = __uint_as_float(raw[e]);
            }
            tc::fence_before();
            mbar_arrive(bars + 8 * (S_EMPTY + sb));

            const int kbase = i * BN;
            if (kbase + BN - 1 > lim_min) {
#pragma unroll
                for (int e = 0; e < BN; ++e) s[e] = (kbase + e <= lim) ? s[e] : -INFINITY;
            }
            float mt = -INFINITY;
#pragma unroll
            for (int e = 0; e < BN; ++e) mt = fmaxf(mt, s[e]);
            mt *= sc;
            float alpha = 1.f;
            bool rescale = false;
            if (m_ref == -INFINITY) {
                m_ref = mt;
            } else if (mt > m_ref + RESCALE_LOG2) {
                alpha = exp2f(m_ref - mt);
                m_ref = mt;
                rescale = true;
            }
            l *= alpha;
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            // in place: s[2e] <- packed P_hi of keys (2e, 2e+1), s[2e+1] <- packed P_lo
#pragma unroll
            for (int e = 0; e < BN / 2; ++e) {
                const float a = exp2f(fmaf(s[2 * e], sc, -mu));
                const float b = exp2f(fmaf(s[2 * e + 1], sc, -mu));
                const uint32_t hi = F::pack_rn(a, b);
                const float2 u = F::unpack(hi);
                s[2 * e] = __uint_as_float(hi);
                s[2 * e + 1] = __uint_as_float(F::pack_rn(a - u.x, b - u.y));
                l += a + b;
            }
            // PV_{i-1} finished: the P buffer is free and O is settled
            if (i > 0 && !__all_sync(0xffffffffu, mbar_wait(bars + 8 * PV_DONE, (i - 1) & 1, p.err))) { ok = false; break; }
            if (__any_sync(0xffffffffu, rescale)) {
                tc::fence_after();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t o[32];
                    tc::ld32(trow + O_COL + 32 * q, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::st32(trow + O_COL + 32 * q, o);
                }
                tc::wait_st();
            }
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint32_t off = (ch >> 3) * SLAB + swz128(r, ch & 7);
                sts128(sP + off, make_uint4(__float_as_uint(s[8 * ch]), __float_as_uint(s[8 * ch + 2]),
                                            __float_as_uint(s[8 * ch + 4]), __float_as_uint(s[8 * ch + 6])));
                sts128(sP + TILE + off, make_uint4(__float_as_uint(s[8 * ch + 1]), __float_as_uint(s[8 * ch + 3]),
                                                   __float_as_uint(s[8 * ch + 5]), __float_as_uint(s[8 * ch + 7])));
            }
            tc::fence_async_smem();
            tc::fence_before();
            mbar_arrive(bars + 8 * P_FULL);
        }
        // epilogue: O / l -> out
        if (ok && __all_sync(0xffffffffu, mbar_wait(bars + 8 * PV_DONE, (n_kt - 1) & 1, p.err))) {
            tc::fence_after();
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            uint16_t* dst = static_cast<uint16_t*>(p.out) + ((size_t)(q0 + jr) * p.n_q_heads + hr) * D;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t o[32];
                tc::ld32(trow + O_COL + 32 * q, o);
                tc::wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = F::pack_rn(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        w.y = F::pack_rn(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        w.z = F::pack_rn(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        w.w = F::pack_rn(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        *reinterpret_cast<uint4*>(dst + 32 * q + 8 * v) = w;
                    }
                }
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ TMA producer warp
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_last();
        const int32_t* bt = p.block_tables + (size_t)c * p.max_blocks_per_seq;
        bool ok = true;
        for (int i = 0; i < n_kt && ok; ++i) {
            const int st = i & 1;
            const uint32_t ph = (i >> 1) & 1;
            int my = p.num_blocks;  // past the sequence (or invalid): out-of-range coordinate, zero fill
            const int b = i * 8 + (lane & 7);
            if (lane < 8 && b < nblk_seq) {
                my = __ldg(bt + b);
                if (my < 0 || my >= p.num_blocks) {
                    flag_error(p.err, PA_DEVERR_BLOCK);
                    my = p.num_blocks;
                }
            }
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t full = bars + 8 * ((kv ? V_FULL : K_FULL) + st);
                const uint32_t empty = bars + 8 * ((kv ? V_EMPTY : K_EMPTY) + st);
                const uint32_t dst0 = (kv ? sV : sK) + st * TILE;
                const CUtensorMap* map = kv ? &tmV : &tmK;
                if (lane == 0 && i >= 2 && !mbar_wait(empty, ph ^ 1, p.err)) ok = false;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(full, TILE);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int blk = __shfl_sync(0xffffffffu, my, j);
                    if (lane == 0) {
                        tma_load_4d(dst0 + j * 2048, map, 0, g, 0, blk, full, pol);
                        tma_load_4d(dst0 + SLAB + j * 2048, map, 64, g, 0, blk, full, pol);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ MMA warp (warp 5)
        constexpr uint32_t ID_QK = tc::idesc_f16(BF16, false, BM, BN);
        constexpr uint32_t ID_PV = tc::idesc_f16(BF16, true, BM, D);
        bool ok = __all_sync(0xffffffffu, mbar_wait(bars + 8 * Q_FULL, 0, p.err));
        int issued_pv = 0;
        auto issue_s = [&](int jt) -> bool {
            const int st = jt & 1;
            bool w = mbar_wait(bars + 8 * (K_FULL + st), (jt >> 1) & 1, p.err);
            if (w && jt >= 2) w = mbar_wait(bars + 8 * (S_EMPTY + st), ((jt - 2) >> 1) & 1, p.err);
            if (!__all_sync(0xffffffffu, w)) return false;
            tc::fence_after();
            if (lane == 0) {
                const uint32_t dS = tmem + (uint32_t)(st * BN);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * SLAB + (k & 3) * 32;
                    tc::mma_f16_ss(dS, tc::sdesc_sw128(sQ + off, 16, 1024), tc::sdesc_sw128(sK + st * TILE + off, 16, 1024),
                                   ID_QK, k > 0);
                }
                tc::commit(bars + 8 * (S_FULL + st));
                tc::commit(bars + 8 * (K_EMPTY + st));
            }
            __syncwarp();
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int i = 0; i < n_kt && ok; ++i) {
            if (i + 1 < n_kt && !issue_s(i + 1)) { ok = false; break; }
            const int st = i & 1;
            bool w = mbar_wait(bars + 8 * P_FULL, i & 1, p.err);
            if (w) w = mbar_wait(bars + 8 * (V_FULL + st), (i >> 1) & 1, p.err);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            if (i == n_kt - 1) {
                // rows of the sequence's last, partial block past kv_len may hold anything
                // (P is 0 there, but 0 * NaN is NaN): zero them in the V tile
                const int z0 = max(kv_len, i * BN), z1 = min(((kv_len + 15) / 16) * 16, (i + 1) * BN);
                const int nz = z1 - z0;
                for (int e = lane; e < 2 * 8 * max(nz, 0); e += 32) {
                    const int row = z0 - i * BN + e / 16;
                    const int half = (e / 8) & 1, ch = e & 7;
                    sts128(sV + st * TILE + half * SLAB + row * 128 + ch * 16, make_uint4(0u, 0u, 0u, 0u));
                }
                tc::fence_async_smem();
                __syncwarp();
            }
            tc::fence_after();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t aoff = (k >> 2) * SLAB + (k & 3) * 32;
                    const uint64_t vdesc = tc::sdesc_sw128(sV + st * TILE + k * 2048, SLAB, 1024);
                    tc::mma_f16_ss(tmem + O_COL, tc::sdesc_sw128(sP + aoff, 16, 1024), vdesc, ID_PV, (i > 0 || k > 0));
                    tc::mma_f16_ss(tmem + O_COL, tc::sdesc_sw128(sP + TILE + aoff, 16, 1024), vdesc, ID_PV, 1u);
                }
                tc::commit(bars + 8 * PV_DONE);
                tc::commit(bars + 8 * (V_EMPTY + st));
            }
            __syncwarp();
            issued_pv = i + 1;
        }
        // make sure every MMA this warp issued has completed before TMEM is released
        if (issued_pv > 0) (void)mbar_wait(bars + 8 * PV_DONE, (issued_pv - 1) & 1, p.err);
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
}

template <int G, bool BF16>
static cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    cudaStream_t st) {
    auto kern = prefill_kernel<G, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = p.tiles_per_chunk * p.num_chunks * p.n_kv_heads;
    kern<<<grid, pf::THREADS, pf::SMEM_BYTES, st>>>(p, tmK, tmV);
    return cudaGetLastError();
}

template <bool BF16>
static cudaError_t by_group(int group, const PrefillParams& p, const CUtensorMap& k, const CUtensorMap& v,
                            cudaStream_t st) {
    switch (group) {
        case 1: return launch_prefill_t<1, BF16>(p, k, v, st);
        case 2: return launch_prefill_t<2, BF16>(p, k, v, st);
        case 4: return launch_prefill_t<4, BF16>(p, k, v, st);
        case 8: return launch_prefill_t<8, BF16>(p, k, v, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prefill(int bf16, int head_dim, int group, const PrefillParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st) {
    if (head_dim != pf::D) return cudaErrorNotSupported;
    return bf16 ? by_group<true>(group, p, tmK, tmV, st) : by_group<false>(group, p, tmK, tmV, st);
}

}  // namespace pa
