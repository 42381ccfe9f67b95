// prefill.cu -- prefill-chunk attention over the paged cache on the tcgen05 tensor cores.
//
// What is computed (mini_engine, "Custom CUDA kernels", paged prefill attention; miniserve,
// "Engine", bottom-right causal mask): for chunk c with q_len query rows and kv length kv_len
// (cached context ctx = kv_len - q_len, plus the chunk's own tokens, already in the cache),
// query row j of head h attends to keys t <= ctx + j of KV head h / G:
//     out[j, h] = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m),  s_t = scale * q[j, h] . K_t.
//
// GB300 design:
//  * A query tile is 128 rows = 128 / G query tokens x the G heads of one KV head, so every
//    K/V tile feeds all G heads (GQA sharing) and the MMA M dimension is a full 128.  One CTA
//    owns two consecutive query tiles of one (chunk, KV head): both read the same K/V tiles.
//  * Warp 8 gathers K and V tiles of 128 keys (8 paged blocks) with one 4-D TMA load per
//    block and 64-column slab, 128-byte swizzled, into two-stage rings.  Block ids come from
//    the chunk's block-table row; blocks past the sequence load zeros (out-of-range block
//    coordinate).
//  * Warp 9 owns all 512 TMEM columns -- S_0 | S_1 | O_0 | O_1, 128 each -- and issues the
//    MMAs from one lane:  S_t = Q_t K^T (both operands from shared memory, K-major) and
//    O_t += P_t V (P from TMEM, V from shared memory, MN-major).  Issue order per key tile
//    j is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): while one softmax warpgroup works on its S,
//    the tensor cores run the other tile's PV and next QK (ping-pong).
//  * Warpgroup t (warps 4t..4t+3; thread = query row = TMEM lane) reads its S row in
//    32-column pieces twice (max, then probabilities), applies the causal mask only on key
//    tiles that reach past the tile's smallest row limit, and keeps an online softmax in
//    base 2 with a lazily updated reference max: O and l are rescaled only when the row max
//    grows by more than 2^8; otherwise weights up to 2^8 are kept (exact in fp32, and the
//    final O / l uses the same reference).  The PV operand is 16-bit, and one 16-bit weight
//    costs up to 2^-9 relative -- too much next to the bf16 output rounding for a 2e-3
//    bound -- so each weight goes in as P_hi = round(p) plus P_lo = round(p - P_hi) (about
//    16 significant bits together), both written over the S columns just read, and the PV
//    step issues one MMA for each half into the same fp32 accumulator.
//  * Every mbarrier wait has a time limit; on expiry the kernel flags PA_DEVERR_TIMEOUT, all
//    roles leave their loops, and the TMEM columns are released before exit.
#include "pa_launch.h"
#include "tcgen05.cuh"

namespace pa {
namespace pf {

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per tile
constexpr int D = 128;                  // head_dim
constexpr int NQT = 2;                  // query tiles per CTA
constexpr int SLAB = BN * 128;          // 128 rows x 128 bytes: one 64-column slab
constexpr int TILE = 2 * SLAB;          // a [128 x 128] 16-bit tile
constexpr int Q_OFF = 0;                // NQT tiles
constexpr int K_OFF = NQT * TILE;       // two stages
constexpr int V_OFF = K_OFF + 2 * TILE; // two stages
constexpr int BAR_OFF = V_OFF + 2 * TILE;
enum Bar { Q_FULL = 0, K_FULL = 1, K_EMPTY = 3, V_FULL = 5, V_EMPTY = 7, S_FULL = 9, P_FULL = 11, PV_DONE = 13,
           DRAIN = 15, NUM_BARS = 16 };
constexpr int TMEM_SLOT_OFF = BAR_OFF + 16 * 8;
constexpr int SMEM_BYTES = TMEM_SLOT_OFF + 16 + 1024;  // + alignment slack
constexpr int THREADS = (4 * NQT + 2) * 32;
constexpr int TMA_WARP = 4 * NQT, MMA_WARP = 4 * NQT + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;         // S_t at columns 128 t, O_t at 256 + 128 t
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
    const uint32_t sQ = sbase + Q_OFF, sK = sbase + K_OFF, sV = sbase + V_OFF;
    const uint32_t bars = sbase + BAR_OFF;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + TMEM_SLOT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTAs with the most keys (largest query offset) are scheduled first
    const int per_unit = p.num_chunks * p.n_kv_heads;
    const int unit = p.tiles_per_chunk - 1 - (int)(blockIdx.x / per_unit);
    const int rem = blockIdx.x % per_unit;
    const int c = rem / p.n_kv_heads, g = rem % p.n_kv_heads;

    const int q0 = __ldg(p.query_start_loc + c);
    const int q_len = __ldg(p.query_start_loc + c + 1) - q0;
    const int kv_len = __ldg(p.seq_lens + c);
    if (q_len < 0 || kv_len < q_len || kv_len > p.max_blocks_per_seq * 16) {
        if (unit == 0 && g == 0 && threadIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
        return;
    }
    const int j0 = unit * NQT * TQ;
    if (j0 >= q_len) return;  // whole CTA: past the chunk
    const int ctx = kv_len - q_len;
    int n_kt[NQT];            // key tiles each query tile needs (0: tile past the chunk)
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
        const int jt = j0 + t * TQ;
        n_kt[t] = (jt < q_len) ? (ctx + min(jt + TQ, q_len) + BN - 1) / BN : 0;
    }
    const int n_max = n_kt[NQT - 1] > n_kt[0] ? n_kt[NQT - 1] : n_kt[0];
    const int nblk_seq = (kv_len + 15) / 16;

    if (threadIdx.x == 0) {
        mbar_init(bars + 8 * Q_FULL, NQT * BM);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bars + 8 * (K_FULL + s), 1);
            mbar_init(bars + 8 * (K_EMPTY + s), 1);
            mbar_init(bars + 8 * (V_FULL + s), 1);
            mbar_init(bars + 8 * (V_EMPTY + s), 1);
            mbar_init(bars + 8 * (S_FULL + s), 1);
            mbar_init(bars + 8 * (P_FULL + s), BM);
            mbar_init(bars + 8 * (PV_DONE + s), 1);
        }
        mbar_init(bars + 8 * DRAIN, 1);
        fence_barrier_init();
    }
    if (warp == MMA_WARP) {
        tc::alloc(smem_addr(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4 * NQT) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;                    // query tile of this warpgroup
        const int r = threadIdx.x & 127;            // row of the tile == TMEM lane
        const int jt0 = j0 + t * TQ;
        const int jr = jt0 + r / G;
        const int hr = g * G + (r % G);
        const bool row_valid = jr < q_len;
        const int lim = row_valid ? ctx + jr : -1;  // keys <= lim are visible
        const int lim_min = ctx + jt0;              // smallest limit among the tile's rows
        const int nkt = (t == 0) ? n_kt[0] : n_kt[NQT - 1];
        {
            const uint16_t* src = static_cast<const uint16_t*>(p.q) + ((size_t)(q0 + jr) * p.n_q_heads + hr) * D;
            const uint32_t qt = sQ + t * TILE;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint4 v = row_valid ? ldg_nc_128(src + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
                sts128(qt + (ch >> 3) * SLAB + swz128(r, ch & 7), v);
            }
            tc::fence_async_smem();
            mbar_arrive(bars + 8 * Q_FULL);
        }
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + (uint32_t)(t * BN);
        const uint32_t tO = tmem + lane_base + O_COL + (uint32_t)(t * D);
        const float sc = p.qk_scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nkt; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * (S_FULL + t), i & 1, p.err))) { ok = false; break; }
            tc::fence_after();
            const int kbase = i * BN;
            const bool masked = kbase + BN - 1 > lim_min;
            // pass 1: row max of this key tile (masked keys excluded)
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t raw[32];
                tc::ld32(tS + 32 * q, raw);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float v = __uint_as_float(raw[e]);
                    if (masked && kbase + 32 * q + e > lim) v = -INFINITY;
                    mx[e & 3] = fmaxf(mx[e & 3], v);
                }
            }
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
            float alpha = 1.f;
            bool rescale = false;
            if (m_ref == -INFINITY) {
                m_ref = mt;
            } else if (mt > m_ref + RESCALE_LOG2) {
                alpha = exp2f(m_ref - mt);
                m_ref = mt;
                rescale = true;
            }
            // O is settled here: this tile's S was issued after the previous PV, and the S
            // commit covers every earlier MMA of the issuing thread
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t o[32];
                    tc::ld32(tO + 32 * q, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::st32(tO + 32 * q, o);
                }
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            // pass 2: weights, written over the S piece just read as P_hi (16 columns) + P_lo (16)
            float ls[2] = {0.f, 0.f};
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t raw[32];
                tc::ld32(tS + 32 * q, raw);
                tc::wait_ld();
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float s0 = __uint_as_float(raw[2 * e]), s1 = __uint_as_float(raw[2 * e + 1]);
                    if (masked) {
                        if (kbase + 32 * q + 2 * e > lim) s0 = -INFINITY;
                        if (kbase + 32 * q + 2 * e + 1 > lim) s1 = -INFINITY;
                    }
                    const float a = exp2f(fmaf(s0, sc, -mu));
                    const float b = exp2f(fmaf(s1, sc, -mu));
                    hi[e] = F::pack_rn(a, b);
                    const float2 u = F::unpack(hi[e]);
                    lo[e] = F::pack_rn(a - u.x, b - u.y);
                    ls[e & 1] += a + b;
                }
                tc::st16(tS + 32 * q, hi);
                tc::st16(tS + 32 * q + 16, lo);
            }
            l = l * alpha + (ls[0] + ls[1]);
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bars + 8 * (P_FULL + t));
        }
        // epilogue: O / l -> out
        if (ok && nkt > 0 && __all_sync(0xffffffffu, mbar_wait(bars + 8 * (PV_DONE + t), (nkt - 1) & 1, p.err))) {
            tc::fence_after();
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            uint16_t* dst = static_cast<uint16_t*>(p.out) + ((size_t)(q0 + jr) * p.n_q_heads + hr) * D;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t o[32];
                tc::ld32(tO + 32 * q, o);
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
    } else if (warp == TMA_WARP) {
        // ------------------------------------------------------------ TMA producer warp
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_last();
        const int32_t* bt = p.block_tables + (size_t)c * p.max_blocks_per_seq;
        bool ok = true;
        for (int i = 0; i < n_max && ok; ++i) {
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
        // ------------------------------------------------------------ MMA warp
        constexpr uint32_t ID_QK = tc::idesc_f16(BF16, false, BM, BN);
        constexpr uint32_t ID_PV = tc::idesc_f16(BF16, true, BM, D);
        bool ok = __all_sync(0xffffffffu, mbar_wait(bars + 8 * Q_FULL, 0, p.err));
        int k_ready = -1, v_ready = -1, issued = 0;
        auto wait_k = [&](int jt) -> bool {
            if (jt <= k_ready) return true;
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * (K_FULL + (jt & 1)), (jt >> 1) & 1, p.err))) return false;
            k_ready = jt;
            return true;
        };
        auto wait_v = [&](int jt) -> bool {
            if (jt <= v_ready) return true;
            if (!__all_sync(0xffffffffu, mbar_wait(bars + 8 * (V_FULL + (jt & 1)), (jt >> 1) & 1, p.err))) return false;
            v_ready = jt;
            return true;
        };
        auto issue_s = [&](int t, int jt) {
            if (lane == 0) {
                const uint32_t q = sQ + t * TILE, k = sK + (jt & 1) * TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * SLAB + (kk & 3) * 32;
                    tc::mma_f16_ss(tmem + (uint32_t)(t * BN), tc::sdesc_sw128(q + off, 16, 1024),
                                   tc::sdesc_sw128(k + off, 16, 1024), ID_QK, kk > 0);
                }
                tc::commit(bars + 8 * (S_FULL + t));
            }
            ++issued;
        };
        auto issue_pv = [&](int t, int jt) {
            if (lane == 0) {
                const uint32_t v = sV + (jt & 1) * TILE;
                const uint32_t pS = tmem + (uint32_t)(t * BN);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // keys 16kk..16kk+15: P_hi at column 32(kk/2) + 8(kk%2) of S_t, P_lo 16 further
                    const uint32_t pc = (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1));
                    const uint64_t vd = tc::sdesc_sw128(v + kk * 2048, SLAB, 1024);
                    tc::mma_f16_ts(tmem + O_COL + (uint32_t)(t * D), pS + pc, vd, ID_PV, (jt > 0 || kk > 0));
                    tc::mma_f16_ts(tmem + O_COL + (uint32_t)(t * D), pS + pc + 16, vd, ID_PV, 1u);
                }
                tc::commit(bars + 8 * (PV_DONE + t));
            }
            ++issued;
        };
        if (ok) ok = wait_k(0);
        if (ok) {
            tc::fence_after();
#pragma unroll
            for (int t = 0; t < NQT; ++t)
                if (n_kt[t] > 0) issue_s(t, 0);
            if (lane == 0) tc::commit(bars + 8 * K_EMPTY);
            __syncwarp();
        }
        for (int i = 0; i < n_max && ok; ++i) {
            bool next_k = false;
            if (i == n_max - 1) {
                // rows of the sequence's last, partial block past kv_len may hold anything
                // (P is 0 there, but 0 * NaN is NaN): zero them in the last V tile
                ok = wait_v(i);
                if (!ok) break;
                const int z0 = max(kv_len, i * BN), z1 = min(((kv_len + 15) / 16) * 16, (i + 1) * BN);
                const int nz = z1 - z0;
                for (int e = lane; e < 16 * max(nz, 0); e += 32) {
                    const int row = z0 - i * BN + e / 16;
                    sts128(sV + (i & 1) * TILE + ((e / 8) & 1) * SLAB + row * 128 + (e & 7) * 16,
                           make_uint4(0u, 0u, 0u, 0u));
                }
                tc::fence_async_smem();
                __syncwarp();
            }
#pragma unroll
            for (int t = 0; t < NQT && ok; ++t) {
                if (i >= n_kt[t]) continue;
                ok = __all_sync(0xffffffffu, mbar_wait(bars + 8 * (P_FULL + t), i & 1, p.err)) && wait_v(i);
                if (!ok) break;
                tc::fence_after();
                issue_pv(t, i);
                if (i + 1 < n_kt[t]) {
                    ok = wait_k(i + 1);
                    if (!ok) break;
                    tc::fence_after();
                    issue_s(t, i + 1);
                    next_k = true;
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) {
                tc::commit(bars + 8 * (V_EMPTY + (i & 1)));
                if (next_k) tc::commit(bars + 8 * (K_EMPTY + ((i + 1) & 1)));
            }
            __syncwarp();
        }
        // every MMA this warp issued must be complete before TMEM is released
        if (issued > 0) {
            if (lane == 0) tc::commit(bars + 8 * DRAIN);
            __syncwarp();
            (void)mbar_wait(bars + 8 * DRAIN, 0, p.err);
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
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
    // one CTA per pair of 128-row query tiles of a (chunk, KV head)
    const int units = (p.tiles_per_chunk + pf::NQT - 1) / pf::NQT;
    PrefillParams q = p;
    q.tiles_per_chunk = units;
    const int grid = units * p.num_chunks * p.n_kv_heads;
    kern<<<grid, pf::THREADS, pf::SMEM_BYTES, st>>>(q, tmK, tmV);
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
