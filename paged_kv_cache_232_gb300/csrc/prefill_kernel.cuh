// prefill_kernel.cuh -- prefill-chunk attention over the paged cache on the tcgen05 tensor cores.
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
//    At head_dim 256 a CTA owns one query tile and streams K/V in stages of 64 keys (its O
//    accumulator takes 256 TMEM columns, and two stages of K and V must fit beside Q).
//  * Two producer warps (one for K, one for V) gather stages of 128 keys (64 at head_dim 256)
//    with one 4-D TMA load per 16-token chunk (or 8-token block) and 64-column slab, 128-byte
//    swizzled, into two-stage rings.
//    Block ids come from the chunk's block-table row; blocks past the sequence load zeros
//    (out-of-range block coordinate); the V producer zeroes the stray rows of the sequence's
//    last, partial block before it hands the last stage over.
//  * TMEM (512 columns): for each query tile t two 64-column S buffers at 128 t and the O
//    accumulator (head_dim columns) at 256 + head_dim t.  Keys are processed in 64-key
//    sub-tiles u: S_t(u) = Q_t K^T
//    (both operands from shared memory, K-major) lands in buffer u % 2, so the next
//    sub-tile's S is computed while the softmax works on this one; O_t += P_t(u) V reads the
//    weights from TMEM (the A operand) and V from shared memory (MN-major).
//  * One thread per query tile issues that tile's MMAs (warps 9 and 11): a wait on an mbarrier
//    costs the issuing thread a few hundred cycles even when the phase is complete (shared
//    memory is saturated by the operand reads), and with two issuers one tile's MMAs keep the
//    tensor pipe busy while the other issuer waits.
//  * Warpgroup t (warps 4t..4t+3; thread = query row = TMEM lane) reads its 64 S values,
//    applies the causal mask only on sub-tiles that reach past the tile's smallest row limit,
//    and keeps an online softmax in base 2 with a lazily updated integer reference max: O and l
//    are rescaled only when the row max grows by more than 2^8; otherwise weights up to 2^8 are
//    kept (exact in fp32, and the final O / l uses the same reference).  The PV operand is
//    16-bit, and one 16-bit weight costs up to 2^-9 relative -- too much next to the bf16
//    output rounding for a 2e-3 bound -- so each weight goes in as P_hi = round(p) plus
//    P_lo = round(p - P_hi) (about 16 significant bits together), both written over the S
//    columns just read, and the PV step issues one MMA for each half into the same fp32
//    accumulator.
//  * Every mbarrier wait has a time limit; on expiry the kernel flags PA_DEVERR_TIMEOUT, all
//    roles leave their loops, and the TMEM columns are released before exit.
#pragma once

#include "pa_launch.h"
#include "tcgen05.cuh"

namespace pa {
namespace pf {

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per unit of the scheduling cost
constexpr int NQT = 2;                  // query-tile roles per CTA (head_dim 256 uses one)
constexpr int BS = 64;                  // keys per S sub-tile
// barriers: K_FULL / V_FULL per ring stage; K_EMPTY / V_EMPTY, S_FULL and P_FULL per (query tile,
// buffer) at index 2 t + b; PV_DONE and DRAIN per query tile; V_ZERO once (last V stage cleaned)
enum Bar { Q_FULL = 0, K_FULL = 1, V_FULL = 3, K_EMPTY = 5, V_EMPTY = 9, S_FULL = 13, P_FULL = 17, PV_DONE = 21,
           DRAIN = 23, V_ZERO = 25, NUM_BARS = 26 };
static_assert(NUM_BARS <= 32, "barrier area");
constexpr int SCHED_BYTES = 24 * 1024;
// Shared-memory layout for head_dim D: a 16-bit tile of R rows x D columns is D / 64 slabs of
// R x 128 bytes.  head_dim 64 / 128: two query tiles per CTA and K/V stages of 128 keys (two S
// sub-tiles); head_dim 256: one query tile (its O takes 256 of the 512 TMEM columns) and stages
// of 64 keys (one sub-tile), so that two stages of K and of V still fit next to the Q tile.
template <int D>
struct Layout {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static constexpr int SLABS = D / 64;
    static constexpr int NQ = (D == 256) ? 1 : 2;       // query tiles per CTA
    static constexpr int SK = (D == 256) ? 64 : 128;    // keys per K/V stage
    static constexpr int SPS = SK / BS;                 // S sub-tiles per stage
    static constexpr int CHUNKS = SK / 16;              // 16-token chunks per stage
    static constexpr int QSLAB = BM * 128, KSLAB = SK * 128;
    static constexpr int QTILE = SLABS * QSLAB, KTILE = SLABS * KSLAB;
    static constexpr int Q_OFF = 0;                     // NQ tiles
    static constexpr int K_OFF = NQ * QTILE;            // two stages
    static constexpr int V_OFF = K_OFF + 2 * KTILE;     // two stages
    static constexpr int BAR_OFF = V_OFF + 2 * KTILE;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + 32 * 8;
    static constexpr int SCHED_OFF = TMEM_SLOT_OFF + 16;  // CTA-order scratch: query_start_loc, seq_lens, histogram
    static constexpr int SMEM_BYTES = SCHED_OFF + SCHED_BYTES + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};
// warpgroups 0..NQT-1: softmax (one per query tile); warpgroup NQT: K loads, MMA issue for tile 0,
// V loads, MMA issue for tile 1
static_assert(NQT == 2, "one MMA-issuing warp per query tile, two tiles");
constexpr int THREADS = (4 * NQT + 4) * 32;
constexpr int TMA_WARP = 4 * NQT, MMA_WARP = 4 * NQT + 1, TMA_V_WARP = 4 * NQT + 2, MMA_WARP_1 = 4 * NQT + 3;
// Register split: the launch gives every thread 168 (65536 / 384, rounded down to 8); the
// producer warpgroup drops to 88 and each softmax warpgroup rises to 208, so the totals match
// (128 x 88 + 256 x 208 = 384 x 168 = 64512) and every SMSP keeps 208 + 208 + 88 per lane.
constexpr int REGS_SOFTMAX = 208, REGS_PRODUCER = 88;
static_assert(NQT * 128 * REGS_SOFTMAX + 128 * REGS_PRODUCER <= THREADS * 168, "register split exceeds the launch");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;         // S_t buffers at columns 128 t + 64 b, O_t (D columns) at 256 + D t

}  // namespace pf

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Key tiles a unit (a pair of query tiles: tokens [j0, j0 + span) of chunk c) streams.
__device__ __forceinline__ int unit_cost(const int* qsl, const int* kvl, int c, int pair, int span, int cap,
                                         int max_q_len) {
    const int q_len = qsl[c + 1] - qsl[c], kv_len = kvl[c];
    const int j0 = pair * span;
    if (q_len < 0 || q_len > max_q_len || kv_len < q_len || kv_len > cap || j0 >= q_len) return 0;
    return (kv_len - q_len + min(j0 + span, q_len) + pf::BN - 1) / pf::BN;
}

// The unit this CTA runs under longest-first order: every CTA computes the same counting sort
// of all units by cost (descending, ties by unit index) and takes the entry at its blockIdx.
// Uses the CTA-order scratch in shared memory; all threads of the CTA must call it.
template <int SPAN>
__device__ __forceinline__ int lpt_unit(const PrefillParams& p, unsigned char* scratch) {
    const int C = p.num_chunks, per_unit = C * p.n_kv_heads;
    const int U = p.tiles_per_chunk * per_unit;
    const int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);
    const int ncost = cap / pf::BN + 2;
    int* qsl = reinterpret_cast<int*>(scratch);
    int* kvl = qsl + C + 1;
    int* hist = kvl + C;
    int* sel = hist + ncost;  // [0] bucket, [1] rank within the bucket, [2] chosen unit, [3..] warp counts
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int i = tid; i <= C; i += nt) qsl[i] = __ldg(p.query_start_loc + i);
    for (int i = tid; i < C; i += nt) kvl[i] = __ldg(p.seq_lens + i);
    for (int i = tid; i < ncost; i += nt) hist[i] = 0;
    __syncthreads();
    for (int u = tid; u < U; u += nt) {
        const int cst = min(unit_cost(qsl, kvl, (u / p.n_kv_heads) % C, u / per_unit, SPAN, cap, p.max_q_len), ncost - 1);
        atomicAdd(&hist[cst], 1);
    }
    __syncthreads();
    const int b = blockIdx.x;
    if (tid < 32) {
        // descending scan of the histogram; find the bucket holding position b
        int before = 0;
        for (int top = ncost - 1; top >= 0; top -= 32) {
            const int k = top - tid;
            const int v = (k >= 0) ? hist[k] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const int start = before + incl - v;
            if (v > 0 && b >= start && b < start + v) {
                sel[0] = k;
                sel[1] = b - start;
            }
            before += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    const int want = sel[0], rank = sel[1];
    // the rank-th unit (ascending index) whose cost is `want`
    int seen = 0;
    for (int base = 0; base < U; base += nt) {
        const int u = base + tid;
        const bool hit = u < U && min(unit_cost(qsl, kvl, (u / p.n_kv_heads) % C, u / per_unit, SPAN, cap, p.max_q_len),
                                      ncost - 1) == want;
        const unsigned bal = __ballot_sync(0xffffffffu, hit);
        if ((tid & 31) == 0) sel[3 + (tid >> 5)] = __popc(bal);
        __syncthreads();
        int off = seen;
        for (int w = 0; w < (tid >> 5); ++w) off += sel[3 + w];
        const int mine = off + __popc(bal & ((1u << (tid & 31)) - 1u));
        if (hit && mine == rank) sel[2] = u;
        int tot = 0;
        for (int w = 0; w < (nt + 31) / 32; ++w) tot += sel[3 + w];
        __syncthreads();
        seen += tot;
        if (seen > rank) break;
    }
    __syncthreads();
    const int chosen = sel[2];
    __syncthreads();
    return chosen;
}

// The whole warp waits for a phase through lane 0 alone (fewer shared-memory polls next to the
// tensor core's operand reads); __syncwarp orders the other lanes after lane 0's acquire.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned* err) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok;
}

// Words src[from], src[from + 2], ..., src[from + 30] into 16 TMEM columns at taddr.
__device__ __forceinline__ void tmem_store16_stride2(uint32_t taddr, const uint32_t (&src)[64], int from) {
    uint32_t v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = src[from + 2 * e];
    tc::st16(taddr, v);
}

// Online softmax for one 64-key S sub-tile (keys kbase .. kbase + 63) of this thread's row,
// read from TMEM at tSb; the weights go back over the same columns -- for each 32-key piece,
// P_hi (16 columns) then P_lo (16 columns) -- and l / m_ref are updated.  m_ref is an integer
// (log2 units), so every rescale is an exact power of two.  Weights may reach 2^8 above the
// reference; a sub-tile whose weights outgrow that is redone with a raised reference (S is
// still intact), after O -- complete through the previous sub-tile's PV -- is rescaled.
template <bool BF16, int D>
// pv_wait: O holds earlier PVs of this row's unit (the previous one must be complete before a
// rescale), pv_parity: the parity of that PV's PV_DONE phase.
__device__ __forceinline__ void softmax_sub64(const uint32_t tSb, const uint32_t tO, const bool masked, const int kbase,
                                              const int lim, const float sc, float& m_ref, float& l,
                                              const uint32_t pv_done, const bool pv_wait, const uint32_t pv_parity,
                                              unsigned* err) {
    using F = F16x2<BF16>;
    constexpr uint32_t kBits256 = BF16 ? 0x4380u : 0x5C00u;  // 2^8 as a packed 16-bit value
    // decided per warp: the branch holds warp-collective TMEM loads and stores
    bool redo = __any_sync(0xffffffffu, m_ref == -INFINITY);
#pragma unroll 1
    for (int attempt = 0; attempt < 2; ++attempt) {
        uint32_t r[64];
        tc::ld64(tSb, r);
        tc::wait_ld();
        if (masked) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
                if (kbase + e > lim) r[e] = __float_as_uint(-INFINITY);
        }
        if (redo) {
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 64; ++e) mx[e & 3] = fmaxf(mx[e & 3], __uint_as_float(r[e]));
            const float mt = ceilf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc);
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                m_ref = mt;
            } else if (mt > m_ref) {
                alpha = ex2(m_ref - mt);
                m_ref = mt;
            }
            l *= alpha;
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                // O must hold every PV before this sub-tile (and none after: its PV waits for
                // these weights)
                if (pv_wait) (void)warp_wait(pv_done, pv_parity, err);
                tc::fence_after();
#pragma unroll 1
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t o[16];
                    tc::ld16(tO + 16 * q, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::st16(tO + 16 * q, o);
                }
            }
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 sc2 = make_float2(sc, sc), nmu2 = make_float2(-mu, -mu);
        float2 ls = make_float2(0.f, 0.f);
        uint32_t pmax = 0;
        // in place: keys (2e, 2e+1) -> r[2e] = P_hi pair, r[2e+1] = P_lo pair
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float2 x = ffma2(make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), sc2, nmu2);
            const float2 w = make_float2(ex2(x.x), ex2(x.y));
            const uint32_t hi = F::pack_rn(w.x, w.y);
            const float2 d = fsub2(w, F::unpack(hi));
            r[2 * e] = hi;
            r[2 * e + 1] = F::pack_rn(d.x, d.y);
            ls = fadd2(ls, w);
            pmax = umax16x2(pmax, hi);
        }
        const uint32_t pm = (pmax & 0xFFFFu) > (pmax >> 16) ? (pmax & 0xFFFFu) : (pmax >> 16);
        if (attempt == 0 && __any_sync(0xffffffffu, pm > kBits256)) {
            redo = true;  // a row of this warp outgrew its reference by more than 2^8
            continue;
        }
        tmem_store16_stride2(tSb + 0, r, 0);    // keys  0..31: P_hi
        tmem_store16_stride2(tSb + 16, r, 1);   //              P_lo
        tmem_store16_stride2(tSb + 32, r, 32);  // keys 32..63: P_hi
        tmem_store16_stride2(tSb + 48, r, 33);  //              P_lo
        l += ls.x + ls.y;
        break;
    }
}

// PREFIX = false: prefill chunks (rows = a chunk's query tokens, keys = its cached context and
// itself, bottom-right causal).  PREFIX = true: the shared-prefix pass of a decode batch (rows =
// the sequences' decode queries, keys = one piece of the prefix all of them share, each row cut
// at its own context length), writing fp32 (m, l, o) partials that the decode merges.
// SMALL: units whose rows fit in 64 run M = 64 tiles (pa_prefill_chunk_small_m, the unified
// launch's A/B); instantiated separately, so that the other kernels carry none of its code.
template <int G, bool BF16, int D, bool PREFIX, bool SMALL = false>
__global__ void __launch_bounds__(pf::THREADS, 1)
prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using namespace pf;
    using L = Layout<D>;
    constexpr int SLABS = L::SLABS, NQ = L::NQ, SPS = L::SPS, SK = L::SK, CHUNKS = L::CHUNKS;
    constexpr int QSLAB = L::QSLAB, KSLAB = L::KSLAB, QTILE = L::QTILE, KTILE = L::KTILE;
    using F = F16x2<BF16>;
    constexpr int TQ = BM / G;  // query tokens per tile
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + L::Q_OFF, sK = sbase + L::K_OFF, sV = sbase + L::V_OFF;
    const uint32_t bars = sbase + L::BAR_OFF;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::TMEM_SLOT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int unit, c, g, q0, q_len, kv_len;
    int k0 = 0, piece = 0;  // shared-prefix mode: the piece and its first key
    // launched as a programmatic dependent of whatever kernel precedes it in the stream: nothing is
    // read before that kernel has completed (a no-op when it never signalled early)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (PREFIX) {
        // the suffix decode, launched as a programmatic dependent, may start now (its inputs are
        // complete: this grid has waited above); it reads these partials only after its own wait
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const int pairs = p.tiles_per_chunk;
        unit = (int)blockIdx.x % pairs;
        const int rest = (int)blockIdx.x / pairs;
        g = rest % p.n_kv_heads;
        piece = rest / p.n_kv_heads;
        c = 0;  // the prefix's block ids are row 0 of the table
        q0 = 0;
        q_len = p.num_seqs;
        k0 = piece * p.piece_tokens;
        // Keys [k0, kv_len): the piece, cut at the longest context among this CTA's sequences.
        // Keys past every row's context are neither streamed nor attended (they may hold anything;
        // below that cut every key belongs to some row's context, so it is finite).
        int* lmax = reinterpret_cast<int*>(smem + L::SCHED_OFF);
        if (threadIdx.x == 0) *lmax = 0;
        __syncthreads();
        const int s0 = unit * NQ * TQ, s1 = min(s0 + NQ * TQ, q_len);
        int mine = 0;
        for (int s = s0 + (int)threadIdx.x; s < s1; s += (int)blockDim.x) mine = max(mine, __ldg(p.context_lens + s));
        mine = __reduce_max_sync(0xffffffffu, mine);
        if (lane == 0 && mine > 0) atomicMax(lmax, mine);
        __syncthreads();
        kv_len = max(k0, min(min(k0 + p.piece_tokens, p.prefix_tokens), *lmax));
    } else {
        // Work unit u = (pair * C + chunk) * Hkv + head.  CTAs are dispatched in blockIdx order,
        // so handing out units longest-first gives longest-processing-time list scheduling.
        const int per_unit = p.num_chunks * p.n_kv_heads;
        int u_sel = (p.tiles_per_chunk - 1 - (int)(blockIdx.x / per_unit)) * per_unit + (int)(blockIdx.x % per_unit);
        if (p.lpt) u_sel = lpt_unit<TQ * NQ>(p, smem + L::SCHED_OFF);
        unit = u_sel / per_unit;
        const int rem = u_sel % per_unit;
        c = rem / p.n_kv_heads;
        g = rem % p.n_kv_heads;

        // the CTA-order step left query_start_loc and seq_lens in shared memory
        const int* sched = reinterpret_cast<const int*>(smem + L::SCHED_OFF);
        q0 = p.lpt ? sched[c] : __ldg(p.query_start_loc + c);
        q_len = (p.lpt ? sched[c + 1] : __ldg(p.query_start_loc + c + 1)) - q0;
        kv_len = p.lpt ? sched[p.num_chunks + 1 + c] : __ldg(p.seq_lens + c);
        // a chunk longer than max_q_len (which sized the grid) would leave rows past the grid unwritten:
        // it is flagged and skipped like the other bad lengths
        if (q_len < 0 || q_len > p.max_q_len || kv_len < q_len ||
            kv_len > table_row_tokens(p.max_blocks_per_seq, p.cpb_log2)) {
            if (unit == 0 && g == 0 && threadIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
            return;
        }
    }
    const int j0 = unit * NQ * TQ;
    if (j0 >= q_len) return;  // whole CTA: past the chunk
    const int ctx = kv_len - q_len;
    // small-M tile: a unit whose rows fit in 64 (a decode row of the unified launch is one token x G
    // heads) runs tile 0 as M = 64 MMAs, half the tensor work of a 128-row tile.  At M = 64 row r
    // of S, P and O sits in TMEM lane (r mod 16) + 32 (r / 16): lanes 0-15 of each warp's quarter.
    const bool small = SMALL && (q_len - j0) * G <= 64;
    int n_sub[NQT];           // 64-key S sub-tiles each query tile needs (0: tile past the chunk)
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
        const int jt = j0 + t * TQ;
        if constexpr (PREFIX)
            n_sub[t] = (t < NQ && jt < q_len) ? (kv_len - k0 + BS - 1) / BS : 0;
        else
            n_sub[t] = (t < NQ && jt < q_len) ? (ctx + min(jt + TQ, q_len) + BS - 1) / BS : 0;
    }
    const int nsub_max = n_sub[NQT - 1] > n_sub[0] ? n_sub[NQT - 1] : n_sub[0];
    const int n_max = (nsub_max + SPS - 1) / SPS;  // K/V stages to stream
    const int nblk_seq = (kv_len + 15) / 16;       // 16-token chunks holding keys below kv_len
    const int kc0 = k0 / 16;                       // the first chunk streamed (k0 is a multiple of 16)

    if (threadIdx.x == 0) {
        mbar_init(bars + 8 * Q_FULL, NQ * BM);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bars + 8 * (K_FULL + s), 1);
            mbar_init(bars + 8 * (V_FULL + s), 1);
            mbar_init(bars + 8 * (PV_DONE + s), 1);
            mbar_init(bars + 8 * (DRAIN + s), 1);
        }
        for (int s = 0; s < 4; ++s) {  // index 2 t + b
            mbar_init(bars + 8 * (K_EMPTY + s), 1);
            mbar_init(bars + 8 * (V_EMPTY + s), 1);
            mbar_init(bars + 8 * (S_FULL + s), 1);
            mbar_init(bars + 8 * (P_FULL + s), 4);  // one arrival per softmax warp
        }
        mbar_init(bars + 8 * V_ZERO, 1);
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
    if (warp < 4 * NQT)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_PRODUCER));

    if (warp < 4 * NQ) {
        // ------------------------------------------------------------ softmax warpgroups (with
        // one query tile per CTA the second warpgroup has no work)
        const int t = warp >> 2;                    // query tile of this warpgroup
        // row of the tile: the TMEM lane, or at M = 64 lanes 0-15 of each quarter (-1: no row)
        const int r = !small ? (int)(threadIdx.x & 127) : (lane < 16 ? 16 * (warp & 3) + lane : -1);
        const int rr = r < 0 ? 0 : r;
        const int jt0 = j0 + t * TQ;
        const int jr = jt0 + rr / G;
        const int hr = g * G + (rr % G);
        const bool row_valid = r >= 0 && jr < q_len;
        int lim, lim_min;  // keys <= lim are visible to this row; lim_min: smallest limit of the warp's rows
        if constexpr (PREFIX) {
            const int Ls = row_valid ? max(__ldg(p.context_lens + jr), 0) : 0;
            lim = min(Ls, kv_len) - 1;
            lim_min = __reduce_min_sync(0xffffffffu, lim);
        } else {
            lim = row_valid ? ctx + jr : -1;
            lim_min = ctx + jt0;  // the tile's smallest limit
        }
        const int nsub = (t == 0) ? n_sub[0] : n_sub[NQT - 1];
        {
            // Q tile t: warp w of the group copies rows 32w .. 32w+31, 32 / CPR rows per
            // instruction (consecutive rows are contiguous when G >= 2), each lane one 16-byte
            // chunk into its 128-byte-swizzled place
            constexpr int CPR = D / 8, RPI = 32 / CPR;  // chunks per row, rows per instruction
            constexpr int PASS = CPR < 16 ? CPR : 16;   // loads in flight per lane
            const uint32_t qt = sQ + t * QTILE;
            const int ch = lane % CPR;
#pragma unroll
            for (int i0 = 0; i0 < CPR; i0 += PASS) {
                uint4 v[PASS];
#pragma unroll
                for (int i = 0; i < PASS; ++i) {
                    const int R = (warp & 3) * 32 + RPI * (i0 + i) + lane / CPR;
                    const int tok = jt0 + R / G;
                    const uint16_t* src = static_cast<const uint16_t*>(p.q) +
                                          ((size_t)(q0 + tok) * p.n_q_heads + g * G + R % G) * p.hd + ch * 8;
                    v[i] = (tok < q_len && ch * 8 < p.hd) ? ldg_nc_128(src) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < PASS; ++i) {
                    const int R = (warp & 3) * 32 + RPI * (i0 + i) + lane / CPR;
                    sts128(qt + (ch >> 3) * QSLAB + swz128(R, ch & 7), v[i]);
                }
            }
            tc::fence_async_smem();
            if (small) {
                // M = 64: zero this warp's lanes of the tile's S buffers before the first QK (the
                // issuer waits for Q_FULL); the lanes without a row keep S = 0 from then on
                uint32_t z[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) z[i] = 0u;
                const uint32_t tSz = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(t * 128);
                tc::st64(tSz, z);
                tc::st64(tSz + 64, z);
                tc::wait_st();
                tc::fence_before();
            }
            mbar_arrive(bars + 8 * Q_FULL);
        }
        // this row's output, formed before the loop so that only the pointer stays live across it
        uint16_t* const dst = PREFIX ? nullptr
                                     : static_cast<uint16_t*>(p.out) + ((size_t)(q0 + jr) * p.n_q_heads + hr) * p.hd;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + (uint32_t)(t * 128);
        const uint32_t tO = tmem + lane_base + O_COL + (uint32_t)(t * D);
        const float sc = p.qk_scale_log2;
        // M = 64: a lane without a row sees S = 0 (its S columns are zeroed before the first QK and
        // it writes back zero weights) and keeps a reference of +inf, so its weights are 0 and it
        // never asks its warp for a max pass or a rescale
        float m_ref = (r < 0) ? INFINITY : -INFINITY, l = 0.f;
        bool ok = true;
        for (int u = 0; u < nsub; ++u) {
            const int b = u & 1;
            if (!warp_wait(bars + 8 * (S_FULL + 2 * t + b), (u >> 1) & 1, p.err)) {
                ok = false;
                break;
            }
            tc::fence_after();
            const int kbase = k0 + u * BS;
            softmax_sub64<BF16, D>(tS + (uint32_t)(b * BS), tO, kbase + BS - 1 > lim_min, kbase, lim, sc, m_ref, l,
                                bars + 8 * (PV_DONE + t), u > 0, (uint32_t)((u - 1) & 1), p.err);
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (P_FULL + 2 * t + b));
        }
        // epilogue: O / l -> out.  With two S buffers, PV_DONE may stand at any of three
        // phases here (S of the last sub-tile only implies the PV two before it), which one
        // parity bit cannot tell apart; DRAIN_t, committed once after this tile's last MMA,
        // completes exactly one phase.
        const bool drained = ok && nsub > 0 && warp_wait(bars + 8 * (DRAIN + t), 0, p.err);
        if constexpr (PREFIX) {
            // the row's partial for this piece: O / l (fp32, all D columns), the reference m_ref
            // (base 2) and l; a row that saw no key of the piece (or a tile without keys) writes
            // m = -inf, l = 0, o = 0, so that the merge never reads a stale partial
            const size_t pr = (size_t)(jr * p.n_q_heads + hr) * p.pf_parts + piece;
            float* const od = p.pf_o + pr * D;
            if (drained) {
                tc::fence_after();
                const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tc::ld32(tO + 32 * q, o);
                    tc::wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *reinterpret_cast<float4*>(od + 32 * q + 4 * v) =
                                make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                            __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
                    }
                }
            } else if (nsub == 0 && row_valid) {
                for (int q = 0; q < D / 4; ++q) *reinterpret_cast<float4*>(od + 4 * q) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (row_valid && (drained || nsub == 0)) {
                p.pf_m[pr] = drained ? m_ref : -INFINITY;
                p.pf_l[pr] = drained ? l : 0.f;
            }
        } else if (drained) {
            tc::fence_after();
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tc::ld32(tO + 32 * q, o);
                tc::wait_ld();
                if (row_valid && 32 * q < p.hd) {
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
    } else if (warp == TMA_WARP || warp == TMA_V_WARP) {
        // ------------------------------------------------------------ TMA producers: K (warp
        // TMA_WARP) and V (warp TMA_V_WARP) rings, issued by separate warps so that the two
        // tiles' box loads are in flight together.  Stage i (keys SK i .. SK i + SK - 1) reuses the
        // buffer of stage i - 2 once every query tile that read stage i - 2 has released it (tile t
        // reads stages 0 .. (n_sub[t] + SPS - 1) / SPS - 1).
        const int kv = (warp == TMA_V_WARP) ? 1 : 0;
        const CUtensorMap* map = kv ? &tmV : &tmK;
        if (lane == 0) tma_prefetch_desc(map);
        const uint64_t pol = l2_policy_evict_last();
        const int32_t* bt = p.block_tables + (size_t)c * p.max_blocks_per_seq;
        const uint32_t full0 = bars + 8 * (kv ? V_FULL : K_FULL), empty0 = bars + 8 * (kv ? V_EMPTY : K_EMPTY);
        const uint32_t dst_base = kv ? sV : sK;
        const bool half8 = p.cpb_log2 < 0;  // blocks of 8 tokens
        bool ok = true;
        for (int i = 0; i < n_max && ok; ++i) {
            const int st = i & 1;
            const uint32_t ph = (i >> 1) & 1;
            // 16-token chunk b: table entry b >> cpb_log2; blocks of 8 tokens: one entry per 8 rows
            int my = p.num_blocks;  // past the sequence (or invalid): out-of-range coordinate, zero fill
            const int ci = kc0 + i * CHUNKS;  // the stage's first chunk
            const int e = half8 ? 2 * ci + lane : (ci + lane % CHUNKS) >> p.cpb_log2;
            if (half8 ? (lane < 2 * CHUNKS && 8 * e < kv_len) : (lane < CHUNKS && ci + lane < nblk_seq)) {
                my = __ldg(bt + e);
                if (my < 0 || my >= p.num_blocks) {
                    if (kv == 0) flag_error(p.err, PA_DEVERR_BLOCK);
                    my = p.num_blocks;
                }
            }
            if (lane == 0 && i >= 2) {
#pragma unroll
                for (int t = 0; t < NQT; ++t)
                    if (ok && (i - 2) * SPS < n_sub[t]) ok = mbar_wait(empty0 + 8 * (2 * t + st), ph ^ 1, p.err);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const uint32_t full = full0 + 8 * st;
            const uint32_t dst0 = dst_base + st * KTILE;
            if (lane == 0) mbar_arrive_expect_tx(full, KTILE);
            __syncwarp();
            if (!half8) {
                // lanes 0 .. CHUNKS SLABS - 1 each issue one box: chunk lane % CHUNKS, slab lane / CHUNKS
                const int c16 = lane % CHUNKS, sl = lane / CHUNKS;
                const int blk = __shfl_sync(0xffffffffu, my, c16);
                const int row0 = ((ci + c16) & ((1 << p.cpb_log2) - 1)) * 16;  // chunk's first row
                if (lane < CHUNKS * SLABS)
                    tma_load_4d(dst0 + sl * KSLAB + c16 * 2048, map, sl * 64, g, row0, blk, full, pol);
            } else {
                // lanes 0 .. 2 CHUNKS SLABS - 1: 8-row block lane % (2 CHUNKS), slab lane / (2 CHUNKS)
                const int b8 = lane % (2 * CHUNKS), sl = lane / (2 * CHUNKS);
                const int blk = __shfl_sync(0xffffffffu, my, b8);
                if (lane < 2 * CHUNKS * SLABS)
                    tma_load_4d(dst0 + sl * KSLAB + b8 * 1024, map, sl * 64, g, 0, blk, full, pol);
            }
            if (kv == 1 && i == n_max - 1) {
                // Rows of the sequence's last, partial block past kv_len may hold anything (P
                // is 0 there, but 0 * NaN is NaN): once the last V stage has landed, zero them,
                // then release the stage to the MMA issuers through V_ZERO.
                if (lane == 0) ok = mbar_wait(full, ph, p.err);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                const int kb = k0 + i * SK;  // the stage's first key
                const int z0 = max(kv_len, kb), z1 = min(((kv_len + 15) / 16) * 16, kb + SK);
                constexpr int CPR = D / 8;  // 16-byte chunks per row
                for (int e = lane; e < CPR * max(z1 - z0, 0); e += 32) {
                    const int row = z0 - kb + e / CPR, chk = e % CPR;
                    sts128(dst0 + (chk >> 3) * KSLAB + row * 128 + (chk & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
                }
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + 8 * V_ZERO);
            }
        }
    } else if ((warp == MMA_WARP || warp == MMA_WARP_1) && lane == 0 && (warp == MMA_WARP ? n_sub[0] : n_sub[1]) > 0) {
        // ------------------------------------------------------------ MMA issue, one thread per
        // query tile.  A wait on an mbarrier costs the issuing thread a few hundred cycles even
        // when the phase is already complete, and the tensor pipe starves meanwhile; with one
        // issuer per tile, one tile's MMAs go out while the other issuer waits.
        const int t = (warp == MMA_WARP) ? 0 : 1;
        const int nst = (t == 0) ? n_sub[0] : n_sub[1];
        const uint32_t ID_QK = small ? tc::idesc_f16(BF16, false, 64, BS) : tc::idesc_f16(BF16, false, BM, BS);
        const uint32_t ID_PV = small ? tc::idesc_f16(BF16, true, 64, D) : tc::idesc_f16(BF16, true, BM, D);
        // descriptors of the tile bases as (low, high) words; a K-step adds its byte offset >> 4
        // to the start-address field in the low word (addresses stay below 256 KB: no carry)
        const uint64_t dq = tc::sdesc_sw128(sQ + t * QTILE, 16, 1024), dk = tc::sdesc_sw128(sK, 16, 1024);
        const uint64_t dv = tc::sdesc_sw128(sV, KSLAB, 1024);
        const uint32_t q_lo = (uint32_t)dq, q_hi = (uint32_t)(dq >> 32);
        const uint32_t k_lo = (uint32_t)dk, k_hi = (uint32_t)(dk >> 32);
        const uint32_t v_lo = (uint32_t)dv, v_hi = (uint32_t)(dv >> 32);
        const uint32_t dS0 = tmem + (uint32_t)(t * 128), dO = tmem + O_COL + (uint32_t)(t * D);
        bool ok = mbar_wait(bars + 8 * Q_FULL, 0, p.err);
        int k_ready = -1, v_ready = -1;
        bool issued = false;
        auto wait_k = [&](int j) -> bool {
            if (j <= k_ready) return true;
            if (!mbar_wait(bars + 8 * (K_FULL + (j & 1)), (j >> 1) & 1, p.err)) return false;
            k_ready = j;
            return true;
        };
        auto wait_v = [&](int j) -> bool {
            if (j <= v_ready) return true;
            // the last stage is handed over through V_ZERO once its stray rows are cleaned
            const bool w = (j == n_max - 1) ? mbar_wait(bars + 8 * V_ZERO, 0, p.err)
                                            : mbar_wait(bars + 8 * (V_FULL + (j & 1)), (j >> 1) & 1, p.err);
            if (!w) return false;
            v_ready = j;
            return true;
        };
        // S_t(v) = Q_t K^T for keys 64v .. 64v+63 (rows (v % SPS) * 64 of stage v / SPS), into buffer v & 1
        auto issue_s = [&](int v) -> bool {
            const int j = v / SPS;
            if (!wait_k(j)) return false;
            tc::fence_after();
            const uint32_t ka = k_lo + (uint32_t)(((j & 1) * KTILE + (v % SPS) * (BS * 128)) >> 4);
            const uint32_t dS = dS0 + (uint32_t)((v & 1) * BS);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                // K-step kk: 32 bytes into slab kk / 4 of the Q tile and of the K stage
                const uint32_t qo = (uint32_t)((((kk >> 2) * QSLAB) + (kk & 3) * 32) >> 4);
                const uint32_t ko = (uint32_t)((((kk >> 2) * KSLAB) + (kk & 3) * 32) >> 4);
                tc::mma_f16_ss_w(dS, q_lo + qo, q_hi, ka + ko, k_hi, ID_QK, kk > 0);
            }
            tc::commit(bars + 8 * (S_FULL + 2 * t + (v & 1)));
            issued = true;
            return true;
        };
        // O_t += P_t(u) V for keys 64u .. 64u+63 (P_hi and P_lo from the S buffer u & 1)
        auto issue_pv = [&](int u) -> bool {
            const int j = u / SPS;
            if (!wait_v(j)) return false;
            tc::fence_after();
            const uint32_t va = v_lo + (uint32_t)(((j & 1) * KTILE + (u % SPS) * (BS * 128)) >> 4);
            const uint32_t pS = dS0 + (uint32_t)((u & 1) * BS);
#pragma unroll
            for (int kk = 0; kk < BS / 16; ++kk) {
                // keys 16kk..16kk+15: P_hi at column 32(kk/2) + 8(kk%2) of the buffer, P_lo 16 further
                const uint32_t pc = (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1));
                const uint32_t vb = va + (uint32_t)((kk * 2048) >> 4);
                tc::mma_f16_ts_w(dO, pS + pc, vb, v_hi, ID_PV, (u > 0 || kk > 0));
                tc::mma_f16_ts_w(dO, pS + pc + 16, vb, v_hi, ID_PV, 1u);
            }
            tc::commit(bars + 8 * (PV_DONE + t));
            issued = true;
            return true;
        };
        // the last of this tile's sub-tiles that reads stage j
        auto stage_last = [&](int j) { return min(SPS * j + SPS - 1, nst - 1); };
        // prologue: both S buffers (a stage's K is released after the QK of its last sub-tile)
        for (int v = 0; v < 2 && v < nst && ok; ++v) {
            ok = issue_s(v);
            if (ok && v == stage_last(v / SPS)) tc::commit(bars + 8 * (K_EMPTY + 2 * t + ((v / SPS) & 1)));
        }
        for (int u = 0; u < nst && ok; ++u) {
            ok = mbar_wait(bars + 8 * (P_FULL + 2 * t + (u & 1)), (u >> 1) & 1, p.err) && issue_pv(u);
            if (ok && u + 2 < nst) ok = issue_s(u + 2);
            if (!ok) break;
            if (u == stage_last(u / SPS)) tc::commit(bars + 8 * (V_EMPTY + 2 * t + ((u / SPS) & 1)));
            const int v = u + 2;
            if (v < nst && v == stage_last(v / SPS)) tc::commit(bars + 8 * (K_EMPTY + 2 * t + ((v / SPS) & 1)));
        }
        // every MMA this thread issued must be complete before TMEM is released
        if (issued) {
            tc::commit(bars + 8 * (DRAIN + t));
            (void)mbar_wait(bars + 8 * (DRAIN + t), 0, p.err);
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
}


}  // namespace pa
