// decode.cuh -- paged decode attention for sm_103a.
//
// What is computed (mini_engine, "Custom CUDA kernels", paged decode attention v1/v2;
// MiniLLM Runtime, "Core class relationships"): for sequence s, query head h and KV head
// g = h / G, over tokens t of the work unit's range, each token translated through the
// block table (physical block block_tables[s][t / block_size], offset t % block_size),
//     out[s, h] = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m),  s_t = scale * q[s, h] . K_t.
//
// GB300 design (not the pages' sm_80 one):
//  * One CTA per work unit (s, g, piece).  A piece is the whole context (one-pass kernel)
//    or a run of `part_tokens` tokens (split-K).  All G query heads of the group are
//    handled by the CTA, so each K/V byte is fetched from HBM once.
//  * A producer warp streams the unit's 16-token blocks with TMA: one 4-D tensor-map
//    load per 128-byte column slab of the [16 rows x head_dim] K and V tiles, 128-byte
//    swizzled, into an NST-stage shared-memory ring guarded by full/empty mbarriers.
//    Block ids are read 32 at a time by the producer warp (block-table prefetch).
//  * Four consumer warps take whole blocks round-robin.  For q.K, 8 lanes split a
//    token's head_dim and 4 tokens run side by side; the 4*G partial dots are reduced
//    across the 8 lanes with a transpose-reduce (each shuffle halves the values a lane
//    keeps), so one lane ends with finished scores of a single head.  Online softmax
//    (running max m, sum l, base-2 exponent with log2(e) folded into q) uses shuffles
//    across the lanes of a head.  For P.V each lane owns 8 columns of head_dim for all G
//    heads and walks its tokens; probabilities come through a small per-warp buffer.
//  * At the end the four warps' (m, l, o) are merged in shared memory and the CTA
//    writes either the final row (rounded to nearest even) or its piece's (m, l, o) for
//    the reduce kernel.
//  * When the one-pass grid is longer than a wave of resident CTAs, CTAs take sequences
//    longest first (a counting sort of the lengths in every CTA); from two waves on, at
//    G <= 2, decode_kernel_persistent runs one CTA per resident slot over a unit list, the
//    producer streaming the next unit while the consumers merge this one.
#pragma once

#include "pa_device.cuh"

namespace pa {

struct DecodeParams {
    void* out;                 // [S, Hq, hd] T
    const void* q;             // [S, Hq, hd] T
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* ws_m;               // [S, Hq, P]   (split-K only)
    float* ws_l;               // [S, Hq, P]
    float* ws_o;               // [S, Hq, P, D]
    unsigned* err;
    int num_seqs, n_q_heads, n_kv_heads, max_blocks_per_seq;
    int part_tokens;           // 0: whole context in one CTA
    int max_parts;             // P (pieces per (s, g): the workspace stride)
    int cover_parts;           // pieces of part_tokens that cover the longest context (the length clamp)
    int tail_tokens;           // decode_kernel_dyn only: > 0 splits each sequence's last part_tokens
                               // into pieces of this many tokens (pieces_of); 0: pieces of part_tokens
    int num_blocks;
    int cpb_log2;              // log2 of the 16-token chunks per cache block; -1: blocks of 8 tokens
    float qk_scale_log2;       // scale * log2(e)
    int hd;                    // head_dim of q, out and the cache (<= D; columns hd .. D-1 are zero)
    int lpt;                   // one-pass grid only: CTAs take sequences longest first
    int persist;               // one-pass grid only: decode_kernel_persistent, gridDim.x CTAs run unit lists
    // Shared prefix: tokens [0, prefix_tokens) of every sequence were attended by the shared-prefix
    // pass (prefill kernel in shared-prefix mode), which left pf_parts partials per (s, h): pf_m (base-2
    // log of the weights' reference), pf_l (their sum), pf_o (normalised output, D columns).  The
    // kernels here cover tokens [prefix_tokens, L) and fold those partials into their merge, after
    // griddepcontrol.wait (they are launched as programmatic dependents of that pass).
    int prefix_tokens;
    int pf_parts;              // 0: no shared prefix
    int dyn;                   // decode_kernel_dyn: gridDim.x CTAs taking pieces from *dyn_counter (split-K, or
                               // whole units, longest first, when dyn_units)
    int dyn_units;             // decode_kernel_dyn over whole units (one piece each, written directly)
    int* dyn_counter;          // the next piece to hand out
    // non-null: the counter is valid only while *dyn_tag == kDynTag, which the split-K merge
    // restores at its end (counter 0, tag set) for the next call; with another value the CTAs
    // take the pieces in a fixed order.  Null: the counter was zeroed before the launch.
    unsigned long long* dyn_tag;
    const float* pf_m;         // [S * Hq][pf_parts]
    const float* pf_l;
    const float* pf_o;         // [S * Hq][pf_parts][D]
    // pa_decode_write on the persistent and the dynamic grids: sequence s's new K and V rows
    // (new_k / new_v row s, row_vecs 16-byte chunks over all KV heads) go into slot new_slots[s] of
    // the cache (-1: none), head g's part by the CTA that decodes the last chunk of (s, g) -- the
    // one holding token context_lens[s] - 1, the slot's token -- before it loads that chunk.
    // new_k null: no write.
    const uint4* new_k;
    const uint4* new_v;
    const int64_t* new_slots;
    uint4* k_cache_w;
    uint4* v_cache_w;
    int row_vecs;
    long long n_slots;         // num_blocks * block_size
};

// The dynamic grid's "counter is at zero" mark in the workspace's control region: the bit
// patterns of two quiet NaNs, which no float the kernels store there takes.
constexpr unsigned long long kDynTag = 0x7FC0A5177FC02C32ull;

// Tokens of a sequence of context L the decode kernels stream: the part past the shared prefix.
__device__ __forceinline__ int streamed_tokens(const DecodeParams& p, int L) { return max(L - p.prefix_tokens, 0); }

// Split-K pieces of a sequence with L (clamped) tokens.  Uniform: pieces of part_tokens.  With
// tail_tokens (the dynamic grid): every piece but the last part_tokens-sized stretch is full, and
// that stretch (1 .. part_tokens tokens) goes in pieces of tail_tokens, so the items handed out
// last are short.  0 pieces: nothing streamed.
__device__ __forceinline__ int full_pieces_of(const DecodeParams& p, int Ls) {
    return Ls > 0 ? (Ls + p.part_tokens - 1) / p.part_tokens - 1 : 0;
}
__device__ __forceinline__ int pieces_of(const DecodeParams& p, int L) {
    const int Ls = streamed_tokens(p, L);
    if (p.tail_tokens == 0) return (Ls + p.part_tokens - 1) / p.part_tokens;
    if (Ls == 0) return 0;
    const int f = full_pieces_of(p, Ls);
    return f + (Ls - f * p.part_tokens + p.tail_tokens - 1) / p.tail_tokens;
}

// Folds the shared-prefix partials of output row `row` into a merge in progress: raises the
// running maximum M (base 2) first (prefix_max), then adds each partial's weight l_k 2^(m_k - M)
// to the sum and its output (normalised) times that weight (prefix_add).  Partials with l = 0 (no
// key of the piece visible) are skipped.  Up to kPfFast pieces, prefix_load reads all of a row's
// l, m and output pair at once beforehand (one round trip to L2 for the fold, not two per piece);
// with more pieces the two passes read them piece by piece.  Same arithmetic either way.
constexpr int kPfFast = 4;
struct PrefixRow {
    int n;  // pieces held; 0: read piece by piece
    float l[kPfFast], m[kPfFast];
    float2 o[kPfFast];
};
__device__ __forceinline__ void prefix_load(const DecodeParams& p, size_t row, int d, int D, PrefixRow& r) {
    r.n = p.pf_parts <= kPfFast ? p.pf_parts : 0;
#pragma unroll
    for (int k = 0; k < kPfFast; ++k)
        if (k < r.n) {
            const size_t i = row * p.pf_parts + k;
            r.l[k] = p.pf_l[i];
            r.m[k] = p.pf_m[i];
            r.o[k] = *reinterpret_cast<const float2*>(p.pf_o + i * D + d);
        }
}
__device__ __forceinline__ float prefix_max(const DecodeParams& p, const PrefixRow& r, size_t row, float M) {
    if (r.n > 0) {
#pragma unroll
        for (int k = 0; k < kPfFast; ++k)
            if (k < r.n && r.l[k] > 0.f) M = fmaxf(M, r.m[k]);
        return M;
    }
    for (int k = 0; k < p.pf_parts; ++k)
        if (p.pf_l[row * p.pf_parts + k] > 0.f) M = fmaxf(M, p.pf_m[row * p.pf_parts + k]);
    return M;
}
__device__ __forceinline__ void prefix_add(const DecodeParams& p, const PrefixRow& r, size_t row, int d, int D,
                                           float M, float& Lsum, float& o0, float& o1) {
    if (r.n > 0) {
#pragma unroll
        for (int k = 0; k < kPfFast; ++k)
            if (k < r.n && r.l[k] > 0.f) {
                const float wt = r.l[k] * ex2(r.m[k] - M);
                Lsum += wt;
                o0 = fmaf(r.o[k].x, wt, o0);
                o1 = fmaf(r.o[k].y, wt, o1);
            }
        return;
    }
    for (int k = 0; k < p.pf_parts; ++k) {
        const size_t i = row * p.pf_parts + k;
        const float lk = p.pf_l[i];
        if (lk > 0.f) {
            const float wt = lk * ex2(p.pf_m[i] - M);
            Lsum += wt;
            const float2 v = *reinterpret_cast<const float2*>(p.pf_o + i * D + d);
            o0 = fmaf(v.x, wt, o0);
            o1 = fmaf(v.y, wt, o1);
        }
    }
}

// Longest-first order of the one-pass grid: sequences ranked by 16-token chunk count
// (descending, ties by index); CTA b takes KV head b mod Hkv of the sequence at rank b / Hkv,
// so the hardware's in-order CTA dispatch becomes longest-processing-time list scheduling and
// the short sequences fill in behind.  Every CTA ranks the same lengths the same way.  scratch
// (ints, S + cap/16 + 2 of them) is shared memory nothing else uses yet; all threads call this;
// the result is valid in warp 0.
__device__ __forceinline__ int seq_at_rank(const DecodeParams& p, int r, int* scratch) {
    const int S = p.num_seqs, tid = threadIdx.x, lane = tid & 31;
    const int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);
    const int nb = (cap + 15) / 16 + 1;
    int* len = scratch;    // chunk count per sequence
    int* hist = scratch + S;
    for (int i = tid; i < nb; i += blockDim.x) hist[i] = 0;
    for (int i = tid; i < S; i += blockDim.x) {
        int L = __ldg(p.context_lens + i);
        L = L < 0 ? 0 : min(L, cap);
        len[i] = (streamed_tokens(p, L) + 15) >> 4;
    }
    __syncthreads();
    for (int i = tid; i < S; i += blockDim.x) atomicAdd(&hist[len[i]], 1);
    __syncthreads();
    if (tid >= 32) return 0;
    // descending scan of the histogram: the chunk count holding rank r, and r's rank inside it
    int want = 0, rank = 0, before = 0;
    for (int top = nb - 1; top >= 0; top -= 32) {
        const int k = top - lane;
        const int v = (k >= 0) ? hist[k] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int start = before + incl - v;
        const unsigned found = __ballot_sync(0xffffffffu, v > 0 && r >= start && r < start + v);
        if (found) {
            const int src = __ffs(found) - 1;
            want = __shfl_sync(0xffffffffu, k, src);
            rank = r - __shfl_sync(0xffffffffu, start, src);
            break;
        }
        before += __shfl_sync(0xffffffffu, incl, 31);
    }
    // the rank-th sequence (ascending index) with that chunk count
    int seen = 0;
    for (int base = 0; base < S; base += 32) {
        const int i = base + lane;
        const bool hit = i < S && len[i] == want;
        const unsigned bal = __ballot_sync(0xffffffffu, hit);
        const int n = __popc(bal);
        if (seen + n > rank) {
            const unsigned mine = __ballot_sync(0xffffffffu, hit && __popc(bal & ((1u << lane) - 1u)) == rank - seen);
            return base + __ffs(mine) - 1;
        }
        seen += n;
    }
    return 0;  // not reached: r < S
}

// The persistent grid's unit lists: the (sequence, KV head) units ranked as in seq_at_rank
// (unit rank r = sequence rank r / Hkv, KV head r mod Hkv); CTA c of P takes ranks
// c, 2P - 1 - c, 2P + c, 4P - 1 - c, ... (a snake over the longest-first order, so that every
// CTA's list sums to about the same length).  scratch (ints, 2 S + 2 (cap/16 + 1) of them) is
// shared memory nothing else uses yet; all threads call this; list gets (seq, KV head, 0) per
// unit; returns the count (valid in thread 0).
__device__ __forceinline__ int lpt_units(const DecodeParams& p, int* scratch, int* list, int list_max) {
    const int S = p.num_seqs, tid = threadIdx.x, lane = tid & 31;
    const int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);
    const int nb = (cap + 15) / 16 + 1;
    int* len = scratch;        // chunk count per sequence
    int* hist = len + S;       // sequences per chunk count
    int* start = hist + nb;    // first rank of each chunk count
    int* order = start + nb;   // sequence at each rank
    for (int i = tid; i < nb; i += blockDim.x) hist[i] = 0;
    for (int i = tid; i < S; i += blockDim.x) {
        int L = __ldg(p.context_lens + i);
        L = L < 0 ? 0 : min(L, cap);
        len[i] = (streamed_tokens(p, L) + 15) >> 4;
    }
    __syncthreads();
    for (int i = tid; i < S; i += blockDim.x) atomicAdd(&hist[len[i]], 1);
    __syncthreads();
    if (tid < 32) {
        // descending exclusive scan: start[k] = sequences with more than k chunks
        int before = 0;
        for (int top = nb - 1; top >= 0; top -= 32) {
            const int k = top - lane;
            const int v = (k >= 0) ? hist[k] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (k >= 0) start[k] = before + incl - v;
            before += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        // stable placement in index order, 32 sequences at a time
        for (int base = 0; base < S; base += 32) {
            const int i = base + lane;
            const int key = i < S ? len[i] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, key);
            if (i < S) order[start[key] + __popc(same & ((1u << lane) - 1u))] = i;
            __syncwarp();
            if (i < S && lane == __ffs(same) - 1) start[key] += __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
    int n = 0;
    if (tid == 0) {
        const int P = (int)gridDim.x, c = (int)blockIdx.x, units = S * p.n_kv_heads;
        for (int k = 0; n < list_max; ++k) {
            const int r = k * P + ((k & 1) ? P - 1 - c : c);
            if (r >= units) break;
            list[3 * n] = order[r / p.n_kv_heads];
            list[3 * n + 1] = r % p.n_kv_heads;
            list[3 * n + 2] = 0;
            ++n;
        }
    }
    return n;
}

template <int D, int G, bool BF16>
struct DecodeCfg {
    static constexpr int BS = 16;
    static constexpr int HALVES = D / 64;             // 128-byte column slabs per row
    static constexpr int SLAB_BYTES = BS * 128;       // one slab of one block tile
    static constexpr int TILE_BYTES = HALVES * SLAB_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile + V tile
    static constexpr int NST = (D == 256) ? 4 : (D == 128) ? 8 : 16;  // 64 KB of K/V in flight
    static constexpr int NCW = 4;                     // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int CPL = HALVES;                // 16-byte chunks per lane for q.K
    static constexpr int NV = 4 * G;                  // partial dots per lane before reduction
    static constexpr int R = (NV >= 8) ? NV / 8 : 1;  // finished scores per lane
    static constexpr int CR = D / 8;                  // 16-byte chunks per row
    static constexpr int TGP = 32 / CR;               // token groups for P.V
    static constexpr int TPL = BS / TGP;              // tokens per lane for P.V
    // shared memory: ring | p buffers | alpha | barriers
    static constexpr int RING_BYTES = NST * STAGE_BYTES;
    static constexpr int P_BYTES = NCW * BS * G * 4;
    static constexpr int A_BYTES = NCW * 8 * 4;
    static constexpr int MERGE_BYTES = NCW * (G * D + 2 * G) * 4;  // aliases the ring
    static constexpr int BAR_OFF = RING_BYTES + P_BYTES + A_BYTES;
    static constexpr int SLOT_OFF = BAR_OFF + 2 * NST * 8;           // the sequence picked by the order step
    static constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;           // + alignment slack
    static_assert(MERGE_BYTES <= RING_BYTES, "merge area must fit in the ring");
    // decode_kernel_persistent: ring | p buffers | alpha | merge area (the ring keeps streaming the
    // next unit during a merge) | barriers | unit list | flags
    static constexpr int P_MERGE_OFF = RING_BYTES + P_BYTES + A_BYTES;
    static constexpr int P_BAR_OFF = P_MERGE_OFF + MERGE_BYTES;
    static constexpr int LIST_MAX = 32;                                 // units one persistent CTA may run
    static constexpr int P_LIST_OFF = P_BAR_OFF + 2 * NST * 8;          // [LIST_MAX][3] (seq, KV head, 0)
    static constexpr int P_FLAG_OFF = P_LIST_OFF + LIST_MAX * 3 * 4;    // unit count, abort flag
    static constexpr int P_SMEM_BYTES = P_FLAG_OFF + 16 + 1024;
    // decode_kernel_dyn: the persistent layout, then (with tail pieces) per sequence of a batch of
    // up to DYN_SMAX: the clamped length, running counts of full and of tail pieces
    static constexpr int DYN_SMAX = 256;
    static constexpr int D_LEN_OFF = P_FLAG_OFF + 16;
    static constexpr int D_CUMA_OFF = D_LEN_OFF + DYN_SMAX * 4;
    static constexpr int D_CUMB_OFF = D_CUMA_OFF + (DYN_SMAX + 1) * 4;
    static constexpr int D_SMEM_BYTES = D_CUMB_OFF + (DYN_SMAX + 1) * 4 + 1024;
    // Consumer warp w takes blocks b = w, w + NCW, ...; with NST a multiple of NCW every ring stage
    // belongs to one warp, which waits on its phases in order -- a stage's full barrier is then
    // never two phases behind the phase its warp waits for (where the parity test would pass early).
    static_assert(NST % NCW == 0, "ring stages must be a multiple of the consumer warps");
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static_assert(D != 256 || G <= 4, "head_dim 256: group size 1, 2 or 4 (q takes 32 G registers)");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size 1, 2, 4 or 8");
};

// One step of the transpose-reduce: the lane keeps half of its N values (the upper half if
// `bit` is set in its lane id) and adds the partner's copy of the same half.
template <int N>
__device__ __forceinline__ void tr_step(float* v, int lane, int bit) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        float send = up ? v[k] : v[k + N / 2];
        float keep = up ? v[k + N / 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
}

// Reduce the 4*G partial dots over the 8 lanes that share a token (lane bits 0..2).
// Afterwards the lane holds R finished dots with flat indices base + k (index = h*4 + i).
template <int G>
__device__ __forceinline__ int transpose_reduce(float* v, int lane) {
    constexpr int N0 = 4 * G;
    int base = 0;
    if constexpr (N0 >= 2) { tr_step<N0>(v, lane, 4); base += (lane & 4) ? N0 / 2 : 0; }
    if constexpr (N0 / 2 >= 2) { tr_step<N0 / 2>(v, lane, 2); base += (lane & 2) ? N0 / 4 : 0; }
    if constexpr (N0 / 4 >= 2) {
        tr_step<N0 / 4>(v, lane, 1);
        base += (lane & 1) ? N0 / 8 : 0;
    } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);  // G == 1: both lanes end with the same sum
    }
    return base;
}

// xor-masks over which the lanes holding one head's scores are spread (tg bits 3,4 plus
// the dl bits that do not encode the head).  For sums, G == 1 skips bit 0 (duplicates).
template <int G>
__device__ __forceinline__ float head_max(float x) {
    if constexpr (G <= 4) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
    if constexpr (G <= 2) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
    if constexpr (G == 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
    return x;
}

template <int G>
__device__ __forceinline__ float head_sum(float x) {
    if constexpr (G == 2 || G == 4) x += __shfl_xor_sync(0xffffffffu, x, 1);
    if constexpr (G <= 2) x += __shfl_xor_sync(0xffffffffu, x, 2);
    if constexpr (G == 1) x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

// One 16-token chunk of K and V (the ring stage at kt, nvalid tokens valid): q.K for the G
// heads, the online-softmax update of (m_run, l_run) and o, and P.V into o.  Shared by the three
// decode kernels; the caller waits for the stage and releases it.  PACKED: the products on packed
// fp32 pairs (fma.rn.f32x2, half the FMA instructions: q.K sums the even and the odd columns of a
// 16-byte chunk apart and adds the two at the end; P.V updates two columns per instruction).
// GB300: 4 x 32K tokens at 32 q / 8 KV heads 104.4 -> 96.2 us, 64 x U[100,2048] at 16 / 8 heads
// 53.8 -> 53.2; the persistent one-pass grid (batch 256) keeps the scalar form (164.9 against
// 166.3 us packed).
template <int D, int G, bool BF16, bool PACKED = true>
__device__ __forceinline__ void consume_chunk(const uint32_t kt, const int nvalid,
                                              const float (&qf)[G][DecodeCfg<D, G, BF16>::CPL][8],
                                              const int (&chunk_col)[DecodeCfg<D, G, BF16>::CPL], const int lane,
                                              const int my_h, const bool rep, float* pw, float* aw, float& m_run,
                                              float& l_run, float (&o)[G][8]) {
    using C = DecodeCfg<D, G, BF16>;
    const int tg = lane >> 3;
    const int dg = lane % C::CR, tgp = lane / C::CR;  // P.V layout
    const uint32_t vt = kt + C::TILE_BYTES;

    // ---- q.K: 4 tokens x G heads of partial dots per lane
    float acc[4 * G];
#pragma unroll
    for (int k = 0; k < 4 * G; ++k) acc[k] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = tg + 4 * i;
        float2 a2[G];  // PACKED: the even and the odd columns apart, added at the end
#pragma unroll
        for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < C::CPL; ++j) {
            const int half = chunk_col[j] >> 6, c = (chunk_col[j] >> 3) & 7;
            const uint4 raw = lds128(kt + half * C::SLAB_BYTES + swz128(t, c));
            if constexpr (PACKED) {
                const float2 k0 = F16x2<BF16>::unpack(raw.x), k1 = F16x2<BF16>::unpack(raw.y);
                const float2 k2 = F16x2<BF16>::unpack(raw.z), k3 = F16x2<BF16>::unpack(raw.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    a2[h] = ffma2(make_float2(qf[h][j][0], qf[h][j][1]), k0, a2[h]);
                    a2[h] = ffma2(make_float2(qf[h][j][2], qf[h][j][3]), k1, a2[h]);
                    a2[h] = ffma2(make_float2(qf[h][j][4], qf[h][j][5]), k2, a2[h]);
                    a2[h] = ffma2(make_float2(qf[h][j][6], qf[h][j][7]), k3, a2[h]);
                }
            } else {
                float kf[8];
                unpack8<BF16>(raw, kf);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[h * 4 + i] = fmaf(qf[h][j][e], kf[e], acc[h * 4 + i]);
            }
        }
        if constexpr (PACKED) {
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h * 4 + i] = a2[h].x + a2[h].y;
        }
    }
    const int base = transpose_reduce<G>(acc, lane);

    // ---- online softmax for this lane's head over the block's 16 tokens
    float sc[C::R];
    float bmax = -INFINITY;
#pragma unroll
    for (int r = 0; r < C::R; ++r) {
        const int i = (base + r) & 3;
        const int t = tg + 4 * i;
        sc[r] = (t < nvalid) ? acc[r] : -INFINITY;
        bmax = fmaxf(bmax, sc[r]);
    }
    bmax = head_max<G>(bmax);
    const float m_new = fmaxf(m_run, bmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int r = 0; r < C::R; ++r) {
        const int i = (base + r) & 3;
        const int t = tg + 4 * i;
        const float pr = (m_new == -INFINITY) ? 0.f : ex2(sc[r] - m_new);
        psum += pr;
        if (G > 1 || (lane & 1) == 0) pw[t * G + my_h] = pr;
    }
    psum = head_sum<G>(psum);
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (rep) aw[my_h] = alpha;
    __syncwarp();

    // ---- P.V: this lane's 8 columns for all G heads, its TPL tokens
    bool rescale = false;
    float al[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        al[h] = aw[h];
        rescale |= (al[h] != 1.f);
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] *= al[h];
    }
    const int half = dg >> 3, c = dg & 7;
#pragma unroll
    for (int i = 0; i < C::TPL; ++i) {
        const int t = tgp + C::TGP * i;
        if (t < nvalid) {
            const uint4 raw = lds128(vt + half * C::SLAB_BYTES + swz128(t, c));
            if constexpr (PACKED) {
                const float2 v0 = F16x2<BF16>::unpack(raw.x), v1 = F16x2<BF16>::unpack(raw.y);
                const float2 v2 = F16x2<BF16>::unpack(raw.z), v3 = F16x2<BF16>::unpack(raw.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pr = pw[t * G + h];
                    const float2 p2 = make_float2(pr, pr);
                    const float2 r0 = ffma2(p2, v0, make_float2(o[h][0], o[h][1]));
                    const float2 r1 = ffma2(p2, v1, make_float2(o[h][2], o[h][3]));
                    const float2 r2 = ffma2(p2, v2, make_float2(o[h][4], o[h][5]));
                    const float2 r3 = ffma2(p2, v3, make_float2(o[h][6], o[h][7]));
                    o[h][0] = r0.x; o[h][1] = r0.y; o[h][2] = r1.x; o[h][3] = r1.y;
                    o[h][4] = r2.x; o[h][5] = r2.y; o[h][6] = r3.x; o[h][7] = r3.y;
                }
            } else {
                float vf[8];
                unpack8<BF16>(raw, vf);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pr = pw[t * G + h];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pr, vf[e], o[h][e]);
                }
            }
        }
    }
}

// Resident CTAs per SM the register allocation must allow: shared memory fits three; G <= 4
// fits in the resulting 136 registers without spills (G = 4 would otherwise take ~150 and lose
// a third of the warps); G = 8 at head_dim 64 fits two, at head_dim 128 only one without spills.
template <int D, int G, bool BF16>
__global__ void __launch_bounds__(DecodeCfg<D, G, BF16>::THREADS,
                                  D == 256 ? (G <= 2 ? 2 : 1) : ((G <= 4) ? 3 : (D == 64 ? 2 : 1)))
decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using C = DecodeCfg<D, G, BF16>;
    using F = F16x2<BF16>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern of TMA
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_addr(smem);
    float* p_buf = reinterpret_cast<float*>(smem + C::RING_BYTES);
    float* a_buf = reinterpret_cast<float*>(smem + C::RING_BYTES + C::P_BYTES);
    const uint32_t bar_full = ring + C::BAR_OFF;
    const uint32_t bar_empty = bar_full + C::NST * 8;

    // launched as a programmatic dependent of whatever kernel precedes it in the stream: nothing is
    // read before that kernel has completed (a no-op when it never signalled early); after a
    // shared-prefix pass, which waited itself before letting this grid launch, only the merge waits
    if (p.pf_parts == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.num_seqs * p.n_kv_heads;
    // split-K: the grid runs the highest piece index first -- only long contexts have one -- so the
    // extra pieces of long sequences start at once and the short, whole-sequence pieces fill in
    // behind them (longest-first without knowing the lengths on the host)
    const int qpos = (int)(blockIdx.x / units);
    const int piece = (p.max_parts - 1) - qpos;
    int s, g;
    if (p.lpt) {
        volatile int* slot = reinterpret_cast<volatile int*>(smem + C::SLOT_OFF);
        const int r = (int)blockIdx.x / p.n_kv_heads;
        const int picked = seq_at_rank(p, r, reinterpret_cast<int*>(smem));
        if (threadIdx.x == 0) *slot = picked;
        fence_proxy_async_smem();  // the scratch (ring) is written by TMA next
        __syncthreads();
        s = *slot;
        g = (int)blockIdx.x - r * p.n_kv_heads;
    } else {
        const int sg = (int)blockIdx.x - qpos * units;
        s = sg / p.n_kv_heads;
        g = sg - s * p.n_kv_heads;
    }

    // a CTA over a whole context from its first token (one pass, no shared prefix, blocks of 16
    // tokens or more): the producer loads the first table entries at once, next to the context
    // length instead of after it (one dependent memory latency less before the first K/V tile)
    const bool spec = p.part_tokens == 0 && p.prefix_tokens == 0 && p.cpb_log2 >= 0;
    int spec_blk = 0;
    if (spec && warp == C::NCW && (lane >> p.cpb_log2) < p.max_blocks_per_seq)
        spec_blk = __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + (lane >> p.cpb_log2));
    // context length, clamped to what the table (and the split-K grid) can address
    int L = __ldg(p.context_lens + s);
    int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);  // tokens the table row addresses
    if (p.part_tokens > 0 && p.prefix_tokens + p.cover_parts * p.part_tokens < cap)
        cap = p.prefix_tokens + p.cover_parts * p.part_tokens;
    if (L < 0 || L > cap) {
        if (piece == 0 && g == 0 && threadIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
        L = L < 0 ? 0 : cap;
    }
    // tokens [base, L) are streamed here (base > 0 past a shared prefix), in pieces for split-K
    const int base = min(L, p.prefix_tokens);
    const int t_begin = p.part_tokens > 0 ? min(L, base + piece * p.part_tokens) : base;
    const int t_end = p.part_tokens > 0 ? min(L, t_begin + p.part_tokens) : L;
    const int n_parts = p.part_tokens > 0 ? (L - base + p.part_tokens - 1) / p.part_tokens : 1;
    if (t_begin >= t_end && piece > 0) return;  // split-K piece past this sequence's context
    const int nblk = (t_end - t_begin + C::BS - 1) / C::BS;
    const int blk0 = t_begin / C::BS;
    const bool direct = (n_parts <= 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == C::NCW) {
        // ------------------------------------------------------------ producer warp
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_first();
        // 16-token chunk c of the sequence: table entry c >> cpb_log2, rows 16 (c mod 2^cpb_log2) + 0..15;
        // with blocks of 8 tokens, entries 2c and 2c + 1 (the second only if the context reaches it),
        // each an 8-row box, the second landing 8 rows (1 KB) further
        const int32_t* bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
        const bool half8 = p.cpb_log2 < 0;
        const int per_load = half8 ? 16 : 32;  // chunks whose table entries one warp-wide load covers
        bool ok = true;
        int n_issued = 0;  // blocks whose loads were issued
        for (int b0 = 0; b0 < nblk && ok; b0 += per_load) {
            const int nb = min(per_load, nblk - b0);
            int my = p.num_blocks;  // outside the tensor map: TMA fills zeros
            const int e = half8 ? 2 * (blk0 + b0) + lane : (blk0 + b0 + lane) >> p.cpb_log2;
            if (half8 ? (lane < 2 * nb && 8 * e < L) : (lane < nb)) {
                my = (spec && b0 == 0) ? spec_blk : __ldg(bt + e);
                if (my < 0 || my >= p.num_blocks) {
                    flag_error(p.err, PA_DEVERR_BLOCK);
                    my = p.num_blocks;
                }
            }
            for (int j = 0; j < nb; ++j) {
                const int blk = __shfl_sync(0xffffffffu, my, half8 ? 2 * j : j);
                const int blk_b = __shfl_sync(0xffffffffu, my, (2 * j + 1) & 31);  // half8 only
                const int b = b0 + j;
                const int st = b % C::NST;
                const uint32_t ph = (b / C::NST) & 1;
                if (lane == 0) {
                    // chunk's first row in its block
                    const int row0 = half8 ? 0 : ((blk0 + b) & ((1 << p.cpb_log2) - 1)) * C::BS;
                    if (b >= C::NST && !mbar_wait(bar_empty + 8 * st, ph ^ 1, p.err)) ok = false;
                    if (ok) {
                        const uint32_t dst = ring + st * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE_BYTES);
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv) {
                            const CUtensorMap* map = kv ? &tmV : &tmK;
                            const uint32_t tile = dst + kv * C::TILE_BYTES;
#pragma unroll
                            for (int hf = 0; hf < C::HALVES; ++hf) {
                                tma_load_4d(tile + hf * C::SLAB_BYTES, map, hf * 64, g, row0, blk, bar_full + 8 * st,
                                            pol);
                                if (half8)
                                    tma_load_4d(tile + hf * C::SLAB_BYTES + 8 * 128, map, hf * 64, g, 0, blk_b,
                                                bar_full + 8 * st, pol);
                            }
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                n_issued = b + 1;
            }
        }
        // No load may still be landing when the consumers reuse the ring for their merge or the
        // CTA exits (after a time-out the consumers may not have taken every stage): wait, with
        // the time limit, for the last phase of every stage that was filled, then release the
        // consumers' merge barrier.  Each of those phases is the one just issued or already done.
        if (lane == 0) {
            for (int st = 0; st < C::NST && st < n_issued; ++st) {
                const int b_last = st + ((n_issued - 1 - st) / C::NST) * C::NST;
                (void)mbar_wait(bar_full + 8 * st, (b_last / C::NST) & 1, p.err);
            }
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(C::THREADS) : "memory");
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int tg = lane >> 3, dl = lane & 7;  // q.K layout: token group, lane within token
    // q for the G heads of this group, this lane's CPL chunks, pre-scaled by scale*log2(e)
    float qf[G][C::CPL][8];
    int chunk_col[C::CPL];  // first column (element index) of each of this lane's chunks
#pragma unroll
    for (int j = 0; j < C::CPL; ++j) {
        // HALVES = 4: chunk dl of every slab; 2: two chunks of one slab, staggered; 1: chunk dl
        const int half = (C::HALVES == 4) ? j : (C::HALVES == 2) ? (dl >> 2) : 0;
        const int c = (C::HALVES == 2) ? ((2 * (dl & 3) + half + j) & 7) : dl;
        chunk_col[j] = half * 64 + c * 8;
    }
    {
        const uint16_t* qrow = static_cast<const uint16_t*>(p.q) + ((size_t)s * p.n_q_heads + (size_t)g * G) * p.hd;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < C::CPL; ++j) {
                uint4 raw = chunk_col[j] < p.hd ? ldg_nc_128(qrow + h * p.hd + chunk_col[j]) : make_uint4(0u, 0u, 0u, 0u);
                unpack8<BF16>(raw, qf[h][j]);
#pragma unroll
                for (int e = 0; e < 8; ++e) qf[h][j][e] *= p.qk_scale_log2;
            }
    }

    // this lane's head in the reduced-score layout, and whether it reports that head
    const int n0 = 4 * G;
    int my_h;
    {
        int base = ((lane & 4) ? n0 / 2 : 0) + ((lane & 2) ? n0 / 4 : 0) + ((n0 >= 8 && (lane & 1)) ? n0 / 8 : 0);
        my_h = base / 4;
    }
    const int hmask = (G == 1) ? 0 : (G == 2) ? 4 : (G == 4) ? 6 : 7;
    const bool rep = (tg == 0) && ((dl & ~hmask) == 0);

    float m_run = -INFINITY, l_run = 0.f;
    float o[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = 0.f;

    const int dg = lane % C::CR, tgp = lane / C::CR;  // P.V layout
    float* pw = p_buf + warp * C::BS * G;
    float* aw = a_buf + warp * 8;

    bool ok = true;
    for (int b = warp; b < nblk; b += C::NCW) {
        const int st = b % C::NST;
        const uint32_t ph = (b / C::NST) & 1;
        const bool arrived = mbar_wait(bar_full + 8 * st, ph, p.err);
        if (!__all_sync(0xffffffffu, arrived)) { ok = false; break; }  // leave the loop warp-uniformly
        const uint32_t kt = ring + st * C::STAGE_BYTES;
        const int nvalid = min(C::BS, t_end - (t_begin + b * C::BS));
        consume_chunk<D, G, BF16>(kt, nvalid, qf, chunk_col, lane, my_h, rep, pw, aw, m_run, l_run, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // fold the token groups of the P.V layout
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float x = o[h][e];
            if constexpr (C::TGP >= 2) x += __shfl_xor_sync(0xffffffffu, x, C::CR);
            if constexpr (C::TGP >= 4) x += __shfl_xor_sync(0xffffffffu, x, 2 * C::CR);
            o[h][e] = x;
        }

    // ---------------------------------------------------------------- merge the 4 warps
    // the consumer warps are done with the ring and the producer has seen every load land
    // (barrier 2 counts the producer warp too); reuse the ring as the merge area
    asm volatile("bar.sync 2, %0;" ::"n"(C::THREADS) : "memory");
    float* mo = reinterpret_cast<float*>(smem);            // [NCW][G][D]
    float* mm = mo + C::NCW * G * D;                        // [NCW][G]
    float* ml = mm + C::NCW * G;                            // [NCW][G]
    if (!ok) { m_run = -INFINITY; l_run = 0.f; }
    if (tgp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4* dst = reinterpret_cast<float4*>(mo + (warp * G + h) * D + dg * 8);
            dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
            dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
        }
    }
    if (rep) {
        mm[warp * G + my_h] = m_run;
        ml[warp * G + my_h] = l_run;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
    // the shared-prefix partials are complete and visible past this point (and this grid completes
    // only after that pass has: the split-K merge relies on it)
    if (p.pf_parts > 0) asm volatile("griddepcontrol.wait;" ::: "memory");

    const int tid = threadIdx.x;  // 0 .. 127
    const int hq0 = g * G;
    for (int idx = 2 * tid; idx < G * D; idx += 2 * C::NCW * 32) {
        const int h = idx / D, d = idx - h * D;
        const size_t row = (size_t)s * p.n_q_heads + hq0 + h;
        const bool fold = direct && p.pf_parts > 0;  // split-K pieces leave the prefix to the reduce
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, mm[w * G + h]);
        PrefixRow pfr;
        if (fold) {
            prefix_load(p, row, d, D, pfr);
            M = prefix_max(p, pfr, row, M);
        }
        float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) {
                const float wt = ex2(mm[w * G + h] - M);
                Lsum = fmaf(ml[w * G + h], wt, Lsum);
                o0 = fmaf(mo[(w * G + h) * D + d], wt, o0);
                o1 = fmaf(mo[(w * G + h) * D + d + 1], wt, o1);
            }
            if (fold) prefix_add(p, pfr, row, d, D, M, Lsum, o0, o1);
        }
        const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
        if (direct) {
            uint32_t packed = F::pack_rn(o0 * inv, o1 * inv);
            if (d < p.hd) *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * p.hd + d) = packed;
        } else {
            const size_t pr = row * p.max_parts + piece;
            *reinterpret_cast<float2*>(p.ws_o + pr * D + d) = make_float2(o0 * inv, o1 * inv);
            if (d == 0) {
                p.ws_m[pr] = M * 0.69314718055994531f;  // back to natural-log units
                p.ws_l[pr] = Lsum;
            }
        }
    }
}

// The persistent one-pass grid (p.persist): gridDim.x CTAs (one per resident slot), each running
// the list of (sequence, KV head) units lpt_units gives it, whole contexts, no split-K.  The
// producer streams the next unit's blocks into the ring while the consumers merge this one, and
// no CTA pays the start-up (barriers, ordering) more than once.  The per-block work is that of
// decode_kernel.
template <int D, int G, bool BF16>
__global__ void __launch_bounds__(DecodeCfg<D, G, BF16>::THREADS,
                                  D == 256 ? (G <= 2 ? 2 : 1) : ((G <= 4) ? 3 : (D == 64 ? 2 : 1)))
decode_kernel_persistent(const DecodeParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using C = DecodeCfg<D, G, BF16>;
    using F = F16x2<BF16>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern of TMA
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_addr(smem);
    float* p_buf = reinterpret_cast<float*>(smem + C::RING_BYTES);
    float* a_buf = reinterpret_cast<float*>(smem + C::RING_BYTES + C::P_BYTES);
    const uint32_t bar_full = ring + C::P_BAR_OFF;
    const uint32_t bar_empty = bar_full + C::NST * 8;

    // launched as a programmatic dependent of whatever kernel precedes it in the stream: nothing is
    // read before that kernel has completed (a no-op when it never signalled early); after a
    // shared-prefix pass, which waited itself before letting this grid launch, only the merge waits
    if (p.pf_parts == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int* list = reinterpret_cast<int*>(smem + C::P_LIST_OFF);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::P_FLAG_OFF);  // [0] units, [1] abort

    // ---- the units this CTA runs
    {
        const int n = lpt_units(p, reinterpret_cast<int*>(smem), list, C::LIST_MAX);
        if (threadIdx.x == 0) flags[0] = n;
    }
    // the new rows of pa_decode_write written (one arrival per consumer warp)
    const uint32_t bar_wdone = ring + C::P_FLAG_OFF + 8;
    if (threadIdx.x == 0) {
        flags[1] = 0;
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        mbar_init(bar_wdone, C::NCW);
        fence_barrier_init();
    }
    fence_proxy_async_smem();  // the ordering scratch (ring) is written by TMA next
    __syncthreads();
    const int n_units = flags[0];

    // a unit: the whole context of (sequence s, KV head g), clamped to what the table addresses,
    // in nblk 16-token chunks
    const int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);
    struct Unit {
        int s, g, L, t0, nblk;  // tokens [t0, L) are streamed (t0 > 0 past a shared prefix)
    };
    auto unit_at = [&](int k, bool report) {
        Unit u;
        u.s = list[3 * k];
        u.g = list[3 * k + 1];
        int L = __ldg(p.context_lens + u.s);
        if (L < 0 || L > cap) {
            if (report && u.g == 0 && threadIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
            L = L < 0 ? 0 : cap;
        }
        u.L = L;
        u.t0 = min(L, p.prefix_tokens);
        u.nblk = (L - u.t0 + C::BS - 1) / C::BS;
        return u;
    };

    if (warp == C::NCW) {
        // ------------------------------------------------------------ producer warp
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_first();
        const bool half8 = p.cpb_log2 < 0;
        const int per_load = half8 ? 16 : 32;  // chunks whose table entries one warp-wide load covers
        bool ok = true;
        bool written = p.new_k == nullptr;  // the consumer warps' new rows seen
        int n_issued = 0;  // blocks (ring stages) whose loads were issued, over all units
        for (int k = 0; k < n_units && ok; ++k) {
            const Unit u = unit_at(k, false);
            // 16-token chunk c of the sequence: table entry c >> cpb_log2, rows 16 (c mod 2^cpb_log2) + 0..15;
            // with blocks of 8 tokens, entries 2c and 2c + 1 (the second only if the context reaches
            // it), each an 8-row box, the second landing 8 rows (1 KB) further
            const int32_t* bt = p.block_tables + (size_t)u.s * p.max_blocks_per_seq;
            const int c0 = u.t0 / C::BS;  // the unit's first chunk (t0 is a multiple of 16)
            for (int b0 = 0; b0 < u.nblk && ok; b0 += per_load) {
                const int nb = min(per_load, u.nblk - b0);
                int my = p.num_blocks;  // outside the tensor map: TMA fills zeros
                const int e = half8 ? 2 * (c0 + b0) + lane : (c0 + b0 + lane) >> p.cpb_log2;
                if (half8 ? (lane < 2 * nb && 8 * e < u.L) : (lane < nb)) {
                    my = __ldg(bt + e);
                    if (my < 0 || my >= p.num_blocks) {
                        flag_error(p.err, PA_DEVERR_BLOCK);
                        my = p.num_blocks;
                    }
                }
                for (int j = 0; j < nb; ++j) {
                    const int blk = __shfl_sync(0xffffffffu, my, half8 ? 2 * j : j);
                    const int blk_b = __shfl_sync(0xffffffffu, my, (2 * j + 1) & 31);  // half8 only
                    const int gb = n_issued;
                    const int st = gb % C::NST;
                    const uint32_t ph = (gb / C::NST) & 1;
                    if (lane == 0) {
                        // chunk's first row in its block
                        const int row0 = half8 ? 0 : ((c0 + b0 + j) & ((1 << p.cpb_log2) - 1)) * C::BS;
                        if (gb >= C::NST && !mbar_wait(bar_empty + 8 * st, ph ^ 1, p.err)) ok = false;
                        // a unit's last chunk holds its sequence's new row: written first
                        if (ok && !written && b0 + j == u.nblk - 1) {
                            ok = mbar_wait(bar_wdone, 0, p.err);
                            written = true;
                        }
                        if (ok) {
                            const uint32_t dst = ring + st * C::STAGE_BYTES;
                            mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE_BYTES);
#pragma unroll
                            for (int kv = 0; kv < 2; ++kv) {
                                const CUtensorMap* map = kv ? &tmV : &tmK;
                                const uint32_t tile = dst + kv * C::TILE_BYTES;
#pragma unroll
                                for (int hf = 0; hf < C::HALVES; ++hf) {
                                    tma_load_4d(tile + hf * C::SLAB_BYTES, map, hf * 64, u.g, row0, blk,
                                                bar_full + 8 * st, pol);
                                    if (half8)
                                        tma_load_4d(tile + hf * C::SLAB_BYTES + 8 * 128, map, hf * 64, u.g, 0, blk_b,
                                                    bar_full + 8 * st, pol);
                                }
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    n_issued = gb + 1;
                }
            }
        }
        // No load may still be landing when the CTA exits (after a time-out the consumers may not
        // have taken every stage): wait, with the time limit, for the last phase of every stage
        // that was filled, then release the consumers' final barrier.  Each of those phases is the
        // one just issued or already done.
        if (lane == 0) {
            for (int st = 0; st < C::NST && st < n_issued; ++st) {
                const int b_last = st + ((n_issued - 1 - st) / C::NST) * C::NST;
                (void)mbar_wait(bar_full + 8 * st, (b_last / C::NST) & 1, p.err);
            }
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(C::THREADS) : "memory");
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int tg = lane >> 3, dl = lane & 7;  // q.K layout: token group, lane within token
    int chunk_col[C::CPL];  // first column (element index) of each of this lane's chunks
#pragma unroll
    for (int j = 0; j < C::CPL; ++j) {
        // HALVES = 4: chunk dl of every slab; 2: two chunks of one slab, staggered; 1: chunk dl
        const int half = (C::HALVES == 4) ? j : (C::HALVES == 2) ? (dl >> 2) : 0;
        const int c = (C::HALVES == 2) ? ((2 * (dl & 3) + half + j) & 7) : dl;
        chunk_col[j] = half * 64 + c * 8;
    }
    // this lane's head in the reduced-score layout, and whether it reports that head
    const int n0 = 4 * G;
    int my_h;
    {
        int base = ((lane & 4) ? n0 / 2 : 0) + ((lane & 2) ? n0 / 4 : 0) + ((n0 >= 8 && (lane & 1)) ? n0 / 8 : 0);
        my_h = base / 4;
    }
    const int hmask = (G == 1) ? 0 : (G == 2) ? 4 : (G == 4) ? 6 : 7;
    const bool rep = (tg == 0) && ((dl & ~hmask) == 0);
    const int dg = lane % C::CR, tgp = lane / C::CR;  // P.V layout
    float* pw = p_buf + warp * C::BS * G;
    float* aw = a_buf + warp * 8;

    if (p.new_k) {
        // pa_decode_write: this CTA's units' new K and V rows into the cache (head g's chunks of
        // row s for unit (s, g)), made visible to the TMA loads (async proxy) before the producer,
        // which waits for every warp's arrival, loads a unit's last chunk
        const int hv = p.hd / 8;  // 16-byte chunks of one head's row
        const int bs = p.cpb_log2 >= 0 ? 16 << p.cpb_log2 : 8;
        for (int idx = (int)threadIdx.x; idx < n_units * 2 * hv; idx += C::NCW * 32) {
            const int k = idx / (2 * hv), r = idx - k * 2 * hv;
            const int kv = r / hv, c = r - kv * hv;
            const int s = list[3 * k], g = list[3 * k + 1];
            const long long slot = p.new_slots[s];
            if (slot < 0) continue;
            if (slot >= p.n_slots) {
                if (r == 0) flag_error(p.err, PA_DEVERR_SLOT);
                continue;
            }
            if (r == 0) {
                // the slot must be that of the context's last token, the one the last chunk holds
                int L = __ldg(p.context_lens + s);
                L = L < 0 ? 0 : min(L, cap);
                const int e = L > 0 ? (L - 1) / bs : 0;
                const long long want = L > 0 && e < p.max_blocks_per_seq
                                           ? (long long)__ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + e) * bs + (L - 1) % bs
                                           : -1;
                if (slot != want) flag_error(p.err, PA_DEVERR_SLOT);
            }
            const size_t from = (size_t)s * p.row_vecs + (size_t)g * hv + c;
            const size_t to = (size_t)slot * p.row_vecs + (size_t)g * hv + c;
            if (kv == 0) p.k_cache_w[to] = __ldg(p.new_k + from);
            else p.v_cache_w[to] = __ldg(p.new_v + from);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_wdone);
    }

    bool ok = true;
    int base_blk = 0;  // ring index of the unit's first block
    for (int k = 0; k < n_units; ++k) {
        int L, t0, nblk, s, g;
        // q for the G heads of this group, this lane's CPL chunks, pre-scaled by scale*log2(e)
        float qf[G][C::CPL][8];
        {
            const Unit u = unit_at(k, true);
            L = u.L;
            t0 = u.t0;
            nblk = u.nblk;
            s = u.s;
            g = u.g;
            const uint16_t* qrow =
                static_cast<const uint16_t*>(p.q) + ((size_t)u.s * p.n_q_heads + (size_t)u.g * G) * p.hd;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int j = 0; j < C::CPL; ++j) {
                    uint4 raw = chunk_col[j] < p.hd ? ldg_nc_128(qrow + h * p.hd + chunk_col[j])
                                                    : make_uint4(0u, 0u, 0u, 0u);
                    unpack8<BF16>(raw, qf[h][j]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) qf[h][j][e] *= p.qk_scale_log2;
                }
        }

        float m_run = -INFINITY, l_run = 0.f;
        float o[G][8];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] = 0.f;

        // this warp's blocks: ring indices base_blk + b with (base_blk + b) mod NCW == warp, so that a
        // ring stage always belongs to the same warp
        for (int b = (warp - base_blk % C::NCW + C::NCW) % C::NCW; ok && b < nblk; b += C::NCW) {
            const int gb = base_blk + b;
            const int st = gb % C::NST;
            const uint32_t ph = (gb / C::NST) & 1;
            const bool arrived = mbar_wait(bar_full + 8 * st, ph, p.err);
            if (!__all_sync(0xffffffffu, arrived)) { ok = false; break; }  // leave the loop warp-uniformly
            const uint32_t kt = ring + st * C::STAGE_BYTES;
            const int nvalid = min(C::BS, L - t0 - b * C::BS);
            consume_chunk<D, G, BF16, false>(kt, nvalid, qf, chunk_col, lane, my_h, rep, pw, aw, m_run, l_run, o);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        }
        base_blk += nblk;

        // fold the token groups of the P.V layout
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float x = o[h][e];
                if constexpr (C::TGP >= 2) x += __shfl_xor_sync(0xffffffffu, x, C::CR);
                if constexpr (C::TGP >= 4) x += __shfl_xor_sync(0xffffffffu, x, 2 * C::CR);
                o[h][e] = x;
            }

        // ------------------------------------------------------------ merge the 4 warps
        float* mo = reinterpret_cast<float*>(smem + C::P_MERGE_OFF);  // [NCW][G][D]
        float* mm = mo + C::NCW * G * D;                             // [NCW][G]
        float* ml = mm + C::NCW * G;                                 // [NCW][G]
        volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::P_FLAG_OFF) + 1;
        if (!ok) {
            m_run = -INFINITY;
            l_run = 0.f;
            if (lane == 0) *abort_flag = 1;  // every consumer warp stops after this unit
        }
        if (tgp == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float4* dst = reinterpret_cast<float4*>(mo + (warp * G + h) * D + dg * 8);
                dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
                dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
            }
        }
        if (rep) {
            mm[warp * G + my_h] = m_run;
            ml[warp * G + my_h] = l_run;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
        // the shared-prefix partials are complete and visible past this point
        if (k == 0 && p.pf_parts > 0) asm volatile("griddepcontrol.wait;" ::: "memory");

        const int tid = threadIdx.x;  // 0 .. 127
        const int hq0 = g * G;
        for (int idx = 2 * tid; idx < G * D; idx += 2 * C::NCW * 32) {
            const int h = idx / D, d = idx - h * D;
            const size_t row = (size_t)s * p.n_q_heads + hq0 + h;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, mm[w * G + h]);
            PrefixRow pfr;
            if (p.pf_parts > 0) {
                prefix_load(p, row, d, D, pfr);
                M = prefix_max(p, pfr, row, M);
            }
            float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) {
                    const float wt = ex2(mm[w * G + h] - M);
                    Lsum = fmaf(ml[w * G + h], wt, Lsum);
                    o0 = fmaf(mo[(w * G + h) * D + d], wt, o0);
                    o1 = fmaf(mo[(w * G + h) * D + d + 1], wt, o1);
                }
                if (p.pf_parts > 0) prefix_add(p, pfr, row, d, D, M, Lsum, o0, o1);
            }
            const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
            if (d < p.hd)
                *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * p.hd + d) =
                    F::pack_rn(o0 * inv, o1 * inv);
        }
        // the merge area is rewritten by the next unit; every warp has seen the abort flag
        asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
        if (*abort_flag) break;
    }
    // the producer has seen every load land (barrier 2 counts it too)
    asm volatile("bar.sync 2, %0;" ::"n"(C::THREADS) : "memory");
}

// decode_kernel_dyn over whole units (dyn_units): the sequences by streamed 16-token chunk count,
// longest first (ties by index), so that the units handed out last are the shortest.  order: S
// ints; scratch: S + 2 (part_tokens / 16 + 1) ints nothing else uses yet.  Every CTA builds the
// same order.  All threads call this.
__device__ __forceinline__ void dyn_unit_order(const DecodeParams& p, int cap, int* order, int* scratch) {
    const int S = p.num_seqs, tid = threadIdx.x, lane = tid & 31;
    const int nb = p.part_tokens / 16 + 1;
    int* key = scratch;     // [S] chunk count
    int* hist = key + S;    // [nb]
    int* start = hist + nb;
    for (int i = tid; i < nb; i += blockDim.x) hist[i] = 0;
    for (int i = tid; i < S; i += blockDim.x) {
        int L = __ldg(p.context_lens + i);
        if (L < 0 || L > cap) {
            if (blockIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
            L = L < 0 ? 0 : cap;
        }
        key[i] = min((streamed_tokens(p, L) + 15) >> 4, nb - 1);
    }
    __syncthreads();
    for (int i = tid; i < S; i += blockDim.x) atomicAdd(&hist[key[i]], 1);
    __syncthreads();
    if (tid < 32) {
        int before = 0;
        for (int top = nb - 1; top >= 0; top -= 32) {
            const int k = top - lane;
            const int v = (k >= 0) ? hist[k] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (k >= 0) start[k] = before + incl - v;
            before += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        for (int b = 0; b < S; b += 32) {
            const int i = b + lane;
            const int k = i < S ? key[i] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, k);
            if (k >= 0) order[start[k] + __popc(same & ((1u << lane) - 1u))] = i;
            __syncwarp();
            if (k >= 0 && lane == __ffs(same) - 1) start[k] += __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
}

// decode_kernel_dyn's per-sequence layout with tail pieces: len[s] = the clamped context length,
// cumA[s] / cumB[s] = full / tail pieces of the sequences before s (a sequence with nothing
// streamed has one empty tail piece, which writes its output row).  All threads call this.
__device__ __forceinline__ void dyn_piece_counts(const DecodeParams& p, int cap, int* len, int* cumA, int* cumB) {
    const int S = p.num_seqs, tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < S; i += blockDim.x) {
        int L = __ldg(p.context_lens + i);
        if (L < 0 || L > cap) {
            if (blockIdx.x == 0) flag_error(p.err, PA_DEVERR_LENGTH);
            L = L < 0 ? 0 : cap;
        }
        const int Ls = streamed_tokens(p, L), f = full_pieces_of(p, Ls);
        len[i] = L;
        cumA[i + 1] = f;
        cumB[i + 1] = Ls > 0 ? pieces_of(p, L) - f : 1;
    }
    __syncthreads();
    if (tid < 32) {
        int runA = 0, runB = 0;
        if (lane == 0) cumA[0] = cumB[0] = 0;
        for (int b = 0; b < S; b += 32) {
            const int i = b + lane;
            int a = i < S ? cumA[i + 1] : 0, c = i < S ? cumB[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int ya = __shfl_up_sync(0xffffffffu, a, o), yc = __shfl_up_sync(0xffffffffu, c, o);
                if (lane >= o) {
                    a += ya;
                    c += yc;
                }
            }
            if (i < S) {
                cumA[i + 1] = runA + a;
                cumB[i + 1] = runB + c;
            }
            runA += __shfl_sync(0xffffffffu, a, 31);
            runB += __shfl_sync(0xffffffffu, c, 31);
        }
    }
    __syncthreads();
}

// The dynamic split-K grid (p.dyn): gridDim.x CTAs, one per resident slot, take work items --
// the split-K pieces, highest piece index first as in decode_kernel's grid, or with tail pieces
// the full pieces and then the tail pieces -- from a counter in the workspace, which the previous
// call's merge left at zero with its tag set (DecodeParams::dyn_tag; without the tag the CTAs
// take the items in a fixed order).  WRITE: the instantiation that also writes pa_decode_write's
// rows.  The producer warp fetches an item, publishes it through a small queue in
// shared memory and streams its chunks into the ring, the next item's while the consumers merge
// this one; the SMs that stream faster take more pieces, so the grid ends evenly, and no CTA pays
// its start-up more than once.  Each item starts on a ring index that is a multiple of the
// consumer-warp count, so consumer warp w always takes the item's chunks w, w + NCW, ... (the
// order of accumulation does not depend on which items a CTA took) and every ring stage keeps one
// owning warp; both sides count each stage's uses for the barrier parities, as the skipped ring
// indices never touch a stage.  The per-chunk work is decode_kernel's.
template <int D, int G, bool BF16, bool WRITE = false>
__global__ void __launch_bounds__(DecodeCfg<D, G, BF16>::THREADS,
                                  D == 256 ? (G <= 2 ? 2 : 1) : ((G <= 4) ? 3 : (D == 64 ? 2 : 1)))
decode_kernel_dyn(const DecodeParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using C = DecodeCfg<D, G, BF16>;
    using F = F16x2<BF16>;
    constexpr int NQS = 4;  // item queue slots
    static_assert(2 * NQS * 8 + NQS * 8 * 4 <= C::LIST_MAX * 3 * 4, "item queue area");
    static_assert(C::NST <= 32, "stage bit masks");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern of TMA
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_addr(smem);
    float* p_buf = reinterpret_cast<float*>(smem + C::RING_BYTES);
    float* a_buf = reinterpret_cast<float*>(smem + C::RING_BYTES + C::P_BYTES);
    const uint32_t bar_full = ring + C::P_BAR_OFF;
    const uint32_t bar_empty = bar_full + C::NST * 8;
    const uint32_t bar_qfull = ring + C::P_LIST_OFF;   // [NQS] an item (or the end) published
    const uint32_t bar_qempty = bar_qfull + NQS * 8;   // [NQS] the consumers are done with the slot
    volatile int* qslot = reinterpret_cast<volatile int*>(smem + C::P_LIST_OFF + 2 * NQS * 8);  // [NQS][8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // launched as a programmatic dependent of whatever kernel precedes it in the stream: nothing is
    // read before that kernel has completed; after a shared-prefix pass only the merge waits
    if (p.pf_parts == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        for (int k = 0; k < NQS; ++k) {
            mbar_init(bar_qfull + 8 * k, 1);
            mbar_init(bar_qempty + 8 * k, 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int units = p.num_seqs * p.n_kv_heads;
    int cap = table_row_tokens(p.max_blocks_per_seq, p.cpb_log2);
    if (p.prefix_tokens + p.cover_parts * p.part_tokens < cap) cap = p.prefix_tokens + p.cover_parts * p.part_tokens;
    // the item order: with tail pieces, each CTA first lays out per sequence its clamped length and
    // running counts of full and of tail pieces (shared memory, batches of up to DYN_SMAX
    // sequences); items are then the full pieces, sequence by sequence (KV head fastest), followed
    // by the tail pieces.  Without: (piece index from the highest down) x unit, skipping the pieces
    // past a context.
    const bool tail = p.tail_tokens > 0;
    // the first claim and the block tables' way into L2 overlap the prologue's length loads: the
    // producer takes its first item now, and every CTA prefetches its share of the table lines
    // (tables of up to 4 MB)
    int first = 0;
    bool fixed = false;  // the counter is not known to start at zero: CTA b takes items b, b + grid, ...
    if (warp == C::NCW && lane == 0) {
        first = atomicAdd(p.dyn_counter, 1);
        if (p.dyn_tag) fixed = __ldcg(p.dyn_tag) != kDynTag;
    }
    {
        long long lines = ((long long)p.num_seqs * p.max_blocks_per_seq * 4 + 127) / 128;
        if (lines > 32768) lines = 0;
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < lines; i += (long long)gridDim.x * blockDim.x)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.block_tables) + i * 128));
    }
    int* o_len = reinterpret_cast<int*>(smem + C::D_LEN_OFF);
    int* o_cumA = reinterpret_cast<int*>(smem + C::D_CUMA_OFF);
    int* o_cumB = reinterpret_cast<int*>(smem + C::D_CUMB_OFF);
    if (tail) dyn_piece_counts(p, cap, o_len, o_cumA, o_cumB);
    int* o_order = o_cumA;  // dyn_units: the sequences longest first
    if (p.dyn_units) dyn_unit_order(p, cap, o_order, reinterpret_cast<int*>(smem));  // (the ring: no load yet)
    const long long n_full = tail ? (long long)o_cumA[p.num_seqs] * p.n_kv_heads : 0;
    const long long total = tail ? n_full + (long long)o_cumB[p.num_seqs] * p.n_kv_heads
                                 : (long long)units * p.max_parts;

    if (warp == C::NCW) {
        // ------------------------------------------------------------ producer warp
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_first();
        const bool half8 = p.cpb_log2 < 0;
        const int per_load = half8 ? 16 : 32;  // chunks whose table entries one warp-wide load covers
        uint32_t fused = 0, fpar = 0;          // per stage: filled before; parity of its fill count
        int ring_next = 0, nq = 0;             // ring index of the next chunk; items published
        bool ok = true;
        int n_claims = 0;
        for (bool claimed = true; ok; claimed = false, ++n_claims) {
            int item = first;
            if (lane == 0 && !claimed && !fixed) item = atomicAdd(p.dyn_counter, 1);
            if (fixed) item = (int)blockIdx.x + n_claims * (int)gridDim.x;
            item = __shfl_sync(0xffffffffu, item, 0);
            const bool end = (long long)item >= total;
            int s = -1, g = 0, piece = 0, t_begin = 0, t_end = 0, n_parts = 0;
            int L_item = -1;  // the item's sequence's clamped context length
            if (!end && tail) {
                const bool full = (long long)item < n_full;
                const int r = full ? item : (int)((long long)item - n_full);
                const int e = r / p.n_kv_heads;
                g = r - e * p.n_kv_heads;
                const int* cum = full ? o_cumA : o_cumB;
                // the sequence s with cum[s] <= e < cum[s + 1]
                int lo = 0, hi = p.num_seqs;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (cum[mid] <= e) lo = mid; else hi = mid;
                }
                s = lo;
                const int L = o_len[s], base = min(L, p.prefix_tokens), Ls = L - base;
                const int f = o_cumA[s + 1] - o_cumA[s];
                L_item = L;
                if (full) {
                    piece = e - o_cumA[s];
                    t_begin = base + piece * p.part_tokens;
                    t_end = t_begin + p.part_tokens;
                } else {
                    const int k = e - o_cumB[s];
                    piece = f + k;
                    t_begin = min(L, base + f * p.part_tokens + k * p.tail_tokens);
                    t_end = min(L, t_begin + p.tail_tokens);
                }
                n_parts = Ls > 0 ? f + (o_cumB[s + 1] - o_cumB[s]) : 0;
            } else if (!end) {
                const int qpos = item / units, sg = item - qpos * units;
                piece = (p.max_parts - 1) - qpos;
                s = sg / p.n_kv_heads;
                g = sg - s * p.n_kv_heads;
                if (p.dyn_units) s = o_order[s];  // units longest first
                int L = __ldg(p.context_lens + s);
                if (L < 0 || L > cap) {
                    if (piece == 0 && g == 0 && lane == 0) flag_error(p.err, PA_DEVERR_LENGTH);
                    L = L < 0 ? 0 : cap;
                }
                L_item = L;
                const int base = min(L, p.prefix_tokens);
                t_begin = min(L, base + piece * p.part_tokens);
                t_end = min(L, t_begin + p.part_tokens);
                n_parts = (L - base + p.part_tokens - 1) / p.part_tokens;
                if (t_begin >= t_end && piece > 0) continue;  // a piece past this sequence's context
            }
            const int nblk = end ? 0 : (t_end - t_begin + C::BS - 1) / C::BS;
            const int r0 = (ring_next + C::NCW - 1) / C::NCW * C::NCW;
            const int k = nq % NQS;
            if (lane == 0) {
                if (nq >= NQS) ok = mbar_wait(bar_qempty + 8 * k, ((nq / NQS) - 1) & 1, p.err);
                if (ok) {
                    volatile int* q = qslot + 8 * k;
                    q[0] = end ? -1 : s;
                    q[1] = g;
                    q[2] = piece;
                    q[3] = t_begin;
                    q[4] = t_end;
                    q[5] = n_parts;
                    q[6] = r0;
                    mbar_arrive(bar_qfull + 8 * k);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ++nq;
            if (end || !ok) break;
            // WRITE (pa_decode_write): the item that ends at its sequence's context length (the one
            // holding the last token, or the empty piece of an empty context) writes head g's part of the
            // sequence's new K and V rows before the chunk holding that token is loaded (generic
            // stores, then the proxy fence, then the TMA); the rows' loads go out now, behind the
            // item's earlier chunks
            const bool row_item = WRITE && t_end == L_item;
            const int hv = p.hd / 8;  // 16-byte chunks of one head's row
            long long nslot = -1;
            uint4 nrow[2];
            if (row_item) {
                nslot = __ldg(p.new_slots + s);
                if (nslot >= p.n_slots) {
                    if (lane == 0) flag_error(p.err, PA_DEVERR_SLOT);
                    nslot = -1;
                }
                if (nslot >= 0) {
#pragma unroll
                    for (int i2 = 0; i2 < 2; ++i2) {
                        const int c = lane + 32 * i2, kv = c / hv, cc = c - kv * hv;
                        if (c < 2 * hv) nrow[i2] = __ldg((kv ? p.new_v : p.new_k) + (size_t)s * p.row_vecs + (size_t)g * hv + cc);
                    }
                }
            }
            // the row into its slot; `want` = the slot of token L - 1 (-1: none)
            auto store_row = [&](long long want) {
                if (nslot >= 0) {
#pragma unroll
                    for (int i2 = 0; i2 < 2; ++i2) {
                        const int c = lane + 32 * i2, kv = c / hv, cc = c - kv * hv;
                        if (c < 2 * hv) (kv ? p.v_cache_w : p.k_cache_w)[nslot * p.row_vecs + (long long)g * hv + cc] = nrow[i2];
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    if (lane == 0 && nslot != want) flag_error(p.err, PA_DEVERR_SLOT);
                }
                __syncwarp();
            };
            if constexpr (WRITE)
                if (row_item && nblk == 0) store_row(-1);
            // the item's chunks into ring indices r0 .. r0 + nblk - 1; 16-token chunk c of the
            // sequence: table entry c >> cpb_log2, rows 16 (c mod 2^cpb_log2) + 0..15 (blocks of 8:
            // entries 2c and 2c + 1, the second only if the context reaches it)
            const int blk0 = t_begin / C::BS;
            const int32_t* bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
            for (int b0 = 0; b0 < nblk && ok; b0 += per_load) {
                const int nb = min(per_load, nblk - b0);
                int my = p.num_blocks;  // outside the tensor map: TMA fills zeros
                const int e = half8 ? 2 * (blk0 + b0) + lane : (blk0 + b0 + lane) >> p.cpb_log2;
                if (half8 ? (lane < 2 * nb && 8 * e < t_end) : (lane < nb)) {
                    my = __ldg(bt + e);
                    if (my < 0 || my >= p.num_blocks) {
                        flag_error(p.err, PA_DEVERR_BLOCK);
                        my = p.num_blocks;
                    }
                }
                for (int j = 0; j < nb; ++j) {
                    const int blk = __shfl_sync(0xffffffffu, my, half8 ? 2 * j : j);
                    const int blk_b = __shfl_sync(0xffffffffu, my, (2 * j + 1) & 31);  // half8 only
                    const int st = (r0 + b0 + j) % C::NST;
                    if constexpr (WRITE) {
                        if (row_item && b0 + j == nblk - 1) {
                            const int tl = L_item - 1;  // the last token, in this chunk
                            store_row(half8 ? (long long)((tl & 15) < 8 ? blk : blk_b) * 8 + (tl & 7)
                                            : (long long)blk * (16 << p.cpb_log2) + (tl & ((16 << p.cpb_log2) - 1)));
                        }
                    }
                    if (lane == 0) {
                        const int row0 = half8 ? 0 : ((blk0 + b0 + j) & ((1 << p.cpb_log2) - 1)) * C::BS;
                        if ((fused >> st) & 1) ok = mbar_wait(bar_empty + 8 * st, ((fpar >> st) & 1) ^ 1, p.err);
                        if (ok) {
                            const uint32_t dst = ring + st * C::STAGE_BYTES;
                            mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE_BYTES);
#pragma unroll
                            for (int kv = 0; kv < 2; ++kv) {
                                const CUtensorMap* map = kv ? &tmV : &tmK;
                                const uint32_t tile = dst + kv * C::TILE_BYTES;
#pragma unroll
                                for (int hf = 0; hf < C::HALVES; ++hf) {
                                    tma_load_4d(tile + hf * C::SLAB_BYTES, map, hf * 64, g, row0, blk, bar_full + 8 * st, pol);
                                    if (half8)
                                        tma_load_4d(tile + hf * C::SLAB_BYTES + 8 * 128, map, hf * 64, g, 0, blk_b,
                                                    bar_full + 8 * st, pol);
                                }
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    fused |= 1u << st;
                    fpar ^= 1u << st;
                }
            }
            ring_next = r0 + nblk;
        }
        // No load may still be landing when the CTA exits (after a time-out the consumers may not
        // have taken every stage): wait, with the time limit, for the last fill of every stage.
        if (lane == 0) {
            for (int st = 0; st < C::NST; ++st)
                if ((fused >> st) & 1) (void)mbar_wait(bar_full + 8 * st, ((fpar >> st) & 1) ^ 1, p.err);
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(C::THREADS) : "memory");
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int tg = lane >> 3, dl = lane & 7;  // q.K layout: token group, lane within token
    int chunk_col[C::CPL];
#pragma unroll
    for (int j = 0; j < C::CPL; ++j) {
        const int half = (C::HALVES == 4) ? j : (C::HALVES == 2) ? (dl >> 2) : 0;
        const int c = (C::HALVES == 2) ? ((2 * (dl & 3) + half + j) & 7) : dl;
        chunk_col[j] = half * 64 + c * 8;
    }
    const int n0 = 4 * G;
    int my_h;
    {
        int base = ((lane & 4) ? n0 / 2 : 0) + ((lane & 2) ? n0 / 4 : 0) + ((n0 >= 8 && (lane & 1)) ? n0 / 8 : 0);
        my_h = base / 4;
    }
    const int hmask = (G == 1) ? 0 : (G == 2) ? 4 : (G == 4) ? 6 : 7;
    const bool rep = (tg == 0) && ((dl & ~hmask) == 0);
    const int dg = lane % C::CR, tgp = lane / C::CR;  // P.V layout
    float* pw = p_buf + warp * C::BS * G;
    float* aw = a_buf + warp * 8;
    float* mo = reinterpret_cast<float*>(smem + C::P_MERGE_OFF);  // [NCW][G][D]
    float* mm = mo + C::NCW * G * D;                             // [NCW][G]
    float* ml = mm + C::NCW * G;                                 // [NCW][G]

    // [0] the slot arrived, [1] abort: decisions every consumer warp takes together, so that all
    // of them meet the named merge barrier the same number of times
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::P_FLAG_OFF);
    if (threadIdx.x == 0) flags[1] = 0;
    uint32_t cpar = 0;  // per stage this warp owns: parity of its consume count
    bool ok = true, waited = false;
    for (int nq = 0;; ++nq) {
        const int k = nq % NQS;
        if (threadIdx.x == 0) flags[0] = mbar_wait(bar_qfull + 8 * k, (nq / NQS) & 1, p.err) ? 1 : 0;
        asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
        if (!flags[0]) break;  // the producer stopped (a wait gave up)
        const volatile int* q = qslot + 8 * k;
        const int s = q[0];
        if (s < 0) break;  // no more items
        const int g = q[1], piece = q[2], t_begin = q[3], t_end = q[4], n_parts = q[5], r0 = q[6];
        const bool direct = n_parts <= 1;
        float qf[G][C::CPL][8];
        {
            const uint16_t* qrow = static_cast<const uint16_t*>(p.q) + ((size_t)s * p.n_q_heads + (size_t)g * G) * p.hd;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int j = 0; j < C::CPL; ++j) {
                    uint4 raw = chunk_col[j] < p.hd ? ldg_nc_128(qrow + h * p.hd + chunk_col[j]) : make_uint4(0u, 0u, 0u, 0u);
                    unpack8<BF16>(raw, qf[h][j]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) qf[h][j][e] *= p.qk_scale_log2;
                }
        }
        float m_run = -INFINITY, l_run = 0.f;
        float o[G][8];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
        const int nblk = (t_end - t_begin + C::BS - 1) / C::BS;
        // r0 is a multiple of NCW: this warp's chunks b = warp, warp + NCW, ... sit at ring indices
        // r0 + b, all in stages it owns
        for (int b = warp; ok && b < nblk; b += C::NCW) {
            const int st = (r0 + b) % C::NST;
            const bool arrived = mbar_wait(bar_full + 8 * st, (cpar >> st) & 1, p.err);
            if (!__all_sync(0xffffffffu, arrived)) { ok = false; break; }
            const uint32_t kt = ring + st * C::STAGE_BYTES;
            const int nvalid = min(C::BS, t_end - (t_begin + b * C::BS));
            consume_chunk<D, G, BF16>(kt, nvalid, qf, chunk_col, lane, my_h, rep, pw, aw, m_run, l_run, o);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            cpar ^= 1u << st;
        }
        // fold the token groups of the P.V layout
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float x = o[h][e];
                if constexpr (C::TGP >= 2) x += __shfl_xor_sync(0xffffffffu, x, C::CR);
                if constexpr (C::TGP >= 4) x += __shfl_xor_sync(0xffffffffu, x, 2 * C::CR);
                o[h][e] = x;
            }
        if (!ok) {
            m_run = -INFINITY;
            l_run = 0.f;
            if (lane == 0) flags[1] = 1;  // every consumer warp stops after this item
        }
        if (tgp == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float4* dst = reinterpret_cast<float4*>(mo + (warp * G + h) * D + dg * 8);
                dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
                dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
            }
        }
        if (rep) {
            mm[warp * G + my_h] = m_run;
            ml[warp * G + my_h] = l_run;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
        // the shared-prefix partials are complete and visible past this point
        if (p.pf_parts > 0 && !waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
        }
        const int tid = threadIdx.x;  // 0 .. 127
        const int hq0 = g * G;
        for (int idx = 2 * tid; idx < G * D; idx += 2 * C::NCW * 32) {
            const int h = idx / D, d = idx - h * D;
            const size_t row = (size_t)s * p.n_q_heads + hq0 + h;
            const bool fold = direct && p.pf_parts > 0;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, mm[w * G + h]);
            PrefixRow pfr;
            if (fold) {
                prefix_load(p, row, d, D, pfr);
                M = prefix_max(p, pfr, row, M);
            }
            float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) {
                    const float wt = ex2(mm[w * G + h] - M);
                    Lsum = fmaf(ml[w * G + h], wt, Lsum);
                    o0 = fmaf(mo[(w * G + h) * D + d], wt, o0);
                    o1 = fmaf(mo[(w * G + h) * D + d + 1], wt, o1);
                }
                if (fold) prefix_add(p, pfr, row, d, D, M, Lsum, o0, o1);
            }
            const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
            if (direct) {
                if (d < p.hd)
                    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * p.hd + d) = F::pack_rn(o0 * inv, o1 * inv);
            } else {
                const size_t pr = row * p.max_parts + piece;
                *reinterpret_cast<float2*>(p.ws_o + pr * D + d) = make_float2(o0 * inv, o1 * inv);
                if (d == 0) {
                    p.ws_m[pr] = M * 0.69314718055994531f;  // back to natural-log units
                    p.ws_l[pr] = Lsum;
                }
            }
        }
        // the merge area and the queue slot are reused by the next item; every warp has seen the
        // abort flag
        asm volatile("bar.sync 1, %0;" ::"n"(C::NCW * 32) : "memory");
        if (threadIdx.x == 0) mbar_arrive(bar_qempty + 8 * k);
        if (flags[1]) break;
    }
    // the producer has seen every load land (barrier 2 counts it too)
    asm volatile("bar.sync 2, %0;" ::"n"(C::THREADS) : "memory");
}

// CW consecutive floats (16-byte aligned when CW >= 4, else 8-byte) into registers.
template <int CW>
__device__ __forceinline__ void load_cols(const float* x, float (&v)[CW]) {
    if constexpr (CW % 4 == 0) {
#pragma unroll
        for (int c = 0; c < CW; c += 4) {
            const float4 t = *reinterpret_cast<const float4*>(x + c);
            v[c] = t.x;
            v[c + 1] = t.y;
            v[c + 2] = t.z;
            v[c + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < CW; c += 2) {
            const float2 t = *reinterpret_cast<const float2*>(x + c);
            v[c] = t.x;
            v[c + 1] = t.y;
        }
    }
}

// Split-K merge (mini_engine, "Custom CUDA kernels", v2 reduce): for each (s, h) with more
// than one piece, M = max_p m_p, w_p = l_p exp(m_p - M), out = sum_p w_p o_p / sum_p w_p.
// The shared-prefix partials (if any) take part as further pieces.
// One warp per (s, h) row, no shared memory: lane i weighs
// pieces i, i + 32, ... and holds D / 32 columns of every piece.  The first 2048 / D pieces'
// columns are loaded before the weights are known, so that in the common case (up to 16 pieces
// at head_dim 128) the merge after the piece kernel is one round trip to L2 for m, l and o
// together, then the store.
template <int D, bool BF16>
__global__ void __launch_bounds__(256, 2) splitk_merge_kernel(const DecodeParams p) {
    using F = F16x2<BF16>;
    constexpr int CW = D / 32;  // columns per lane: 2, 4 or 8
    constexpr int PRE = 64 / CW;  // pieces whose columns are loaded up front: 32, 16 or 8
    constexpr float kLn2 = 0.69314718055994531f;  // the prefix partials' m is base 2
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // once the dynamic grid has ended: its counter back to zero, and marked so, for the next call
    if (p.dyn_tag && blockIdx.x == 0 && threadIdx.x == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        *p.dyn_counter = 0;
        *p.dyn_tag = kDynTag;
    }
    const int row = blockIdx.x * (blockDim.x >> 5) + warp;  // s * Hq + h
    if (row >= p.num_seqs * p.n_q_heads) return;
    const int s = row / p.n_q_heads;
    int L = __ldg(p.context_lens + s);
    const int cap = min(table_row_tokens(p.max_blocks_per_seq, p.cpb_log2), p.prefix_tokens + p.cover_parts * p.part_tokens);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int n_parts = pieces_of(p, L);
    if (n_parts <= 1) return;  // written directly by the piece kernel
    // launched as a programmatic dependent of the piece kernel: its partials (and, through it, the
    // shared-prefix pass's) are complete and visible past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float* m = p.ws_m + (size_t)row * p.max_parts;
    const float* l = p.ws_l + (size_t)row * p.max_parts;
    const float* ob = p.ws_o + (size_t)row * p.max_parts * D + lane * CW;
    const int KP = p.pf_parts;

    float pre[PRE][CW];
#pragma unroll
    for (int i = 0; i < PRE; ++i) {
        if (i < n_parts) {
            load_cols<CW>(ob + (size_t)i * D, pre[i]);
        } else {
#pragma unroll
            for (int c = 0; c < CW; ++c) pre[i][c] = 0.f;
        }
    }
    float M = -INFINITY;
    for (int i = lane; i < n_parts; i += 32)
        if (l[i] > 0.f) M = fmaxf(M, m[i]);
    for (int k = lane; k < KP; k += 32)
        if (p.pf_l[(size_t)row * KP + k] > 0.f) M = fmaxf(M, p.pf_m[(size_t)row * KP + k] * kLn2);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float acc[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c) acc[c] = 0.f;
    float W = 0.f;
    for (int i0 = 0; i0 < n_parts; i0 += 32) {
        float wl = 0.f;
        if (i0 + lane < n_parts) {
            const float li = l[i0 + lane];
            if (li > 0.f) wl = li * __expf(m[i0 + lane] - M);
        }
        W += wl;
        const int nb = min(32, n_parts - i0);
        int j = 0;
        if (i0 == 0) {
#pragma unroll
            for (; j < PRE; ++j) {
                const float wj = __shfl_sync(0xffffffffu, wl, j);
#pragma unroll
                for (int c = 0; c < CW; ++c) acc[c] = fmaf(wj, pre[j][c], acc[c]);
            }
        }
#pragma unroll 4
        for (; j < nb; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            float v[CW];
            load_cols<CW>(ob + (size_t)(i0 + j) * D, v);
#pragma unroll
            for (int c = 0; c < CW; ++c) acc[c] = fmaf(wj, v[c], acc[c]);
        }
    }
    for (int k0 = 0; k0 < KP; k0 += 32) {
        float wl = 0.f;
        if (k0 + lane < KP) {
            const size_t i = (size_t)row * KP + k0 + lane;
            const float lk = p.pf_l[i];
            if (lk > 0.f) wl = lk * __expf(p.pf_m[i] * kLn2 - M);
        }
        W += wl;
        const int nb = min(32, KP - k0);
        for (int j = 0; j < nb; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            if (wj > 0.f) {
                float v[CW];
                load_cols<CW>(p.pf_o + ((size_t)row * KP + k0 + j) * D + lane * CW, v);
#pragma unroll
                for (int c = 0; c < CW; ++c) acc[c] = fmaf(wj, v[c], acc[c]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    const float inv = (W > 0.f) ? 1.f / W : 0.f;
    const int c0 = lane * CW;
    if (c0 < p.hd) {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + (size_t)row * p.hd + c0;
#pragma unroll
        for (int c = 0; c < CW; c += 2)
            reinterpret_cast<uint32_t*>(dst)[c / 2] = F::pack_rn(acc[c] * inv, acc[c + 1] * inv);
    }
}

}  // namespace pa
