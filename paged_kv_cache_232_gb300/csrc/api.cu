// api.cu -- the C ABI of libpagedattn (include/pagedattn.h): host-side validation, tensor
// maps for the paged caches, the decode dispatcher, the per-device error word, and the
// KV-cache write launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kv_write.cuh"
#include "rope_write.cuh"
#include "pa_launch.h"
#include "pagedattn.h"

// Error word written by the kernels (PA_DEVERR_* bits); one per device that loads the library.
__device__ unsigned g_pa_device_errors;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    unsigned* err = nullptr;  // device address of g_pa_device_errors
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up, done once with that device current.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PA_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_device_errors) != cudaSuccess) return PA_ERR_CUDA;
        d.err = static_cast<unsigned*>(p);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return PA_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over a paged cache [num_blocks, block_size, n_kv_heads, head_dim]: box of
// 64 columns x 1 head x 16 rows x 1 block, 128-byte swizzled (one TMA load moves one 128-byte
// column slab of one head's 16-token chunk; with block_size 32..128 the kernels address the
// chunk's rows inside its block by the row coordinate).  Out-of-range block ids read zeros.
int encode_cache_map(CUtensorMap* m, const void* base, int dtype, int64_t num_blocks, int block_size,
                     int n_kv_heads, int head_dim) {
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)n_kv_heads, (cuuint64_t)block_size,
                          (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_kv_heads * head_dim * 2,
                             (cuuint64_t)block_size * n_kv_heads * head_dim * 2};
    // one 16-token chunk of a block (an 8-token block is loaded whole, two per chunk)
    cuuint32_t box[4] = {64, 1, (cuuint32_t)(block_size < 16 ? block_size : 16), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int check_heads(int n_q_heads, int n_kv_heads, int head_dim, int block_size, int dtype) {
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return PA_ERR_SHAPE;
    const int G = n_q_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 96 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (head_dim == 256 && G > 4) return PA_ERR_UNSUPPORTED;  // decode keeps q for the group in registers
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
        return PA_ERR_UNSUPPORTED;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// head_dim the attention kernels are instantiated for: 96 runs in the 128-column kernels, the
// columns past 96 zero (the tensor maps fill them, q loads and output stores skip them)
int kernel_dim(int head_dim) { return head_dim == 96 ? 128 : head_dim; }

// log2 of the 16-token chunks per cache block; -1 for blocks of 8 tokens (two per chunk)
int cpb_log2_of(int block_size) {
    return block_size == 8 ? -1 : block_size == 16 ? 0 : block_size == 32 ? 1 : block_size == 64 ? 2 : 3;
}

int partition_or_default(int part) { return part > 0 ? part : PA_DEFAULT_PARTITION_TOKENS; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t m_off, l_off, o_off, ctl_off, total;
};

// A 256-byte control region (the dynamic grid's piece counter at byte 0, its tag at byte 8),
// then the m, l, o regions.  The control region sits at the start whatever the sizes, so that the
// counter a call leaves at zero is where the next call on the workspace looks for it.
WsLayout ws_layout(int num_seqs, int n_q_heads, int head_dim, int max_parts) {
    const size_t rows = (size_t)num_seqs * n_q_heads * max_parts;
    WsLayout w;
    w.ctl_off = 0;
    w.m_off = 256;
    w.l_off = w.m_off + align256(rows * sizeof(float));
    w.o_off = w.l_off + align256(rows * sizeof(float));
    w.total = w.o_off + align256(rows * head_dim * sizeof(float));
    return w;
}

// Shared argument checks of the decode entry points.
int check_decode(const void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* bt,
                 int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int n_q_heads, int n_kv_heads,
                 int head_dim, int block_size, int64_t num_blocks, int dtype) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
    int st = check_heads(n_q_heads, n_kv_heads, head_dim, block_size, dtype);
    if (st != PA_OK) return st;
    if (num_blocks > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !bt || !context_lens) return PA_ERR_NULL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
    return PA_OK;
}

// Partials of a shared-prefix pass that the decode folds into its merge (see pa_decode_shared_prefix).
struct PrefixPartials {
    int tokens;  // the decode streams tokens [tokens, L) of each sequence
    int parts;
    const float *m, *l, *o;
    int* dyn_counter;  // non-null: run the one-pass suffix as the dynamic grid over whole units,
                       // taking them from this counter (zeroed on the stream before the prefix pass)
};

// pa_decode_write: one new K/V row per sequence (row s of key / value) for slot_mapping[s].
struct NewRows {
    const void* key;
    const void* value;
    const int64_t* slot_mapping;
};

// The KV-write kernel over num_tokens rows of row_vecs 16-byte chunks.
int launch_kv_write(const void* key, const void* value, void* k_cache, void* v_cache, const int64_t* slot_mapping,
                    int64_t num_tokens, int row_vecs, int64_t num_blocks, int block_size, const DeviceState* dev,
                    cudaStream_t stream) {
    // one thread per 16-byte chunk of the (K row ++ V row) pair, at most 512 (then each loops)
    const int threads = 2 * row_vecs < 512 ? 2 * row_vecs : 512;
    const int64_t iters = (num_tokens + pa::kKvWriteRowsPerIter - 1) / pa::kKvWriteRowsPerIter;
    const int64_t max_grid = (int64_t)dev->sm_count * (2048 / threads);
    const int grid = (int)(iters < max_grid ? iters : max_grid);
    pa::kv_write_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), slot_mapping, num_tokens, row_vecs, num_blocks * block_size, dev->err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
                int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                int dtype, int part_tokens, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                const PrefixPartials* pf = nullptr, const NewRows* nr = nullptr) {
    int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                          n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (st != PA_OK || num_seqs == 0) return st;
    if (!std::isfinite(scale)) return PA_ERR_SHAPE;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != PA_OK) return st;

    pa::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.err = dev->err;
    p.num_seqs = num_seqs;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = (int)num_blocks;
    p.cpb_log2 = cpb_log2_of(block_size);
    p.qk_scale_log2 = scale * 1.4426950408889634f;
    p.hd = head_dim;
    if (pf) {
        p.prefix_tokens = pf->tokens;
        p.pf_parts = pf->parts;
        p.pf_m = pf->m;
        p.pf_l = pf->l;
        p.pf_o = pf->o;
    }
    const int units = num_seqs * n_kv_heads;
    int grid = units;
    bool reduce = false;
    if (part_tokens > 0) {
        if (part_tokens % (block_size < 16 ? 16 : block_size)) return PA_ERR_UNSUPPORTED;  // whole chunks and blocks
        if (max_context_len < 0 || (int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size)
            return PA_ERR_BOUNDS;
        // pieces cover the tokens past the shared prefix, if any
        const int streamed = max_context_len - std::min(max_context_len, p.prefix_tokens);
        const int max_parts = streamed > 0 ? (streamed + part_tokens - 1) / part_tokens : 1;
        if ((int64_t)units * max_parts > INT32_MAX) return PA_ERR_UNSUPPORTED;
        const WsLayout w = ws_layout(num_seqs, n_q_heads, kernel_dim(head_dim), max_parts);
        if (max_parts > 1) {
            if (!workspace || workspace_bytes < w.total) return PA_ERR_WORKSPACE;
            if (!aligned16(workspace)) return PA_ERR_ALIGN;
            char* base = static_cast<char*>(workspace);
            p.ws_m = reinterpret_cast<float*>(base + w.m_off);
            p.ws_l = reinterpret_cast<float*>(base + w.l_off);
            p.ws_o = reinterpret_cast<float*>(base + w.o_off);
            p.dyn_counter = reinterpret_cast<int*>(base + w.ctl_off);
            reduce = true;
        }
        p.part_tokens = part_tokens;
        p.max_parts = max_parts;
        p.cover_parts = max_parts;
        grid = units * max_parts;
        if (reduce && n_q_heads / n_kv_heads <= 2) {
            // the dynamic grid: one CTA per resident slot taking pieces from the counter, when
            // there are more pieces than slots; with fewer it would run the static grid's CTAs
            // plus the counter's upkeep.  Group sizes 1 and
            // 2 only: at 4 its piece loop spills registers and the static grid is faster (GB300,
            // 4 sequences of 32K tokens at 32 q / 8 KV heads: 113.7 against 105.5 us)
            const int resident = pa::decode_dyn_resident_ctas(dtype == PA_BF16, kernel_dim(head_dim),
                                                              n_q_heads / n_kv_heads);
            if (resident <= 0) return PA_ERR_CUDA;
            const int64_t slots = (int64_t)dev->sm_count * resident;
            if ((int64_t)grid > slots) {
                p.dyn = 1;
                grid = (int)slots;
                // tail pieces (batches of up to kDynTailMaxSeqs sequences, when the workspace has
                // room for the extra pieces): the last part_tokens of every context go in pieces
                // of a quarter of that, so the items handed out last are short and the CTAs end
                // together
                const int align = block_size < 16 ? 16 : block_size;
                const int tail_tokens = ((part_tokens / 4 + align - 1) / align) * align;
                const int tail_parts = max_parts - 1 + (part_tokens + tail_tokens - 1) / tail_tokens;
                const WsLayout wt = ws_layout(num_seqs, n_q_heads, kernel_dim(head_dim), tail_parts);
                if (num_seqs <= pa::kDynTailMaxSeqs && workspace_bytes >= wt.total &&
                    (int64_t)units * tail_parts <= INT32_MAX) {
                    char* base = static_cast<char*>(workspace);
                    p.ws_m = reinterpret_cast<float*>(base + wt.m_off);
                    p.ws_l = reinterpret_cast<float*>(base + wt.l_off);
                    p.ws_o = reinterpret_cast<float*>(base + wt.o_off);
                    p.dyn_counter = reinterpret_cast<int*>(base + wt.ctl_off);
                    p.tail_tokens = tail_tokens;
                    p.max_parts = tail_parts;
                }
                // The counter: after a shared-prefix pass zeroed here, in the stream, before the
                // launch.  Otherwise no zeroing: the merge kernel leaves it at zero with the tag
                // beside it set, for the next call on this workspace, and a call that finds no
                // tag (a fresh or reused workspace) hands the pieces out in a fixed order instead
                // (a 4-byte memset costs ~1.2 us of a ~55 us batch-64 decode on GB300).
                if (pf) {
                    if (cudaMemsetAsync(p.dyn_counter, 0, sizeof(int), stream) != cudaSuccess) return PA_ERR_CUDA;
                } else {
                    p.dyn_tag = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(p.dyn_counter) + 8);
                }
            }
        }
    } else if (pf && pf->dyn_counter) {
        // one piece per unit (the whole streamed context, written directly), handed out longest
        // first by the dynamic grid, whose CTAs take work off the SMs the prefix pass holds
        const int streamed = max_context_len - std::min(max_context_len, p.prefix_tokens);
        p.part_tokens = std::max(16, (streamed + 15) / 16 * 16);
        p.max_parts = 1;
        p.cover_parts = 1;
        p.dyn = 1;
        p.dyn_units = 1;
        p.dyn_counter = pf->dyn_counter;
        const int resident = pa::decode_dyn_resident_ctas(dtype == PA_BF16, kernel_dim(head_dim), n_q_heads / n_kv_heads);
        if (resident <= 0) return PA_ERR_CUDA;
        grid = (int)std::min<int64_t>((int64_t)dev->sm_count * resident, (int64_t)units);
    } else {
        p.part_tokens = 0;
        p.max_parts = 1;
        // longest-first order pays only when the grid is longer than one wave of resident CTAs,
        // and needs its scratch (lengths + a chunk-count histogram) to fit in the ring; from two
        // waves on, at group size 1 or 2, one CTA per resident slot runs a list of units
        // (decode_kernel_persistent: no start-up per unit, the next unit's loads overlap this
        // one's merge) when the lists fit
        const int resident = pa::decode_resident_ctas(dtype == PA_BF16, kernel_dim(head_dim), n_q_heads / n_kv_heads);
        const int64_t slots = (int64_t)dev->sm_count * resident;
        const int64_t nb = ((int64_t)max_blocks_per_seq * block_size + 15) / 16 + 2;
        const int ring = pa::decode_ring_bytes(kernel_dim(head_dim));
        p.lpt = (resident > 0 && units > slots && ((int64_t)num_seqs + nb) * 4 <= ring) ? 1 : 0;
        // (not after a shared-prefix pass: its CTAs hold some SMs at the start, and the persistent
        // grid's fixed unit lists cannot move work off those SMs; hardware dispatch can -- GB300,
        // mixed batch decode rows 64.2 -> 62.1 us)
        p.persist = (p.lpt && p.pf_parts == 0 && n_q_heads / n_kv_heads <= 2 && units >= 2 * slots &&
                     units <= (int64_t)pa::decode_list_max() * slots && (2 * (int64_t)num_seqs + 2 * nb) * 4 <= ring)
                        ? 1 : 0;
        if (p.persist) grid = (int)slots;
    }
    CUtensorMap tk, tv;
    if ((st = encode_cache_map(&tk, k_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    if ((st = encode_cache_map(&tv, v_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    if (nr) {
        // pa_decode_write: the persistent and the dynamic grids write each unit's new row
        // themselves, just before loading the chunk that holds it; the other grids get the
        // KV-write kernel launched first
        const int row_vecs = n_kv_heads * head_dim * 2 / 16;
        if (p.persist || p.dyn) {
            p.new_k = static_cast<const uint4*>(nr->key);
            p.new_v = static_cast<const uint4*>(nr->value);
            p.new_slots = nr->slot_mapping;
            p.k_cache_w = static_cast<uint4*>(const_cast<void*>(k_cache));
            p.v_cache_w = static_cast<uint4*>(const_cast<void*>(v_cache));
            p.row_vecs = row_vecs;
            p.n_slots = (long long)num_blocks * block_size;
        } else if ((st = launch_kv_write(nr->key, nr->value, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                         nr->slot_mapping, num_seqs, row_vecs, num_blocks, block_size, dev,
                                         stream)) != PA_OK) {
            return st;
        }
    }
    cudaError_t e = pa::launch_decode(dtype == PA_BF16, kernel_dim(head_dim), n_q_heads / n_kv_heads, p, tk, tv, grid, reduce,
                                      stream);
    // a piece grid whose merge did not launch has left the counter wherever it stopped: clear the
    // tag, so that the next call does not trust it
    if (e != cudaSuccess && p.dyn_tag) (void)cudaMemsetAsync(p.dyn_tag, 0, sizeof(unsigned long long), stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Dispatcher (mini_engine, "Custom CUDA kernels": split-K when few sequences or long
// contexts cannot fill the GPU, the one-pass kernel when there is enough parallelism).
// The thresholds are this library's, set from GB300 measurements: the one-pass kernel wins
// from two waves of (sequence, KV head) units on (and for contexts under 1024 tokens) once
// there is a unit per SM and contexts are at most 8192 tokens; otherwise split-K.  The piece length sizes the grid in whole waves of resident CTAs: taking
// every context at the maximum, n equal pieces per unit cost waves(n) x (piece(n) + 64), the
// 64 tokens standing for a CTA's pipeline start and its share of the merge (fitted to GB300
// timings of 32 units of 32K tokens: one full wave of 2352-token pieces beats two of 1184 by
// 3 % and 2.25 waves of 1024 by 10 %), and the plan takes the fewest pieces whose cost is
// within 2 % of the best.  Pieces are at least 256 tokens, so a workspace sized for the
// default piece fits every plan.
int plan(int64_t units, int max_context_len, int sm_count, int resident, int block_size, int group,
         int* part_tokens) {
    const int min_piece = PA_DEFAULT_PARTITION_TOKENS;
    if (part_tokens) *part_tokens = min_piece;
    if (max_context_len <= min_piece) return 1;
    const int64_t slots = (int64_t)sm_count * (resident > 0 ? resident : 1);
    const int64_t L = max_context_len;
    const int64_t align = block_size < 16 ? 16 : block_size;  // pieces hold whole chunks and blocks
    if (units >= sm_count && max_context_len <= 8192) {
        // between one and two waves of units the one-pass grid ends on a few long contexts
        // streaming alone; quarter-context pieces keep every SM busy to the end (GB300, 64
        // sequences of 100..2048 tokens: 62.2 us against 65.0 one-pass)
        if (units >= 2 * slots || max_context_len < 1024) return 1;
        int64_t piece = std::max<int64_t>(min_piece, ((L + 3) / 4 + align - 1) / align * align);
        // at group size 1 or 2 the split-K grid is dynamic (CTAs take pieces as they free up):
        // there pieces of at most 512 tokens balance best (GB300, 64 sequences of 100..4096 /
        // 100..8192 tokens: 97.3 / 179.2 us at 512 against 103.4 / 197.6 at a quarter context)
        if (group <= 2) piece = std::min<int64_t>(piece, 512);
        if (part_tokens) *part_tokens = (int)piece;
        return 2;
    }
    const int n_max = (int)std::min<int64_t>((L + min_piece - 1) / min_piece, 1024);
    int64_t best = INT64_MAX;
    for (int n = 2; n <= n_max; ++n) {
        const int64_t piece = std::max<int64_t>(min_piece, ((L + n - 1) / n + align - 1) / align * align);
        const int64_t ctas = units * ((L + piece - 1) / piece);
        best = std::min(best, (ctas + slots - 1) / slots * (piece + 64));
    }
    int chosen = min_piece;
    for (int n = 2; n <= n_max; ++n) {
        const int64_t piece = std::max<int64_t>(min_piece, ((L + n - 1) / n + align - 1) / align * align);
        const int64_t ctas = units * ((L + piece - 1) / piece);
        if ((ctas + slots - 1) / slots * (piece + 64) * 50 <= best * 51) {
            chosen = (int)piece;
            break;
        }
    }
    if (part_tokens) *part_tokens = chosen;
    return 2;
}

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_NULL: return "null pointer argument";
        case PA_ERR_SHAPE: return "inconsistent sizes";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_CUDA: return "CUDA call failed";
        case PA_ERR_BOUNDS: return "size out of range";
        case PA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case PA_ERR_WORKSPACE: return "split-K workspace missing or too small";
        default: return "unknown status";
    }
}

int pa_device_errors(int clear) {
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st != PA_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pa_device_errors, sizeof(v)) != cudaSuccess) return PA_ERR_CUDA;
    if (clear) {
        unsigned z = 0;
        if (cudaMemcpyToSymbol(g_pa_device_errors, &z, sizeof(z)) != cudaSuccess) return PA_ERR_CUDA;
    }
    return (int)v;
}

int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int n_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int dtype, void* stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_SHAPE;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    const int64_t row_bytes = (int64_t)n_kv_heads * head_dim * 2;
    if (row_bytes % 16) return PA_ERR_UNSUPPORTED;  // 16-byte chunks
    if (row_bytes / 16 > INT32_MAX / 2) return PA_ERR_SHAPE;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st != PA_OK) return st;
    return launch_kv_write(key, value, k_cache, v_cache, slot_mapping, num_tokens, (int)(row_bytes / 16), num_blocks,
                           block_size, dev, static_cast<cudaStream_t>(stream));
}

int pa_rope_table(float* out, int64_t max_position, int head_dim, double theta) {
    if (!out) return PA_ERR_NULL;
    if (max_position <= 0 || head_dim <= 0 || (head_dim & 1) || !(theta > 0.0)) return PA_ERR_SHAPE;
    const int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double f = std::pow(theta, -2.0 * (double)i / (double)head_dim);
        for (int64_t m = 0; m < max_position; ++m) {
            const double a = (double)m * f;
            out[m * head_dim + i] = (float)std::cos(a);
            out[m * head_dim + half + i] = (float)std::sin(a);
        }
    }
    return PA_OK;
}

int pa_rope_reshape_and_cache(void* q, const void* key, const void* value, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, const int64_t* positions, const float* cos_sin,
                              int64_t num_tokens, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, int64_t max_position, int dtype, void* stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        max_position <= 0 || (q && n_q_heads <= 0))
        return PA_ERR_SHAPE;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 96 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping || !positions || !cos_sin) return PA_ERR_NULL;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(cos_sin) ||
        (q && !aligned16(q)))
        return PA_ERR_ALIGN;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st != PA_OK) return st;
    const int pairs = head_dim / 16;
    const int units = (q ? n_q_heads * pairs : 0) + n_kv_heads * pairs + n_kv_heads * (head_dim / 8);
    const int threads = units >= 512 ? 512 : ((units + 31) / 32) * 32;
    // two rows per thread in flight once there are at least four rows per SM, else one (more CTAs)
    const int rows = num_tokens >= 4 * (int64_t)dev->sm_count ? 2 : 1;
    const int64_t iters = (num_tokens + rows - 1) / rows;
    const int64_t max_grid = (int64_t)dev->sm_count * (2048 / threads);
    const int grid = (int)(iters < max_grid ? iters : max_grid);
    auto launch = [&](auto kern) {
        kern<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<uint4*>(q), static_cast<const uint4*>(key), static_cast<const uint4*>(value),
            static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, positions, cos_sin, num_tokens,
            n_q_heads, n_kv_heads, num_blocks * block_size, max_position, dev->err);
    };
    const bool bf = dtype == PA_BF16;
    auto by_dim = [&](auto k64, auto k96, auto k128, auto k256) {
        if (head_dim == 256) launch(k256);
        else if (head_dim == 128) launch(k128);
        else if (head_dim == 96) launch(k96);
        else launch(k64);
    };
    if (rows == 2) {
        if (bf) by_dim(pa::rope_write_kernel<true, 64, 2>, pa::rope_write_kernel<true, 96, 2>,
                       pa::rope_write_kernel<true, 128, 2>, pa::rope_write_kernel<true, 256, 2>);
        else by_dim(pa::rope_write_kernel<false, 64, 2>, pa::rope_write_kernel<false, 96, 2>,
                    pa::rope_write_kernel<false, 128, 2>, pa::rope_write_kernel<false, 256, 2>);
    } else {
        if (bf) by_dim(pa::rope_write_kernel<true, 64, 1>, pa::rope_write_kernel<true, 96, 1>,
                       pa::rope_write_kernel<true, 128, 1>, pa::rope_write_kernel<true, 256, 1>);
        else by_dim(pa::rope_write_kernel<false, 64, 1>, pa::rope_write_kernel<false, 96, 1>,
                    pa::rope_write_kernel<false, 128, 1>, pa::rope_write_kernel<false, 256, 1>);
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int head_dim, int max_context_len,
                                int partition_tokens) {
    if (num_seqs <= 0 || n_q_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    const int part = partition_or_default(partition_tokens);
    const int max_parts = max_context_len > 0 ? (max_context_len + part - 1) / part : 1;
    if (max_parts <= 1) return 0;
    // room for the dynamic grid's tail pieces: at most three more than the uniform split
    return ws_layout(num_seqs, n_q_heads, kernel_dim(head_dim), max_parts + 3).total;
}

int pa_decode_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
                   int dtype, int* partition_tokens) {
    if (num_seqs < 0 || max_context_len < 0) return PA_ERR_SHAPE;
    int st = check_heads(n_q_heads, n_kv_heads, head_dim, block_size, dtype);
    if (st != PA_OK) return st;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != PA_OK) return st;
    const int resident = pa::decode_resident_ctas(dtype == PA_BF16, kernel_dim(head_dim), n_q_heads / n_kv_heads);
    if (resident <= 0) return PA_ERR_CUDA;
    return plan((int64_t)num_seqs * n_kv_heads, max_context_len, dev->sm_count, resident, block_size,
                n_q_heads / n_kv_heads, partition_tokens);
}

int pa_decode_v1(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int n_q_heads,
                 int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale, int dtype,
                 void* stream) {
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       max_blocks_per_seq * block_size, num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                       num_blocks, scale, dtype, 0, nullptr, 0, static_cast<cudaStream_t>(stream));
}

int pa_decode_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                     int max_context_len, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                     int block_size, int64_t num_blocks, float scale, int dtype, int partition_tokens,
                     void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                       partition_or_default(partition_tokens), workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
              int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
              int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (max_context_len < 0 || (int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size)
        return PA_ERR_BOUNDS;
    if (num_seqs == 0)  // an empty batch: the shapes checked, nothing launched
        return check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 0, n_q_heads,
                            n_kv_heads, head_dim, block_size, num_blocks, dtype);
    int part = 0;
    const int which = pa_decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_context_len, dtype,
                                     &part);
    if (which < 0) return which;
    if (which == 1)
        return pa_decode_v1(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                            n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype, stream);
    return pa_decode_splitk(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                            num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype, part,
                            workspace, workspace_bytes, stream);
}

int pa_decode_write(void* out, const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
                    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                    int dtype, const void* key, const void* value, const int64_t* slot_mapping, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (max_context_len < 0 || (int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size)
        return PA_ERR_BOUNDS;
    if (num_seqs == 0)  // an empty batch: the shapes checked, nothing launched
        return check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 0, n_q_heads,
                            n_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (!key || !value || !slot_mapping) return PA_ERR_NULL;
    if (!aligned16(key) || !aligned16(value)) return PA_ERR_ALIGN;
    int part = 0;
    const int which = pa_decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_context_len, dtype,
                                     &part);
    if (which < 0) return which;
    const NewRows nr{key, value, slot_mapping};
    if (which == 1)
        return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           max_blocks_per_seq * block_size, num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                           num_blocks, scale, dtype, 0, nullptr, 0, static_cast<cudaStream_t>(stream), nullptr, &nr);
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype, part,
                       workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, &nr);
}

static int prefill_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                        const int32_t* seq_lens, int num_chunks, int max_q_len, int n_q_heads, int n_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, float scale, int dtype, void* stream,
                        bool small_m) {
    if (num_chunks < 0 || max_q_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
    int st = check_heads(n_q_heads, n_kv_heads, head_dim, block_size, dtype);
    if (st != PA_OK) return st;
    if (num_blocks > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (num_chunks == 0 || max_q_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !query_start_loc || !seq_lens) return PA_ERR_NULL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
    if (!std::isfinite(scale)) return PA_ERR_SHAPE;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != PA_OK) return st;
    const int G = n_q_heads / n_kv_heads;
    pa::PrefillParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.query_start_loc = query_start_loc;
    p.seq_lens = seq_lens;
    p.err = dev->err;
    p.num_chunks = num_chunks;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = (int)num_blocks;
    p.cpb_log2 = cpb_log2_of(block_size);
    p.tiles_per_chunk = (int)(((int64_t)max_q_len * G + 127) / 128);
    p.max_q_len = max_q_len;
    p.qk_scale_log2 = scale * 1.4426950408889634f;
    p.hd = head_dim;
    if ((int64_t)p.tiles_per_chunk * num_chunks * n_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if ((st = encode_cache_map(&tk, k_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    if ((st = encode_cache_map(&tv, v_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    cudaError_t e = small_m ? pa::launch_prefill_small(dtype == PA_BF16, kernel_dim(head_dim), G, p, tk, tv,
                                                       static_cast<cudaStream_t>(stream))
                            : pa::launch_prefill(dtype == PA_BF16, kernel_dim(head_dim), G, p, tk, tv,
                                                 static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_prefill_chunk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                     const int32_t* seq_lens, int num_chunks, int max_q_len, int n_q_heads, int n_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, float scale, int dtype, void* stream) {
    return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, query_start_loc, seq_lens,
                        num_chunks, max_q_len, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                        stream, false);
}

int pa_prefill_chunk_small_m(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int num_chunks, int max_q_len, int n_q_heads, int n_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, float scale, int dtype, void* stream) {
    return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, query_start_loc, seq_lens,
                        num_chunks, max_q_len, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                        stream, true);
}

// ---- shared prefix --------------------------------------------------------------------------

// Layout of pa_decode_shared_prefix's workspace: the prefix pass's partials (m, l: [S * Hq][KP];
// o: [S * Hq][KP][kernel head_dim]; KP sized for the smallest piece), then the suffix's split-K
// region (pa_decode_workspace_size over the tokens past the prefix), each 256-byte aligned.
static constexpr int kMinPrefixPiece = 128;

static int prefix_tokens_used(int prefix_tokens, int max_context_len) {
    // whole 16-token chunks of the prefix within the longest context; the rest of a shared
    // prefix is streamed by each sequence's decode like its own tokens
    const int p = prefix_tokens < max_context_len ? prefix_tokens : max_context_len;
    return p > 0 ? (p / 16) * 16 : 0;
}

static WsLayout pf_layout(int num_seqs, int n_q_heads, int kdim, int parts) {
    return ws_layout(num_seqs, n_q_heads, kdim, parts);  // same three regions, one column per piece
}

size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int n_q_heads, int head_dim, int max_context_len,
                                              int prefix_tokens) {
    if (num_seqs <= 0 || n_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 || prefix_tokens < 0) return 0;
    const int P = prefix_tokens_used(prefix_tokens, max_context_len);
    if (P == 0) return pa_decode_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len, 0);
    const int kp = (P + kMinPrefixPiece - 1) / kMinPrefixPiece;
    return pf_layout(num_seqs, n_q_heads, kernel_dim(head_dim), kp).total +
           pa_decode_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len - P, 0);
}

int pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int max_context_len, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale, int dtype, int prefix_tokens,
                            int prefix_piece_tokens, void* workspace, size_t workspace_bytes, void* stream) {
    int st = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                          n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (st != PA_OK || num_seqs == 0) return st;
    const int64_t row_tokens = (int64_t)max_blocks_per_seq * block_size;
    if (max_context_len < 0 || max_context_len > row_tokens || prefix_tokens < 0 || prefix_tokens > row_tokens)
        return PA_ERR_BOUNDS;
    if (prefix_piece_tokens < 0 || prefix_piece_tokens % kMinPrefixPiece) return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PA_ERR_SHAPE;
    const int P = prefix_tokens_used(prefix_tokens, max_context_len);
    if (P == 0)  // nothing shared: the plain dispatcher, same workspace
        return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                         num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                         workspace_bytes, stream);
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != PA_OK) return st;
    const int G = n_q_heads / n_kv_heads;
    const int kdim = kernel_dim(head_dim);
    if (workspace_bytes < pa_decode_shared_prefix_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len,
                                                                 prefix_tokens) ||
        !workspace)
        return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGN;

    // the suffix: the dispatcher's plan over the tokens past the prefix.  A one-pass suffix at group
    // size 1 or 2 with more units than the dynamic grid's slots (batches of up to 256 sequences)
    // runs as that grid over whole units; its counter sits in the prefix region's control area and
    // is zeroed now, before the prefix pass, so that the suffix still launches as the pass's
    // programmatic dependent (GB300, mixed batch decode rows: 58.5-61.1 -> 57.0-58.6 us)
    const int resident = pa::decode_resident_ctas(dtype == PA_BF16, kdim, G);
    if (resident <= 0) return PA_ERR_CUDA;
    int part = 0;
    const int which = plan((int64_t)num_seqs * n_kv_heads, max_context_len - P, dev->sm_count, resident, block_size,
                           G, &part);
    int* dyn_counter = nullptr;
    if (which == 1 && G <= 2 && num_seqs <= pa::kDynTailMaxSeqs && (max_context_len - P) / 16 + 1 <= 8000) {
        const int dres = pa::decode_dyn_resident_ctas(dtype == PA_BF16, kdim, G);
        if (dres <= 0) return PA_ERR_CUDA;
        if ((int64_t)num_seqs * n_kv_heads > (int64_t)dev->sm_count * dres) {
            // the control area at the start of the prefix region (and of the workspace), before
            // the partials of any piece length; the tag beside the counter is cleared with it, since
            // this grid leaves the counter where its claims stopped (the next pa_decode on this
            // workspace then hands its pieces out in the fixed order)
            const WsLayout pw0 = pf_layout(num_seqs, n_q_heads, kdim, (P + kMinPrefixPiece - 1) / kMinPrefixPiece);
            dyn_counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + pw0.ctl_off);
            if (cudaMemsetAsync(dyn_counter, 0, 16, static_cast<cudaStream_t>(stream)) != cudaSuccess)
                return PA_ERR_CUDA;
        }
    }

    // the prefix pass: CTAs of (query-tile pair, KV head, piece); the default piece keeps about a
    // quarter of the SMs on it (its CTAs run beside the suffix decode, which starts at once), a
    // sixteenth when the suffix runs on the dynamic grid, whose CTAs take over the rest (GB300,
    // mixed batch decode rows: 57.0 us at 512-token pieces against 58.4 at 256)
    const int tiles = (int)(((int64_t)num_seqs * G + 127) / 128);
    const int pairs = (tiles + 1) / 2;
    int piece = prefix_piece_tokens;
    if (piece == 0) {
        const int64_t per_piece = (int64_t)pairs * n_kv_heads;
        const int64_t want = dyn_counter ? dev->sm_count / 16 : dev->sm_count / 4;
        const int64_t kp = std::max<int64_t>(1, (want + per_piece - 1) / per_piece);
        piece = (int)((((int64_t)P + kp - 1) / kp + 127) / 128 * 128);
        piece = std::max(piece, 256);
    }
    const int kp = (P + piece - 1) / piece;
    if ((int64_t)tiles * n_kv_heads * kp > INT32_MAX) return PA_ERR_UNSUPPORTED;
    const WsLayout pw = pf_layout(num_seqs, n_q_heads, kdim, (P + kMinPrefixPiece - 1) / kMinPrefixPiece);
    // the partials are laid out for kp pieces inside the region sized for the smallest piece
    const WsLayout pk = pf_layout(num_seqs, n_q_heads, kdim, kp);
    char* base = static_cast<char*>(workspace);
    float* pf_m = reinterpret_cast<float*>(base + pk.m_off);
    float* pf_l = reinterpret_cast<float*>(base + pk.l_off);
    float* pf_o = reinterpret_cast<float*>(base + pk.o_off);

    CUtensorMap tk, tv;
    if ((st = encode_cache_map(&tk, k_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    if ((st = encode_cache_map(&tv, v_cache, dtype, num_blocks, block_size, n_kv_heads, head_dim)) != PA_OK) return st;
    pa::PrefillParams pp{};
    pp.q = q;
    pp.block_tables = block_tables;
    pp.err = dev->err;
    pp.n_q_heads = n_q_heads;
    pp.n_kv_heads = n_kv_heads;
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.num_blocks = (int)num_blocks;
    pp.cpb_log2 = cpb_log2_of(block_size);
    pp.tiles_per_chunk = tiles;
    pp.qk_scale_log2 = scale * 1.4426950408889634f;
    pp.hd = head_dim;
    pp.context_lens = context_lens;
    pp.pf_m = pf_m;
    pp.pf_l = pf_l;
    pp.pf_o = pf_o;
    pp.num_seqs = num_seqs;
    pp.prefix_tokens = P;
    pp.piece_tokens = piece;
    pp.pf_parts = kp;
    cudaError_t e = pa::launch_prefix(dtype == PA_BF16, kdim, G, pp, tk, tv, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PA_ERR_CUDA;

    const PrefixPartials pin{P, kp, pf_m, pf_l, pf_o, dyn_counter};
    void* ws2 = base + pw.total;
    const size_t ws2_bytes = workspace_bytes - pw.total;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                       which == 2 ? part : 0, ws2, ws2_bytes, static_cast<cudaStream_t>(stream), &pin);
}

}  // extern "C"
