/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline / reference arm may load this library.  It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it computes is the plain definition of attention over a block-paged
 * cache, written out loop by loop:
 *
 *  - Address translation (MiniLLM Runtime, "Core class relationships"): token t
 *    of a sequence lives in logical block t / block_size at offset
 *    t % block_size; the block table maps the logical block to a physical block,
 *    and the cache [num_blocks, block_size, n_kv_heads, head_dim] is read there,
 *    without first copying the sequence into a contiguous tensor.
 *  - Slot mapping for the cache write (miniserve, "Engine"):
 *    slot = block_id * block_size + offset; rows whose slot is -1 are padding and
 *    are skipped (mini_engine, "Custom CUDA kernels", KV-cache write).
 *  - Decode attention (mini_engine, "Custom CUDA kernels", paged decode
 *    attention): for each sequence and query head h, with KV head h / G
 *    (query heads of one GQA group share one KV head),
 *        s_t = scale * sum_d q[h, d] K_t[d],  t < context_len,
 *        o   = sum_t exp(s_t - max s) V_t / sum_t exp(s_t - max s).
 *  - Split-K partitions (same section, "v2"): the same over 256-token pieces of
 *    the context, each returning its own max m_p, exp-sum l_p and normalised
 *    output o_p; pieces merge with weights l_p * exp(m_p - max_p m_p).
 *  - Prefill chunk (mini_engine paged prefill; miniserve "Engine", bottom-right
 *    causal mask): query row j of a chunk of q_len rows whose kv length is
 *    kv_len sees keys t <= (kv_len - q_len) + j.
 *  - Rotary position embedding fused into the KV write (mini_engine, "Roadmap":
 *    the rotary embedding is to be applied inside the KV-cache write; "Features":
 *    Qwen3 with RoPE): the
 *    textbook rotation of each dimension pair (i, i + head_dim/2) by m * f_i.
 *  - Materialise-then-attend (MiniLLM Runtime, "Key benchmark results"): copy the
 *    sequence's K/V into contiguous arrays first, then run the same textbook
 *    attention; used only as an invariant (paged == contiguous).
 *
 * Every sum is accumulated in double; inputs are fp16 / bf16 bit patterns
 * widened exactly to double.  exp() is the C library's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PAO_F16 0
#define PAO_BF16 1
#define PAO_MAX_HEAD_DIM 1024

#define PAO_OK 0
#define PAO_EARG -1
#define PAO_EBOUNDS -2

/* ---- number formats ------------------------------------------------------ */

/* Exact value of an IEEE binary16 bit pattern. */
static double pao_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* Exact value of a bfloat16 bit pattern (the upper half of a binary32). */
static double pao_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double pao_to_double(uint16_t bits, int dtype) {
    return dtype == PAO_BF16 ? pao_bf16_to_double(bits) : pao_f16_to_double(bits);
}

/*
 * Round a double to the nearest representable value of the 16-bit format
 * (ties to even), returning the bit pattern.  Done by brute force on the
 * value grid: find the binade, scale to an integer number of units, round.
 */
uint16_t pao_from_double(double x, int dtype) {
    int mant_bits = dtype == PAO_BF16 ? 7 : 10;
    int exp_bits = dtype == PAO_BF16 ? 8 : 5;
    int bias = (1 << (exp_bits - 1)) - 1;
    int emin = 1 - bias;              /* smallest normal exponent */
    int emax = bias;                  /* largest normal exponent */
    uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    uint16_t exp_all = (uint16_t)(((1u << exp_bits) - 1) << mant_bits);
    if (isnan(x)) return (uint16_t)(exp_all | (1u << (mant_bits - 1)));
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                     /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
    int ue = e - 1;
    if (ue < emin) ue = emin;         /* subnormal range shares the emin unit */
    double unit = ldexp(1.0, ue - mant_bits);
    double n = a / unit;              /* exact: power-of-two scaling */
    double fl = floor(n);
    double r = n - fl;
    double k = fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) == 1.0)) k = fl + 1.0;
    /* k counts units of 2^(ue-mant_bits); k may reach 2^(mant_bits+1) (carry into next binade) */
    double val = k * unit;
    if (val > ldexp(2.0 - ldexp(1.0, -mant_bits), emax)) return (uint16_t)(sign | exp_all); /* overflow */
    if (val == 0.0) return sign;
    /* re-encode val exactly */
    frexp(val, &e);
    ue = e - 1;
    if (ue < emin) { /* subnormal */
        uint32_t m = (uint32_t)(val / ldexp(1.0, emin - mant_bits));
        return (uint16_t)(sign | m);
    }
    uint32_t m = (uint32_t)(val / ldexp(1.0, ue - mant_bits)) - (1u << mant_bits);
    return (uint16_t)(sign | ((uint32_t)(ue + bias) << mant_bits) | m);
}

void pao_round_array(const double* x, int64_t n, int dtype, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = pao_from_double(x[i], dtype);
}

void pao_widen_array(const uint16_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = pao_to_double(bits[i], dtype);
}

/* ---- KV-cache write ------------------------------------------------------ */

/*
 * k_cache / v_cache: [num_blocks, block_size, n_kv_heads, head_dim] bit patterns.
 * key / value: [num_tokens, n_kv_heads, head_dim].  Row i goes to slot
 * slot_mapping[i] (block slot / block_size, offset slot % block_size); -1 skips.
 * Returns PAO_EBOUNDS (and writes nothing for that row) for a slot outside the pool.
 */
int pao_kv_write(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* key, const uint16_t* value,
                 const int64_t* slot_mapping, int64_t num_tokens, int n_kv_heads, int head_dim,
                 int block_size, int64_t num_blocks) {
    int status = PAO_OK;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_blocks * block_size) { status = PAO_EBOUNDS; continue; }
        int64_t block = slot / block_size, offset = slot % block_size;
        for (int h = 0; h < n_kv_heads; ++h)
            for (int d = 0; d < head_dim; ++d) {
                int64_t dst = ((block * block_size + offset) * n_kv_heads + h) * head_dim + d;
                int64_t src = (i * n_kv_heads + h) * head_dim + d;
                k_cache[dst] = key[src];
                v_cache[dst] = value[src];
            }
    }
    return status;
}

/* ---- rotary position embedding (fused into the KV write) ------------------ */

/*
 * Rotary position embedding (mini_engine, "Features": the Qwen3 decoder uses RoPE;
 * "Roadmap": the rotary embedding applied inside the KV-cache write).  The textbook rotation, in the
 * rotate-half pairing: with half = head_dim / 2 and f_i = theta^(-2 i / head_dim), a row x of
 * a token at position m becomes, for i < half,
 *     x'[i]        = x[i] cos(m f_i) - x[i + half] sin(m f_i)
 *     x'[i + half] = x[i + half] cos(m f_i) + x[i] sin(m f_i).
 * pao_rope_exact rotates doubles (no rounding; for the invariants); pao_rope_kv_write works on
 * 16-bit rows and rounds each result once, to nearest even.
 */
void pao_rope_exact(const double* x, double* out, int head_dim, double m, double theta) {
    const int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double f = pow(theta, -2.0 * (double)i / (double)head_dim);
        const double c = cos(m * f), sn = sin(m * f);
        const double x0 = x[i], x1 = x[i + half];
        out[i] = x0 * c - x1 * sn;
        out[i + half] = x1 * c + x0 * sn;
    }
}

static void pao_rope_bits(const uint16_t* x, uint16_t* out, int head_dim, int64_t m, double theta, int dtype) {
    double in[PAO_MAX_HEAD_DIM], rot[PAO_MAX_HEAD_DIM];
    for (int e = 0; e < head_dim; ++e) in[e] = pao_to_double(x[e], dtype);
    pao_rope_exact(in, rot, head_dim, (double)m, theta);
    for (int e = 0; e < head_dim; ++e) out[e] = pao_from_double(rot[e], dtype);
}

/*
 * Fused rotary embedding + KV write.  For each row i with positions[i] in [0, max_position):
 * every head of q (when q is not NULL, [num_tokens, n_q_heads, head_dim]) is rotated in place;
 * if slot_mapping[i] != -1 the rotated key row goes to k_cache and the value row to v_cache at
 * that slot, exactly as pao_kv_write places rows.  A row whose position is out of range is
 * left untouched (status PAO_EBOUNDS); a slot outside the pool drops the row's write (same).
 */
int pao_rope_kv_write(uint16_t* q, uint16_t* k_cache, uint16_t* v_cache, const uint16_t* key,
                      const uint16_t* value, const int64_t* slot_mapping, const int64_t* positions,
                      int64_t num_tokens, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                      int64_t num_blocks, int64_t max_position, double theta, int dtype) {
    if (head_dim <= 0 || head_dim > PAO_MAX_HEAD_DIM || head_dim % 2) return PAO_EARG;
    int status = PAO_OK;
    uint16_t rot[PAO_MAX_HEAD_DIM];
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t m = positions[i];
        if (m < 0 || m >= max_position) { status = PAO_EBOUNDS; continue; }
        if (q) {
            for (int h = 0; h < n_q_heads; ++h) {
                uint16_t* row = q + (i * n_q_heads + h) * head_dim;
                pao_rope_bits(row, rot, head_dim, m, theta, dtype);
                memcpy(row, rot, (size_t)head_dim * sizeof(uint16_t));
            }
        }
        const int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_blocks * block_size) { status = PAO_EBOUNDS; continue; }
        const int64_t block = slot / block_size, offset = slot % block_size;
        for (int h = 0; h < n_kv_heads; ++h) {
            const int64_t dst = ((block * block_size + offset) * n_kv_heads + h) * head_dim;
            const int64_t src = (i * n_kv_heads + h) * head_dim;
            pao_rope_bits(key + src, k_cache + dst, head_dim, m, theta, dtype);
            for (int d = 0; d < head_dim; ++d) v_cache[dst + d] = value[src + d];
        }
    }
    return status;
}

/* ---- paged gather of one token's K or V row ------------------------------ */

typedef struct {
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    int n_kv_heads, head_dim, block_size;
    int64_t num_blocks;
    int dtype;
} pao_cache;

/* Physical element index of (token t of the sequence with block-table row bt, kv head g, dim 0). */
static int pao_row_index(const pao_cache* c, const int32_t* bt, int64_t t, int g, int64_t* idx) {
    int64_t logical_block = t / c->block_size;
    int64_t offset = t % c->block_size;
    int64_t phys = bt[logical_block];
    if (phys < 0 || phys >= c->num_blocks) return PAO_EBOUNDS;
    *idx = ((phys * c->block_size + offset) * c->n_kv_heads + g) * c->head_dim;
    return PAO_OK;
}

/*
 * Attention of one query vector over tokens [t0, t1) of one sequence, keys
 * visible per the caller's range.  Writes o[head_dim] (normalised), and the
 * softmax statistics m = max s_t, l = sum exp(s_t - m).  weights (optional,
 * length t1 - t0) receives exp(s_t - m) / l.  An empty range gives o = 0,
 * m = -inf, l = 0.
 */
static int pao_attend(const pao_cache* c, const int32_t* bt, const double* qv, int g, int64_t t0, int64_t t1,
                      double scale, double* o, double* m_out, double* l_out, double* weights) {
    int D = c->head_dim;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (t1 <= t0) { *m_out = -INFINITY; *l_out = 0.0; return PAO_OK; }
    int64_t n = t1 - t0;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!s) return PAO_EARG;
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        int64_t idx = 0;
        if (pao_row_index(c, bt, t, g, &idx) != PAO_OK) { free(s); return PAO_EBOUNDS; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qv[d] * pao_to_double(c->k_cache[idx + d], c->dtype);
        s[t - t0] = scale * dot;
        if (s[t - t0] > m) m = s[t - t0];
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        double p = exp(s[t - t0] - m);
        s[t - t0] = p;
        l += p;
    }
    for (int64_t t = t0; t < t1; ++t) {
        int64_t idx = 0;
        pao_row_index(c, bt, t, g, &idx);
        double p = s[t - t0];
        for (int d = 0; d < D; ++d) o[d] += p * pao_to_double(c->v_cache[idx + d], c->dtype);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    if (weights)
        for (int64_t t = 0; t < n; ++t) weights[t] = s[t] / l;
    *m_out = m;
    *l_out = l;
    free(s);
    return PAO_OK;
}

/* ---- decode -------------------------------------------------------------- */

/*
 * out: [num_seqs, n_q_heads, head_dim] doubles.
 * q: [num_seqs, n_q_heads, head_dim] bits.  block_tables: [num_seqs, max_blocks_per_seq].
 * weights (optional): [num_seqs, n_q_heads, max_blocks_per_seq * block_size] softmax weights,
 * zero past the context.
 */
int pao_decode(double* out, double* weights, const uint16_t* q, const uint16_t* k_cache,
               const uint16_t* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* context_lens, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
               int block_size, int64_t num_blocks, double scale, int dtype) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads || head_dim <= 0 || head_dim > PAO_MAX_HEAD_DIM) return PAO_EARG;
    pao_cache c = {k_cache, v_cache, n_kv_heads, head_dim, block_size, num_blocks, dtype};
    int G = n_q_heads / n_kv_heads;
    int64_t wlen = (int64_t)max_blocks_per_seq * block_size;
    int status = PAO_OK;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int s = 0; s < num_seqs; ++s)
        for (int h = 0; h < n_q_heads; ++h) {
            int64_t L = context_lens[s];
            double qv[PAO_MAX_HEAD_DIM];
            double m, l;
            for (int d = 0; d < head_dim; ++d)
                qv[d] = pao_to_double(q[((int64_t)s * n_q_heads + h) * head_dim + d], dtype);
            double* o = out + ((int64_t)s * n_q_heads + h) * head_dim;
            double* w = weights ? weights + ((int64_t)s * n_q_heads + h) * wlen : NULL;
            if (w) for (int64_t t = 0; t < wlen; ++t) w[t] = 0.0;
            if (L > wlen) L = wlen;
            int st = pao_attend(&c, block_tables + (int64_t)s * max_blocks_per_seq, qv, h / G, 0, L, scale,
                                o, &m, &l, w);
            if (st != PAO_OK) {
#pragma omp critical
                status = st;
            }
        }
    return status;
}

/*
 * Split-K pieces: piece p covers tokens [p*P, min((p+1)*P, L)).
 * m, l: [num_seqs, n_q_heads, max_parts]; o: [num_seqs, n_q_heads, max_parts, head_dim].
 * Pieces past the context get m = -inf, l = 0, o = 0.
 */
int pao_decode_partitions(double* m, double* l, double* o, const uint16_t* q, const uint16_t* k_cache,
                          const uint16_t* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int n_q_heads, int n_kv_heads,
                          int head_dim, int block_size, int64_t num_blocks, double scale, int dtype,
                          int partition_tokens, int max_parts) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads || partition_tokens <= 0 || head_dim <= 0 ||
        head_dim > PAO_MAX_HEAD_DIM)
        return PAO_EARG;
    pao_cache c = {k_cache, v_cache, n_kv_heads, head_dim, block_size, num_blocks, dtype};
    int G = n_q_heads / n_kv_heads;
    int status = PAO_OK;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int s = 0; s < num_seqs; ++s)
        for (int h = 0; h < n_q_heads; ++h) {
            double qv[PAO_MAX_HEAD_DIM];
            for (int d = 0; d < head_dim; ++d)
                qv[d] = pao_to_double(q[((int64_t)s * n_q_heads + h) * head_dim + d], dtype);
            int64_t L = context_lens[s];
            for (int p = 0; p < max_parts; ++p) {
                int64_t t0 = (int64_t)p * partition_tokens;
                int64_t t1 = t0 + partition_tokens;
                if (t1 > L) t1 = L;
                int64_t k = ((int64_t)s * n_q_heads + h) * max_parts + p;
                int st = pao_attend(&c, block_tables + (int64_t)s * max_blocks_per_seq, qv, h / G, t0, t1,
                                    scale, o + k * head_dim, &m[k], &l[k], NULL);
                if (st != PAO_OK) {
#pragma omp critical
                    status = st;
                }
            }
        }
    return status;
}

/*
 * Merge of split-K pieces: M = max_p m_p, w_p = l_p exp(m_p - M),
 * o = sum_p w_p o_p / sum_p w_p.  out: [rows, head_dim]; rows = num_seqs * n_q_heads.
 */
void pao_merge_partitions(double* out, const double* m, const double* l, const double* o, int64_t rows,
                          int max_parts, int head_dim) {
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < max_parts; ++p)
            if (m[r * max_parts + p] > M) M = m[r * max_parts + p];
        double W = 0.0;
        for (int d = 0; d < head_dim; ++d) out[r * head_dim + d] = 0.0;
        if (M == -INFINITY) continue;
        for (int p = 0; p < max_parts; ++p) {
            double lp = l[r * max_parts + p];
            if (lp == 0.0) continue;
            double w = lp * exp(m[r * max_parts + p] - M);
            W += w;
            for (int d = 0; d < head_dim; ++d) out[r * head_dim + d] += w * o[(r * max_parts + p) * head_dim + d];
        }
        for (int d = 0; d < head_dim; ++d) out[r * head_dim + d] /= W;
    }
}

/* ---- prefill chunk --------------------------------------------------------- */

/*
 * out: [total_q, n_q_heads, head_dim] doubles; q: [total_q, n_q_heads, head_dim] bits.
 * Chunk c owns query rows [query_start_loc[c], query_start_loc[c+1]); its kv length
 * is seq_lens[c] (cached context plus the chunk itself, already in the cache).
 * Row j of chunk c attends to keys 0 .. (seq_lens[c] - q_len) + j.
 */
int pao_prefill_chunk(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                      const int32_t* seq_lens, int num_chunks, int n_q_heads, int n_kv_heads, int head_dim,
                      int block_size, int64_t num_blocks, double scale, int dtype) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads || head_dim <= 0 || head_dim > PAO_MAX_HEAD_DIM) return PAO_EARG;
    pao_cache c = {k_cache, v_cache, n_kv_heads, head_dim, block_size, num_blocks, dtype};
    int G = n_q_heads / n_kv_heads;
    int status = PAO_OK;
    for (int ch = 0; ch < num_chunks; ++ch) {
        int64_t r0 = query_start_loc[ch], r1 = query_start_loc[ch + 1];
        int64_t q_len = r1 - r0, kv_len = seq_lens[ch];
        if (kv_len < q_len || kv_len > (int64_t)max_blocks_per_seq * block_size) return PAO_EARG;
        int64_t ctx = kv_len - q_len;
        const int32_t* bt = block_tables + (int64_t)ch * max_blocks_per_seq;
#pragma omp parallel for collapse(2) schedule(dynamic)
        for (int64_t r = r0; r < r1; ++r)
            for (int h = 0; h < n_q_heads; ++h) {
                double qv[PAO_MAX_HEAD_DIM];
                double m, l;
                for (int d = 0; d < head_dim; ++d)
                    qv[d] = pao_to_double(q[(r * n_q_heads + h) * head_dim + d], dtype);
                int64_t j = r - r0;
                int st = pao_attend(&c, bt, qv, h / G, 0, ctx + j + 1, scale,
                                    out + (r * n_q_heads + h) * head_dim, &m, &l, NULL);
                if (st != PAO_OK) {
#pragma omp critical
                    status = st;
                }
            }
    }
    return status;
}

/* ---- materialise, then attend ---------------------------------------------- */

/*
 * The baseline the direct paged read replaces: for each sequence, copy its
 * context into contiguous K[L][Hkv][D], V[L][Hkv][D] arrays first, then run
 * textbook softmax attention on those arrays.  Same output layout as pao_decode.
 */
int pao_naive_contiguous(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                         int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, double scale, int dtype) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads) return PAO_EARG;
    int G = n_q_heads / n_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t L = context_lens[s];
        int64_t row = (int64_t)n_kv_heads * head_dim;
        double* K = (double*)malloc(sizeof(double) * (size_t)(L * row + 1));
        double* V = (double*)malloc(sizeof(double) * (size_t)(L * row + 1));
        double* sc = (double*)malloc(sizeof(double) * (size_t)(L + 1));
        if (!K || !V || !sc) { free(K); free(V); free(sc); return PAO_EARG; }
        /* materialise: walk the block table block by block */
        int64_t t = 0;
        for (int b = 0; t < L; ++b) {
            int64_t phys = block_tables[(int64_t)s * max_blocks_per_seq + b];
            if (phys < 0 || phys >= num_blocks) { free(K); free(V); free(sc); return PAO_EBOUNDS; }
            for (int off = 0; off < block_size && t < L; ++off, ++t)
                for (int64_t e = 0; e < row; ++e) {
                    int64_t src = (phys * block_size + off) * row + e;
                    K[t * row + e] = pao_to_double(k_cache[src], dtype);
                    V[t * row + e] = pao_to_double(v_cache[src], dtype);
                }
        }
        for (int h = 0; h < n_q_heads; ++h) {
            int g = h / G;
            const uint16_t* qh = q + ((int64_t)s * n_q_heads + h) * head_dim;
            double* o = out + ((int64_t)s * n_q_heads + h) * head_dim;
            double mx = -INFINITY, den = 0.0;
            for (int64_t i = 0; i < L; ++i) {
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += pao_to_double(qh[d], dtype) * K[i * row + g * head_dim + d];
                sc[i] = dot * scale;
                if (sc[i] > mx) mx = sc[i];
            }
            for (int64_t i = 0; i < L; ++i) { sc[i] = exp(sc[i] - mx); den += sc[i]; }
            for (int d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int64_t i = 0; i < L; ++i) acc += sc[i] * V[i * row + g * head_dim + d];
                o[d] = L ? acc / den : 0.0;
            }
        }
        free(K); free(V); free(sc);
    }
    return PAO_OK;
}

/* Threads the OpenMP loops use from now on (the bench times the oracle on one core as well as on
 * all of them); no effect on any result: every row is computed the same way by whichever thread. */
void pao_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int pao_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
