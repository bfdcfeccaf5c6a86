/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV decode
 * attention and its two copy companions (append one token, copy blocks).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path: it has its own element decoding, its own indexing and its own loops.
 *
 * Pages this file restates (cited by title and section):
 *   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析"
 *            - the standard attention formula softmax(QK^T / sqrt(d_k)) V
 *            - the multi-pass softmax it describes (max pass, sum pass,
 *              normalise pass)
 *            - the OnlineSoftmax recurrence for M_new, L_new and O_new
 *            - PagedAttention: per-sequence pages addressed via a page table
 *            - swap_blocks(src_kv_cache, dst_kv_cache, src_to_dst), where
 *              src_to_dst[i] = j copies source block i to target block j
 *   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
 *            PagedAttention 显存物理布局深度剖析"
 *            - section 一: KV-cache size formula 2*2*n_layers*n_heads*d*s*b
 *            - section 二.2: logical blocks of 16 tokens mapped to physical
 *              blocks through a block table; a new block on a full page
 *            - section 三: append_token / allocator walkthrough
 *   [OPT]    "vLLM中FlashAttention与KVCache优化解析"
 *            - "关键公式推导" (the M and L merge) and "Block Table 管理"
 *            - "Swap Blocks 机制": Key and Value caches copied separately
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - GQA: query head h reads KV head h / (n_heads / n_kv_heads)
 *     (contiguous groups; [SWAP] only says several query heads share one
 *     KV head through indexing).
 *   - context length 0 gives an all-zero output row.
 *   - the caller passes `scale` (configs use 1/sqrt(d)).
 *
 * Parity status: every function here is pinned by tests under tests/
 * (library routines, closed forms, invariants and the pages' printed
 * examples); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element type codes of the oracle's own (they happen to match the usual
 * order f16, bf16, f32, f64 but are defined here independently). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_F64 = 3 };

enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 2, ORC_NO_MEM = 3 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 is zero/subnormal (fraction * 2^-24), exponent 31 is
 * infinity (fraction 0) or NaN. */
double orc_f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Exponent 0 is zero/subnormal (fraction * 2^-133), exponent 255 is
 * infinity or NaN. */
double orc_bf16_bits_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134);
    return sign ? -mag : mag;
}

/* Read element `i` of a buffer holding elements of type `dtype`. */
static double orc_load(const void* base, size_t i, int dtype)
{
    if (dtype == ORC_F16) {
        uint16_t v;
        memcpy(&v, (const char*)base + 2 * i, 2);
        return orc_f16_bits_to_double(v);
    }
    if (dtype == ORC_BF16) {
        uint16_t v;
        memcpy(&v, (const char*)base + 2 * i, 2);
        return orc_bf16_bits_to_double(v);
    }
    if (dtype == ORC_F32) {
        float v;
        memcpy(&v, (const char*)base + 4 * i, 4);
        return (double)v;
    }
    {
        double v;
        memcpy(&v, (const char*)base + 8 * i, 8);
        return v;
    }
}

/* Convert a whole buffer (used by tests to pin the decoders). */
void orc_decode_elements(double* out, const void* in, size_t n, int dtype)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = orc_load(in, i, dtype);
}

/* [LAYOUT] section 一, KV-cache size formula: 2 (K and V) * bytes per
 * element * n_layers * n_heads * d_head * seq_len * batch.  The page uses 2
 * bytes per element (FP16). */
uint64_t orc_kv_cache_bytes(uint64_t n_layers, uint64_t n_heads, uint64_t d_head,
                            uint64_t seq_len, uint64_t batch, uint64_t elem_bytes)
{
    return 2u * elem_bytes * n_layers * n_heads * d_head * seq_len * batch;
}

/* Shared argument checks of the attention oracles. */
static int orc_check(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* seq_ids, int n_sel,
                     int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                     int block_size, int num_blocks)
{
    if (num_seqs < 0 || n_sel < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0)
        return ORC_BAD_ARG;
    if (n_heads % n_kv_heads != 0)
        return ORC_BAD_ARG;
    for (int r = 0; r < n_sel; ++r) {
        int s = seq_ids ? seq_ids[r] : r;
        if (s < 0 || s >= num_seqs)
            return ORC_BAD_INDEX;
        int n = context_lens[s];
        if (n < 0 || (int64_t)n > (int64_t)max_blocks_per_seq * block_size)
            return ORC_BAD_INDEX;
        int nb = (n + block_size - 1) / block_size;
        for (int j = 0; j < nb; ++j) {
            int p = block_tables[(size_t)s * max_blocks_per_seq + j];
            if (p < 0 || p >= num_blocks)
                return ORC_BAD_INDEX;
        }
    }
    return ORC_OK;
}

/* Element index of component i of the K (or V) vector of logical token t of
 * sequence s for KV head kvh.  [SWAP] PagedAttention / [LAYOUT] section 二.2:
 * logical block t / B of sequence s lives in physical block
 * block_tables[s][t / B]; inside it the token sits at row t % B.  Pool layout
 * [num_blocks, block_size, n_kv_heads, head_dim]. */
static size_t orc_kv_index(const int32_t* block_tables, int max_blocks_per_seq, int s, int t,
                           int kvh, int i, int n_kv_heads, int head_dim, int block_size)
{
    size_t p = (size_t)block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
    size_t row = (size_t)(t % block_size);
    return ((p * block_size + row) * n_kv_heads + kvh) * head_dim + i;
}

/*
 * The plain definition: for every selected sequence s and query head h,
 *     x_t = scale * sum_i q[s,h,i] * K_t[i]          (t < context_lens[s])
 *     o   = sum_t softmax(x)_t * V_t
 * with softmax taken the way [SWAP] describes the traditional method: one
 * pass for the maximum, one for the sum of exponentials, one to normalise.
 *
 *   out     : fp64 [n_sel, n_heads, head_dim]  (row r is sequence seq_ids[r];
 *             seq_ids == NULL selects 0..n_sel-1)
 *   q       : [num_seqs, n_heads, head_dim] of `dtype`
 *   k_pool, v_pool : [num_blocks, block_size, n_kv_heads, head_dim] of `dtype`
 *   block_tables   : int32 [num_seqs, max_blocks_per_seq]
 *   context_lens   : int32 [num_seqs]
 * Returns ORC_OK, or an error code without touching `out` further.
 */
int orc_paged_decode_two_pass(double* out, const void* q, const void* k_pool, const void* v_pool,
                              int dtype, const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, const int32_t* seq_ids, int n_sel,
                              int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                              int block_size, int num_blocks, double scale)
{
    int rc = orc_check(block_tables, max_blocks_per_seq, context_lens, seq_ids, n_sel, num_seqs,
                       n_heads, n_kv_heads, head_dim, block_size, num_blocks);
    if (rc != ORC_OK)
        return rc;
    int group = n_heads / n_kv_heads;
    for (int r = 0; r < n_sel; ++r) {
        int s = seq_ids ? seq_ids[r] : r;
        int n = context_lens[s];
        for (int h = 0; h < n_heads; ++h) {
            double* o = out + ((size_t)r * n_heads + h) * head_dim;
            for (int i = 0; i < head_dim; ++i)
                o[i] = 0.0;
            if (n == 0)
                continue;
            int kvh = h / group;
            double* x = (double*)malloc(sizeof(double) * (size_t)n);
            if (!x)
                return ORC_NO_MEM;
            /* scores */
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int i = 0; i < head_dim; ++i) {
                    double qi = orc_load(q, ((size_t)s * n_heads + h) * head_dim + i, dtype);
                    double ki = orc_load(k_pool,
                                         orc_kv_index(block_tables, max_blocks_per_seq, s, t, kvh,
                                                      i, n_kv_heads, head_dim, block_size),
                                         dtype);
                    acc += qi * ki;
                }
                x[t] = scale * acc;
            }
            /* pass 1: maximum */
            double m = x[0];
            for (int t = 1; t < n; ++t)
                if (x[t] > m)
                    m = x[t];
            /* pass 2: sum of exponentials */
            double z = 0.0;
            for (int t = 0; t < n; ++t)
                z += exp(x[t] - m);
            /* pass 3: normalised weights times V */
            for (int t = 0; t < n; ++t) {
                double w = exp(x[t] - m) / z;
                for (int i = 0; i < head_dim; ++i) {
                    double vi = orc_load(v_pool,
                                         orc_kv_index(block_tables, max_blocks_per_seq, s, t, kvh,
                                                      i, n_kv_heads, head_dim, block_size),
                                         dtype);
                    o[i] += w * vi;
                }
            }
            free(x);
        }
    }
    return ORC_OK;
}

/*
 * Several query tokens per sequence (a prefill chunk, or tokens to verify):
 * sequence s owns query rows q_start[s] .. q_start[s+1]-1 of q; they are its
 * last q_len = q_start[s+1] - q_start[s] tokens, so row i (0-based within
 * the sequence) sits at position p = context_lens[s] - q_len + i and attends
 * to the keys t <= p (causal).  Per (row, head) the plain definition as in
 * orc_paged_decode_two_pass: scores, maximum pass, sum pass, normalise pass.
 *   out : fp64 [q_start[num_seqs], n_heads, head_dim]
 * ([SWAP] standard attention formula and its FlashAttention tiling over many
 * query rows; the causal restriction is the plain reading of prefill, where a
 * token attends to itself and the tokens before it.)
 */
int orc_paged_multi_query(double* out, const void* q, const void* k_pool, const void* v_pool,
                          int dtype, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                          int n_heads, int n_kv_heads, int head_dim, int block_size,
                          int num_blocks, double scale)
{
    int rc = orc_check(block_tables, max_blocks_per_seq, context_lens, NULL, num_seqs, num_seqs,
                       n_heads, n_kv_heads, head_dim, block_size, num_blocks);
    if (rc != ORC_OK)
        return rc;
    int group = n_heads / n_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = q_start[s + 1] - q_start[s];
        int n = context_lens[s];
        if (q_len < 0 || q_len > n)
            return ORC_BAD_INDEX;
        for (int i = 0; i < q_len; ++i) {
            int row = q_start[s] + i;
            int pos = n - q_len + i;      /* keys 0 .. pos */
            int cnt = pos + 1;
            for (int h = 0; h < n_heads; ++h) {
                double* o = out + ((size_t)row * n_heads + h) * head_dim;
                int kvh = h / group;
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                double* x = (double*)malloc(sizeof(double) * (size_t)cnt);
                if (!x)
                    return ORC_NO_MEM;
                for (int t = 0; t < cnt; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d) {
                        double qi = orc_load(q, ((size_t)row * n_heads + h) * head_dim + d, dtype);
                        double ki = orc_load(k_pool,
                                             orc_kv_index(block_tables, max_blocks_per_seq, s, t,
                                                          kvh, d, n_kv_heads, head_dim,
                                                          block_size),
                                             dtype);
                        acc += qi * ki;
                    }
                    x[t] = scale * acc;
                }
                double m = x[0];
                for (int t = 1; t < cnt; ++t)
                    if (x[t] > m)
                        m = x[t];
                double z = 0.0;
                for (int t = 0; t < cnt; ++t)
                    z += exp(x[t] - m);
                for (int t = 0; t < cnt; ++t) {
                    double w = exp(x[t] - m) / z;
                    for (int d = 0; d < head_dim; ++d) {
                        double vi = orc_load(v_pool,
                                             orc_kv_index(block_tables, max_blocks_per_seq, s, t,
                                                          kvh, d, n_kv_heads, head_dim,
                                                          block_size),
                                             dtype);
                        o[d] += w * vi;
                    }
                }
                free(x);
            }
        }
    }
    return ORC_OK;
}

/*
 * The pages' one-pass method: [SWAP] OnlineSoftmax, [OPT] "关键公式推导".
 * The logical context is cut into consecutive tiles of `tile_tokens` keys;
 * per tile X_i (scaled scores of the tile):
 *     M_new = max(M_old, max(X_i))
 *     L_new = L_old * exp(M_old - M_new) + sum exp(X_i - M_new)
 *     O_new = (L_old * exp(M_old - M_new) / L_new) * O_old
 *             + sum exp(X_i - M_new) * V_i / L_new
 * starting from M = -inf, L = 0, O = 0 (the pages leave the start open;
 * exp(-inf) = 0 makes the first tile's old-state terms vanish).
 *
 * If state_m / state_l are non-NULL the final (M, L) of every (row, head)
 * are stored there ([n_sel, n_heads]) so that tests can merge states.
 * Token range: only logical tokens [t_begin, t_end) of each sequence are
 * visited (t_end < 0 means the whole context); an empty range leaves
 * M = -inf, L = 0, O = 0.
 */
int orc_paged_decode_online(double* out, double* state_m, double* state_l, const void* q,
                            const void* k_pool, const void* v_pool, int dtype,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, const int32_t* seq_ids, int n_sel,
                            int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                            int block_size, int num_blocks, double scale, int tile_tokens,
                            int t_begin, int t_end)
{
    if (tile_tokens <= 0 || t_begin < 0)
        return ORC_BAD_ARG;
    int rc = orc_check(block_tables, max_blocks_per_seq, context_lens, seq_ids, n_sel, num_seqs,
                       n_heads, n_kv_heads, head_dim, block_size, num_blocks);
    if (rc != ORC_OK)
        return rc;
    int group = n_heads / n_kv_heads;
    double* xt = (double*)malloc(sizeof(double) * (size_t)tile_tokens);
    double* acc_v = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!xt || !acc_v) {
        free(xt);
        free(acc_v);
        return ORC_NO_MEM;
    }
    for (int r = 0; r < n_sel; ++r) {
        int s = seq_ids ? seq_ids[r] : r;
        int n = context_lens[s];
        int lo = t_begin < n ? t_begin : n;
        int hi = (t_end < 0 || t_end > n) ? n : t_end;
        if (hi < lo)
            hi = lo;
        for (int h = 0; h < n_heads; ++h) {
            double* o = out + ((size_t)r * n_heads + h) * head_dim;
            int kvh = h / group;
            double M = -INFINITY, L = 0.0;
            for (int i = 0; i < head_dim; ++i)
                o[i] = 0.0;
            for (int t0 = lo; t0 < hi; t0 += tile_tokens) {
                int cnt = hi - t0 < tile_tokens ? hi - t0 : tile_tokens;
                /* X_i: the tile's scaled scores */
                double tile_max = -INFINITY;
                for (int u = 0; u < cnt; ++u) {
                    double acc = 0.0;
                    for (int i = 0; i < head_dim; ++i) {
                        double qi = orc_load(q, ((size_t)s * n_heads + h) * head_dim + i, dtype);
                        double ki = orc_load(k_pool,
                                             orc_kv_index(block_tables, max_blocks_per_seq, s,
                                                          t0 + u, kvh, i, n_kv_heads, head_dim,
                                                          block_size),
                                             dtype);
                        acc += qi * ki;
                    }
                    xt[u] = scale * acc;
                    if (xt[u] > tile_max)
                        tile_max = xt[u];
                }
                double M_new = M > tile_max ? M : tile_max;
                double sum_e = 0.0;
                for (int i = 0; i < head_dim; ++i)
                    acc_v[i] = 0.0;
                for (int u = 0; u < cnt; ++u) {
                    double e = exp(xt[u] - M_new);
                    sum_e += e;
                    for (int i = 0; i < head_dim; ++i) {
                        double vi = orc_load(v_pool,
                                             orc_kv_index(block_tables, max_blocks_per_seq, s,
                                                          t0 + u, kvh, i, n_kv_heads, head_dim,
                                                          block_size),
                                             dtype);
                        acc_v[i] += e * vi;
                    }
                }
                double carry = L * exp(M - M_new); /* L_old * exp(M_old - M_new) */
                double L_new = carry + sum_e;
                for (int i = 0; i < head_dim; ++i)
                    o[i] = (carry / L_new) * o[i] + acc_v[i] / L_new;
                M = M_new;
                L = L_new;
            }
            if (state_m)
                state_m[(size_t)r * n_heads + h] = M;
            if (state_l)
                state_l[(size_t)r * n_heads + h] = L;
        }
    }
    free(xt);
    free(acc_v);
    return ORC_OK;
}

/*
 * Merge of independent partial states (M_k, L_k, O_k), k < n_parts, of one
 * output row: the same recurrence applied with a whole partial state as the
 * "new block".  O_k are normalised partial outputs (as the online form above
 * produces); a part with L_k == 0 is empty and contributes nothing.
 *   m: [n_parts], l: [n_parts], o: [n_parts, head_dim] -> out: [head_dim]
 */
void orc_merge_states(double* out, const double* m, const double* l, const double* o, int n_parts,
                      int head_dim)
{
    double M = -INFINITY, L = 0.0;
    for (int i = 0; i < head_dim; ++i)
        out[i] = 0.0;
    for (int k = 0; k < n_parts; ++k) {
        if (l[k] == 0.0)
            continue;
        double M_new = M > m[k] ? M : m[k];
        double carry = L * exp(M - M_new);
        double part = l[k] * exp(m[k] - M_new);
        double L_new = carry + part;
        for (int i = 0; i < head_dim; ++i)
            out[i] = (carry / L_new) * out[i] + (part / L_new) * o[(size_t)k * head_dim + i];
        M = M_new;
        L = L_new;
    }
}

/*
 * Append one token per sequence (reshape-and-cache): copy the new K and V
 * rows of sequence s, [n_kv_heads, head_dim] elements each, into flat slot
 * slot_mapping[s] of the pools, i.e. physical block slot / B, row slot % B.
 * A negative slot skips the sequence; a slot past the pool is an error
 * (nothing is written for any sequence in that case).
 * [LAYOUT] section 三 append_token; [SWAP] PagedAttention pages.
 */
int orc_kv_append(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                  int elem_bytes, const int64_t* slot_mapping, int num_seqs, int n_kv_heads,
                  int head_dim, int block_size, int64_t num_blocks)
{
    if (elem_bytes <= 0 || num_seqs < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return ORC_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s)
        if (slot_mapping[s] >= num_blocks * block_size)
            return ORC_BAD_INDEX;
    size_t row_bytes = (size_t)n_kv_heads * head_dim * elem_bytes;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t slot = slot_mapping[s];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int64_t row = slot % block_size;
        size_t dst = ((size_t)blk * block_size + (size_t)row) * row_bytes;
        memcpy((char*)k_pool + dst, (const char*)k_new + (size_t)s * row_bytes, row_bytes);
        memcpy((char*)v_pool + dst, (const char*)v_new + (size_t)s * row_bytes, row_bytes);
    }
    return ORC_OK;
}

/*
 * [SWAP] swap_blocks: for each pair (i, j) = (pairs[2k], pairs[2k+1]) copy
 * source block i to destination block j, block_bytes bytes each; [OPT]
 * "Swap Blocks 机制" calls it once for the Key cache and once for the Value
 * cache.  A pair with a negative entry is skipped (the -1 "invalid" marker
 * of the [SWAP] mock); a pair out of range is skipped and counted.
 * Returns the number of pairs skipped for being out of range.
 */
int64_t orc_swap_blocks(void* dst_pool, const void* src_pool, int64_t block_bytes,
                        const int64_t* pairs, int64_t n_pairs, int64_t num_src_blocks,
                        int64_t num_dst_blocks)
{
    int64_t bad = 0;
    for (int64_t k = 0; k < n_pairs; ++k) {
        int64_t i = pairs[2 * k], j = pairs[2 * k + 1];
        if (i < 0 || j < 0)
            continue;
        if (i >= num_src_blocks || j >= num_dst_blocks) {
            ++bad;
            continue;
        }
        memmove((char*)dst_pool + j * block_bytes, (const char*)src_pool + i * block_bytes,
                (size_t)block_bytes);
    }
    return bad;
}
