/*
 * pa_oracle.c -- plain CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * Every function is the plain definition of one step, written for a reader
 * to check against the sources by eye: scalar loops, no blocking, no
 * fusion, no reordering of sums, double-precision arithmetic throughout
 * (bf16 inputs are widened exactly), libm exp().
 *
 * Sources (the web pages this path is defined by):
 *   [NV12]  "12. 推理加速(二):nano-vllm — 1200 行手写 vLLM" (chuoer47.github.io),
 *           §12.6 "Attention 层: Paged KV Cache" and §12.7 "ModelRunner".
 *   [NV05]  kyonqi.github.io "nano-vllm/05" (ModelRunner: prepare_prefill,
 *           prepare_decode, prepare_block_tables, run_model).
 *   [VD]    "vLLM 深度解读" (luoboask.github.io), §3 "PagedAttention CUDA Kernel".
 *   [PA3]   "Nano-vLLM 源码解读 - 3. PagedAttention" (yeyulingfeng.com),
 *           §3 two-level mapping, §4 slot_mapping (prefill and decode paths).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - a query head h uses kv head h / (Hq/Hkv) (contiguous GQA groups);
 *   - prefill causality is aligned bottom-right: query i of a sequence with
 *     c = Lk - Lq cached tokens sits at absolute position c + i and sees keys
 *     at positions <= c + i;
 *   - a decode query (the token at position ctx-1) sees all ctx keys;
 *   - a slot < 0 is padding and is skipped; context_len == 0 gives zeros.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC pa_oracle.c -lm
 * (-ffp-contract=off keeps x86 and aarch64 results identical.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1   /* bad argument or out-of-range index */
#define ORACLE_EDUP -2     /* two tokens target the same slot */

/* bf16 is the upper half of an IEEE binary32 word; widening is exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int pa_oracle_version(void) { return 1; }

/* ------------------------------------------------------------------------ */
/* Slot mapping.                                                             */
/* ------------------------------------------------------------------------ */

/*
 * Slots for the tokens at positions [start, end) of one sequence, written
 * block by block as [PA3 §4 "Prefill 路径"] describes (and [NV12 §12.7]
 * prepare_prefill): for every logical block i the sequence touches, the run
 * of slots begins at block_table[i]*B (shifted by start % B in the first
 * block) and ends at block_table[i]*B + B, or at block_table[i]*B + end - i*B
 * in the last block.  Returns the number of slots written (end - start) or
 * ORACLE_EINVAL.
 */
int pa_oracle_slot_mapping(const int32_t *block_table, int32_t table_len, int32_t block_size,
                           int32_t start, int32_t end, int32_t *out) {
    if (block_size <= 0 || start < 0 || end < start) return ORACLE_EINVAL;
    if (end == start) return 0;
    int32_t start_block = start / block_size;
    int32_t end_block = (end + block_size - 1) / block_size;
    if (end_block > table_len) return ORACLE_EINVAL;
    int32_t n = 0;
    for (int32_t i = start_block; i < end_block; ++i) {
        if (block_table[i] < 0) return ORACLE_EINVAL;
        int64_t first = (int64_t)block_table[i] * block_size;
        int64_t slot_start = first;
        int64_t slot_end;
        if (i == start_block) slot_start += start % block_size;
        if (i != end_block - 1)
            slot_end = first + block_size;
        else
            slot_end = first + (int64_t)end - (int64_t)i * block_size;
        for (int64_t s = slot_start; s < slot_end; ++s) out[n++] = (int32_t)s;
    }
    return n;
}

/*
 * The decode slot of one sequence [PA3 §4 "Decode 路径"; NV05 prepare_decode]:
 * the slot of its newest token = last_block * B + tokens_in_last_block - 1,
 * where the last block is block_table[ceil(ctx/B) - 1] (a padded table row
 * carries -1 after it).  ctx == 0 is a padding row: slot -1.  An invalid
 * argument returns INT32_MIN.
 */
int32_t pa_oracle_decode_slot(const int32_t *block_table, int32_t table_len, int32_t block_size,
                              int32_t context_len) {
    if (context_len <= 0) return -1;
    int32_t num_blocks = (context_len + block_size - 1) / block_size;
    if (num_blocks > table_len || block_table[num_blocks - 1] < 0) return INT32_MIN;
    int32_t last_block_num_tokens = context_len - (num_blocks - 1) * block_size;
    return block_table[num_blocks - 1] * block_size + last_block_num_tokens - 1;
}

/* ------------------------------------------------------------------------ */
/* store_kvcache [NV12 §12.6 "Triton KV Cache Store Kernel"].                */
/* ------------------------------------------------------------------------ */

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * For every token i whose slot_mapping[i] is not negative, copy its
 * num_kv_heads*head_dim K values to k_cache[slot*num_kv_heads*head_dim ...]
 * and its V values likewise.  Values are copied as raw 16-bit words.  Rows
 * of key/value are key_row_stride / value_row_stride elements apart.
 * Two tokens naming the same slot is rejected (the pages never produce it).
 */
int pa_oracle_store_kvcache(const uint16_t *key, int64_t key_row_stride, const uint16_t *value,
                            int64_t value_row_stride, uint16_t *k_cache, uint16_t *v_cache,
                            const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                            int32_t head_dim, int64_t num_slots) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0) return ORACLE_EINVAL;
    int64_t D = (int64_t)num_kv_heads * head_dim;
    int32_t *sorted = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_tokens > 0 ? num_tokens : 1));
    if (!sorted) return ORACLE_EINVAL;
    int32_t n = 0;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if ((int64_t)slot >= num_slots) { free(sorted); return ORACLE_EINVAL; }
        sorted[n++] = slot;
    }
    qsort(sorted, (size_t)n, sizeof(int32_t), cmp_i32);
    for (int32_t i = 1; i < n; ++i)
        if (sorted[i] == sorted[i - 1]) { free(sorted); return ORACLE_EDUP; }
    free(sorted);

    for (int32_t i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0) continue; /* padding */
        for (int64_t j = 0; j < D; ++j) {
            k_cache[(int64_t)slot * D + j] = key[(int64_t)i * key_row_stride + j];
            v_cache[(int64_t)slot * D + j] = value[(int64_t)i * value_row_stride + j];
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention over gathered rows.                                             */
/* ------------------------------------------------------------------------ */

/*
 * Row of kv head g for logical position p of a sequence, found through its
 * block table by the two-level mapping of [PA3 §3]: the physical slot is
 * block_table[p / B] * B + p % B.  Returns NULL if the block id is invalid.
 */
static const uint16_t *paged_row(const uint16_t *cache, const int32_t *block_table, int32_t B,
                                 int32_t Hkv, int32_t D, int32_t num_blocks, int32_t p, int32_t g) {
    int32_t block = block_table[p / B];
    if (block < 0 || block >= num_blocks) return NULL;
    int64_t slot = (int64_t)block * B + p % B;
    return cache + (slot * Hkv + g) * D;
}

/*
 * softmax(scale * q.K^T) V over n rows, the textbook two-pass form:
 * s_j = scale * sum_d q[d] K_j[d];  m = max_j s_j;  w_j = exp(s_j - m);
 * out[d] = sum_j w_j V_j[d] / sum_j w_j.   n == 0 writes zeros.
 * K_rows[j] / V_rows[j] point at the j-th key / value row (D bf16 values).
 */
static void attend(double *out, const uint16_t *q, const uint16_t *const *K_rows,
                   const uint16_t *const *V_rows, int64_t n, int32_t D, double scale,
                   double *s /* scratch [n] */) {
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(K_rows[j][d]);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double w = exp(s[j] - m);
        denom += w;
        for (int32_t d = 0; d < D; ++d) out[d] += w * bf16_to_double(V_rows[j][d]);
    }
    for (int32_t d = 0; d < D; ++d) out[d] /= denom;
}

/*
 * Paged decode attention [NV12 §12.6 flash_attn_with_kvcache; VD §3
 * paged_attention_v1_kernel]: one query token per sequence b, which sees
 * the context_lens[b] tokens of its sequence, read through
 * block_tables[b, :].  q row b starts at q + b*q_row_stride and holds Hq
 * heads of D values.  Output for (b, h) goes to out[r*D ...] where r runs
 * over the requested rows: rows == NULL means all b*Hq + h in order, else
 * rows[r] = b*Hq + h.  Unsplit by design: split-KV results are checked
 * against this.
 */
int pa_oracle_decode(double *out, const uint16_t *q, int64_t q_row_stride, const uint16_t *k_cache,
                     const uint16_t *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     double softmax_scale, const int64_t *rows, int64_t n_rows) {
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0)
        return ORACLE_EINVAL;
    int32_t group = num_q_heads / num_kv_heads;
    int64_t total = rows ? n_rows : (int64_t)batch * num_q_heads;
    int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    const uint16_t **K_rows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    const uint16_t **V_rows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    int rc = ORACLE_OK;
    if (!s || !K_rows || !V_rows) { rc = ORACLE_EINVAL; goto done; }
    for (int64_t r = 0; r < total; ++r) {
        int64_t row = rows ? rows[r] : r;
        int32_t b = (int32_t)(row / num_q_heads), h = (int32_t)(row % num_q_heads);
        if (b < 0 || b >= batch) { rc = ORACLE_EINVAL; goto done; }
        int32_t g = h / group;
        int32_t ctx = context_lens[b];
        if (ctx < 0 || ctx > max_ctx) { rc = ORACLE_EINVAL; goto done; }
        const int32_t *bt = block_tables + (int64_t)b * max_blocks_per_seq;
        for (int32_t p = 0; p < ctx; ++p) {
            K_rows[p] = paged_row(k_cache, bt, block_size, num_kv_heads, head_dim, num_blocks, p, g);
            V_rows[p] = paged_row(v_cache, bt, block_size, num_kv_heads, head_dim, num_blocks, p, g);
            if (!K_rows[p] || !V_rows[p]) { rc = ORACLE_EINVAL; goto done; }
        }
        attend(out + r * head_dim, q + (int64_t)b * q_row_stride + (int64_t)h * head_dim, K_rows,
               V_rows, ctx, head_dim, softmax_scale, s);
    }
done:
    free(s);
    free(K_rows);
    free(V_rows);
    return rc;
}

/*
 * Varlen prefill attention [NV12 §12.6 flash_attn_varlen_func and the
 * cu_seqlens example; NV05 prepare_prefill].  Sequence s owns query rows
 * [cu_q[s], cu_q[s+1]) and has Lk = cu_k[s+1] - cu_k[s] keys, of which the
 * first c = Lk - Lq were cached earlier.  Query i of it sits at position
 * c + i; with causal != 0 it sees keys 0..c+i, else all Lk keys.
 * Keys come from the pool through block_tables[s, :] when block_tables is
 * not NULL (prefix cache), else from contiguous k/v rows cu_k[s] + j with
 * row stride kv_row_stride elements.  Output row r (rows == NULL: all
 * token*Hq + h in order; else rows[r] = token*Hq + h) goes to out[r*D ...].
 */
int pa_oracle_prefill(double *out, const uint16_t *q, int64_t q_row_stride, const uint16_t *k,
                      const uint16_t *v, int64_t kv_row_stride, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                      const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                      double softmax_scale, int32_t causal, const int64_t *rows, int64_t n_rows) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ORACLE_EINVAL;
    if (block_tables && block_size <= 0) return ORACLE_EINVAL;
    int32_t group = num_q_heads / num_kv_heads;
    int64_t total_q = cu_seqlens_q[num_seqs];
    int64_t total = rows ? n_rows : total_q * num_q_heads;
    int64_t max_lk = 1;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        int64_t lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        if (lq < 0 || lk < lq) return ORACLE_EINVAL;
        if (block_tables && lk > (int64_t)max_blocks_per_seq * block_size) return ORACLE_EINVAL;
        if (lk > max_lk) max_lk = lk;
    }
    double *sc = (double *)malloc(sizeof(double) * (size_t)max_lk);
    const uint16_t **K_rows = (const uint16_t **)malloc(sizeof(void *) * (size_t)max_lk);
    const uint16_t **V_rows = (const uint16_t **)malloc(sizeof(void *) * (size_t)max_lk);
    int rc = ORACLE_OK;
    if (!sc || !K_rows || !V_rows) { rc = ORACLE_EINVAL; goto done; }
    for (int64_t r = 0; r < total; ++r) {
        int64_t row = rows ? rows[r] : r;
        int64_t t = row / num_q_heads;
        int32_t h = (int32_t)(row % num_q_heads), g = h / group;
        if (t < 0 || t >= total_q) { rc = ORACLE_EINVAL; goto done; }
        int32_t s = 0; /* the sequence that owns query row t */
        while (!(cu_seqlens_q[s] <= t && t < cu_seqlens_q[s + 1])) ++s;
        int64_t lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int64_t lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        int64_t i = t - cu_seqlens_q[s];
        int64_t pos = (lk - lq) + i;
        int64_t nkeys = causal ? pos + 1 : lk;
        for (int64_t j = 0; j < nkeys; ++j) {
            if (block_tables) {
                const int32_t *bt = block_tables + (int64_t)s * max_blocks_per_seq;
                K_rows[j] = paged_row(k, bt, block_size, num_kv_heads, head_dim, num_blocks, (int32_t)j, g);
                V_rows[j] = paged_row(v, bt, block_size, num_kv_heads, head_dim, num_blocks, (int32_t)j, g);
                if (!K_rows[j] || !V_rows[j]) { rc = ORACLE_EINVAL; goto done; }
            } else {
                int64_t kr = cu_seqlens_k[s] + j;
                K_rows[j] = k + kr * kv_row_stride + (int64_t)g * head_dim;
                V_rows[j] = v + kr * kv_row_stride + (int64_t)g * head_dim;
            }
        }
        attend(out + r * head_dim, q + t * q_row_stride + (int64_t)h * head_dim, K_rows, V_rows,
               nkeys, head_dim, softmax_scale, sc);
    }
done:
    free(sc);
    free(K_rows);
    free(V_rows);
    return rc;
}
