/*
 * pa.h -- C ABI of the paged-KV attention library (libpa.so), sm_103a.
 *
 * Three operations make up the path, in the order one model layer calls them
 * on a stream: pa_store_kvcache writes this step's new K/V rows into the
 * block pool, then pa_decode (one query token per sequence) or
 * pa_prefill_varlen (many query tokens per sequence, causal) reads K/V back
 * through the block tables.  Two helpers, pa_slot_mapping_decode and
 * pa_slot_mapping_prefill, build the slot_mapping the store consumes.
 *
 * Sources (web pages that define the operations):
 *   [NV12] "12. 推理加速(二):nano-vllm — 1200 行手写 vLLM" (chuoer47.github.io),
 *          §12.6 "Attention 层: Paged KV Cache", §12.7 "ModelRunner".
 *   [NV05] kyonqi.github.io "nano-vllm/05", ModelRunner: prepare_prefill,
 *          prepare_decode, prepare_block_tables, run_model.
 *   [VD]   "vLLM 深度解读" (luoboask.github.io), §3 "PagedAttention CUDA Kernel".
 *   [PA3]  "Nano-vLLM 源码解读 - 3. PagedAttention" (yeyulingfeng.com),
 *          §3 two-level mapping, §4 slot_mapping, §5 block size.
 *
 * Conventions shared by every entry point
 *   - Element type: bf16 for q, k, v, caches and outputs (passed as void*).
 *   - KV pool: one layer's k_cache and v_cache are each a contiguous
 *     [num_blocks, block_size, num_kv_heads, head_dim] array; slot s is the
 *     row k_cache + s*num_kv_heads*head_dim ([NV12 §12.7 allocate_kv_cache];
 *     [PA3 §3]).  The physical slot of logical position p of a sequence is
 *     block_table[p / block_size] * block_size + p % block_size.
 *   - block_tables: int32 [batch, max_blocks_per_seq], row-major; entries
 *     past a sequence's ceil(len/block_size) blocks are never read and may be
 *     -1 ([NV05 prepare_block_tables]).
 *   - head_dim must be 128 and num_q_heads a multiple of num_kv_heads with
 *     num_q_heads/num_kv_heads in {1, 2, 4, 8}; query head h reads kv head
 *     h / (num_q_heads/num_kv_heads).  Other shapes return PA_ERR_UNSUPPORTED.
 *   - block_size must be a positive multiple of 16 (256 is the tuned case).
 *   - Pointers are device pointers unless stated.  Base pointers of bf16
 *     arrays must be 16-byte aligned and row strides multiples of 8 elements.
 *   - Ownership: the caller owns every buffer and the stream.  No entry point
 *     allocates or frees device memory, and none synchronises the stream
 *     except pa_get_device_error.  Work is enqueued on `stream` in call order,
 *     so a store followed by an attention call on the same stream is ordered.
 *   - Errors: host-side argument checks return a status before anything is
 *     enqueued; pa_last_error_message() gives the detail (thread-local).  A
 *     launch failure returns PA_ERR_CUDA.  Problems only visible on the device
 *     (an out-of-range slot or block id, a context longer than its table, a
 *     wait that timed out) never fault: the kernel skips the access, records
 *     the first one in a device error word and carries on; read it with
 *     pa_get_device_error.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, bad stride */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim != 128, ...) */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
    PA_ERR_DEVICE_CHECK = 5   /* a kernel recorded a device-side error */
} pa_status;

/* Device-side error codes reported by pa_get_device_error. */
enum {
    PA_DEV_OK = 0,
    PA_DEV_TIMEOUT = 1,        /* a bounded wait gave up; where = kernel id */
    PA_DEV_BAD_SLOT = 2,       /* store: slot >= num_slots; where = token index */
    PA_DEV_BAD_CONTEXT = 3,    /* context length < 0 or > max_blocks_per_seq*block_size;
                                  where = sequence index */
    PA_DEV_BAD_BLOCK = 4,      /* checked mode: block id outside [0, num_blocks);
                                  where = sequence*max_blocks_per_seq + logical block */
    PA_DEV_BAD_SEQLENS = 5,    /* prefill: cu_seqlens not monotone or Lq > Lk;
                                  where = sequence index */
    PA_DEV_SMEM_ALIGN = 6,     /* a kernel could not align its shared-memory tiles
                                  (no work done); where = bytes of padding needed */
    PA_DEV_BAD_TEMPERATURE = 7 /* sampler: temperature not > 1e-10; where = row */
};

/* Library version (major*10000 + minor*100 + patch). */
PA_API int pa_version(void);

/* Static string for a status code. */
PA_API const char *pa_status_str(pa_status status);

/* Detail of the last non-OK status returned on the calling thread ("" if none). */
PA_API const char *pa_last_error_message(void);

/*
 * pa_store_kvcache -- scatter this step's K/V rows into the pool.
 * [NV12 §12.6 store_kvcache / store_kvcache_kernel; PA3 §4]
 *
 * For each token i in [0, num_tokens) with slot = slot_mapping[i] >= 0:
 *   k_cache[slot*Hkv*D + j] = key[i*key_row_stride + j]   for j < Hkv*D,
 * and the same for value -> v_cache.  Negative slots are padding (CUDA-graph
 * batches are padded with -1) and write nothing.  A slot >= num_slots is not
 * written and is recorded as PA_DEV_BAD_SLOT.
 *
 *   key, value           bf16 [num_tokens, *]: token i's Hkv*D values start at
 *                        key + i*key_row_stride (elements) and are contiguous
 *                        ([Hkv, D] row-major), so fused-QKV views are allowed.
 *   key_row_stride,
 *   value_row_stride     elements between tokens; >= Hkv*D, multiple of 8.
 *   k_cache, v_cache     bf16 pools [num_slots / block_size, block_size, Hkv, D].
 *   slot_mapping         int32 [num_tokens]; non-negative entries must be distinct.
 *   num_slots            num_blocks * block_size (bounds check only).
 * Copies are bit-exact.  num_tokens == 0 is a no-op.
 */
PA_API pa_status pa_store_kvcache(const void *key, int64_t key_row_stride, const void *value,
                           int64_t value_row_stride, void *k_cache, void *v_cache,
                           const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int64_t num_slots, pa_stream_t stream);

/*
 * pa_slot_mapping_decode -- slot of each sequence's newest token.
 * [PA3 §4 "Decode 路径"; NV05 prepare_decode]
 *
 * slot_mapping[b] = block_tables[b][(ctx-1)/B]*B + (ctx-1)%B with
 * ctx = context_lens[b], i.e. last block * B + tokens in last block - 1;
 * context_lens[b] == 0 (a padded row) gives -1.
 *   slot_mapping   int32 [batch] (output, device).
 */
PA_API pa_status pa_slot_mapping_decode(int32_t *slot_mapping, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                 int32_t batch, int32_t block_size, pa_stream_t stream);

/*
 * pa_slot_mapping_prefill -- slots of the uncached suffix of every sequence.
 * [PA3 §4 "Prefill 路径"; NV12 §12.7 prepare_prefill]
 *
 * Sequence s computes positions [c, Lk) with Lk = cu_seqlens_k[s+1] -
 * cu_seqlens_k[s], Lq = cu_seqlens_q[s+1] - cu_seqlens_q[s], c = Lk - Lq (c
 * may sit mid-block: chunked prefill).  Query row cu_seqlens_q[s] + i gets
 * the slot of position c + i.
 *   slot_mapping   int32 [total_q] (output, device), total_q = cu_seqlens_q[num_seqs].
 */
PA_API pa_status pa_slot_mapping_prefill(int32_t *slot_mapping, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                  const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                  int32_t block_size, pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs.
 * It depends only on the GQA group (num_q_heads / num_kv_heads) and is at
 * most about 4.3 MB; 0 for shapes pa_decode does not support.
 */
PA_API size_t pa_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim);

/*
 * pa_decode -- paged split-KV GQA decode attention, one query per sequence.
 * [NV12 §12.6 flash_attn_with_kvcache; VD §3 paged_attention_v1_kernel]
 *
 * For sequence b, query head h, kv head g = h / (Hq/Hkv), ctx = context_lens[b]:
 *   s_p = softmax_scale * <q[b,h,:], K[slot(b,p), g, :]>   for p < ctx,
 *   out[b,h,:] = sum_p softmax(s)_p * V[slot(b,p), g, :]    (bf16, RNE),
 * where slot(b,p) = block_tables[b][p/B]*B + p%B.  The query is the token at
 * position ctx-1 and sees all ctx keys, including its own (store it first).
 * ctx == 0 writes zeros and reads nothing.  The tiles of all (sequence, kv
 * head) pairs are cut into contiguous ranges (one per CTA, then small chunks
 * taken dynamically); a pair cut between ranges is combined in the same
 * kernel by the CTA that finishes its last part (log-sum-exp of the
 * online-softmax partials).  The kernel is launched as a programmatic
 * dependent launch and reads its inputs only after the preceding work on
 * the stream has completed.
 *
 *   out                bf16 [batch, Hq, D] contiguous.
 *   q                  bf16; row b (Hq*D contiguous values) at q + b*q_row_stride.
 *   k_cache, v_cache   the layer's pools (see conventions); num_blocks blocks.
 *   block_tables       int32 [batch, max_blocks_per_seq].
 *   context_lens       int32 [batch], each in [0, max_blocks_per_seq*block_size].
 *   softmax_scale      usually 1/sqrt(head_dim).
 *   workspace          device scratch of >= pa_decode_workspace_size(...)
 *                      bytes, 16-byte aligned, ZERO-FILLED before its first
 *                      use (fp32 split partials and work counters).  Every
 *                      call leaves it zero-filled again, so one memset at
 *                      allocation is enough; after a call that recorded a
 *                      device error, zero it again.  One workspace must not be
 *                      used by two calls that may run at the same time.
 * batch == 0 is a no-op; batch <= 2048.
 */
PA_API pa_status pa_decode(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                    float softmax_scale, void *workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/*
 * pa_decode_store -- pa_decode that first stores the step's new token.
 * [NV12 §12.6: store_kvcache then attention, fused]
 *
 * For every sequence b with ctx = context_lens[b] > 0, the new token's K and
 * V rows (new_k[b], new_v[b]: Hkv*D bf16 each, row stride in elements) are
 * written to slot block_tables[b][(ctx-1)/B]*B + (ctx-1)%B of k_cache /
 * v_cache -- the token at position ctx-1, which the query is -- and the
 * attention then reads them like every other key.  The write is done inside
 * the decode kernel by the consumer warp that owns the token's key in the
 * sequence's last tile: it puts the row into that landed tile and into the
 * slot (one kv head's 256-byte row each), so the step needs neither a slot
 * mapping nor a separate store launch.  Afterwards the caches hold exactly what
 * pa_slot_mapping_decode + pa_store_kvcache would have written.  Other
 * arguments, the workspace contract and the outputs are those of pa_decode;
 * new_k / new_v 16-byte aligned.
 */
PA_API pa_status pa_decode_store(void *out, const void *q, int64_t q_row_stride, const void *new_k,
                                 int64_t new_k_row_stride, const void *new_v, int64_t new_v_row_stride,
                                 void *k_cache, void *v_cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t num_blocks, float softmax_scale, void *workspace,
                                 size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_shared_prefix -- pa_decode / pa_decode_store for batches in which
 * sequences share prefix-cache blocks.  [NV12 §12.8 BlockManager prefix
 * caching: sequences whose prompts begin with the same full blocks hold the
 * same physical blocks (ref_count > 1); NV12 §12.6 flash_attn_with_kvcache]
 *
 * Same result as pa_decode (new_k == new_v == NULL) or pa_decode_store (both
 * given, same layout and contract), within the attention tolerance: only the
 * summation order differs.  Sequences are grouped on the device by the id of
 * their first block; a group's shared prefix is the longest run of leading
 * block ids all its members agree on, limited for each member to the full
 * blocks before the one holding its newest token.  For groups of two or more
 * sequences a first kernel attends every member's query heads to the shared
 * prefix once per kv head (each of its K/V rows is read once, not once per
 * member) and leaves fp32 (m, l, o) partials in the workspace; the decode
 * kernel then streams only each member's own suffix and merges the prefix
 * partial into the member's result (log-sum-exp).  Batches without sharing
 * pay for the grouping pass and one extra launch; prefer pa_decode there.
 *
 *   workspace   >= pa_decode_shared_prefix_workspace_size(...) bytes (the
 *               pa_decode workspace plus the groups and the prefix partials
 *               of up to 8192 (member, q head) rows: ~8.6 MB more), same
 *               zero-filling contract as pa_decode.  Members beyond
 *               8192 / num_q_heads (in batch order) read the shared prefix
 *               themselves.
 *   batch       <= 1024.
 * Every other argument, the ordering and the error behaviour are those of
 * pa_decode / pa_decode_store.
 */
PA_API size_t pa_decode_shared_prefix_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim);
PA_API pa_status pa_decode_shared_prefix(void *out, const void *q, int64_t q_row_stride, const void *new_k,
                                         int64_t new_k_row_stride, const void *new_v, int64_t new_v_row_stride,
                                         void *k_cache, void *v_cache, const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t num_blocks, float softmax_scale, void *workspace,
                                         size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_static -- pa_decode for callers that cannot allocate device memory.
 * (An addition of this library: the source pages have no counterpart.)
 *
 * Same arguments and result as pa_decode, minus the workspace.  Some callers
 * cannot call cudaMalloc or an allocating library: code running inside
 * another framework's memory pool, plugins that must not touch the
 * allocator, or hosts that forbid device allocation after start-up.  This
 * entry point allocates nothing.  The split partials go to an 8 MiB scratch
 * array compiled into the library, which holds the workspace of every
 * supported shape (a shape needing more returns PA_ERR_UNSUPPORTED); every
 * GPU that loads the library holds those 8 MiB until the process exits.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *   - The partials need no initial value, but the work counters at the
 *     front of the array must be zero when the kernel starts.  Every call
 *     therefore clears them first (a cudaMemsetAsync of a few KiB on
 *     `stream`, which allocates nothing), so a call that stopped on a device
 *     error (PA_DEV_TIMEOUT) leaves nothing behind that a later call could
 *     trip on.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Calls that may overlap on the GPU (other streams, other threads) race
 *     on it and must be serialised by the caller.
 */
PA_API pa_status pa_decode_static(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_blocks, float softmax_scale,
                                  pa_stream_t stream);

/*
 * pa_decode_static_scratch -- device address (on the current device) and size
 * in bytes of the scratch array pa_decode_static uses, for inspection and
 * tests.  Performs the same once-per-device look-up as pa_decode_static's
 * first call; allocates nothing.
 */
PA_API pa_status pa_decode_static_scratch(void **device_ptr, size_t *bytes);

/*
 * pa_prefill_varlen -- varlen causal attention for prompt (prefill) tokens.
 * [NV12 §12.6 flash_attn_varlen_func and its cu_seqlens example; NV05 prepare_prefill]
 *
 * Sequence s owns query rows [cu_seqlens_q[s], cu_seqlens_q[s+1]) (Lq rows)
 * and Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s] >= Lq keys; the first
 * c = Lk - Lq keys were cached earlier (prefix-cache hits).  Query i sits at
 * position c + i and, with causal != 0, sees keys 0..c+i (bottom-right
 * alignment); with causal == 0 it sees all Lk keys.  Sequences never
 * interact.  Tensor cores (tcgen05, bf16 in, fp32 accumulate) compute
 * Q.K^T and P.V; the softmax runs in fp32 with P rounded to bf16.
 *   out            bf16 [total_q, Hq, D] contiguous.
 *   q              bf16; row t at q + t*q_row_stride, Hq*D contiguous values.
 *   total_q        rows of q (= cu_seqlens_q[num_seqs]); bounds the q reads.
 *   k, v           block_tables != NULL: the layer's caches (keys of sequence s
 *                  at slot(s, j)); the suffix must already be stored.
 *                  block_tables == NULL: contiguous rows, key j of sequence s
 *                  at k + (cu_seqlens_k[s] + j)*kv_row_stride, Hkv*D values.
 *   kv_row_stride  elements between rows in the contiguous case (ignored otherwise).
 *   total_k        rows of contiguous k/v (ignored when paged); bounds the reads.
 *   max_seqlen_q   an upper bound of Lq (sizes the grid); max_seqlen_k of Lk.
 *   num_blocks     pool size in blocks (paged case).
 */
PA_API pa_status pa_prefill_varlen(void *out, const void *q, int64_t q_row_stride, int32_t total_q,
                                   const void *k, const void *v, int64_t kv_row_stride, int32_t total_k,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                   int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, float softmax_scale,
                                   int32_t causal, pa_stream_t stream);

/*
 * pa_prefill_store_varlen -- pa_prefill_varlen (paged) that first stores the
 * uncached suffix.  [NV12 §12.6: store_kvcache then flash_attn_varlen_func,
 * fused; PA3 §4: the slot of position p is block_table[p/B]*B + p%B]
 *
 * new_k / new_v hold the suffix tokens' K and V rows in cu_seqlens_q order
 * ([total_q, Hkv, D] bf16, row strides in elements, multiples of 8, 16-byte
 * aligned): token t of sequence s sits at position (Lk - Lq) + (t -
 * cu_seqlens_q[s]), Lq / Lk its query / key lengths.  Each row is written to
 * that position's slot of k_cache / v_cache, exactly what
 * pa_slot_mapping_prefill + pa_store_kvcache would write (a block id outside
 * [0, num_blocks) is recorded as PA_DEV_BAD_SLOT with where = t, and that row
 * is not written); then the attention of pa_prefill_varlen runs over the
 * pool, with the same arguments and output.  block_tables is required.
 *
 * One launch: the CTAs copy the rows, meet at a grid barrier, then attend.
 * The launch is cooperative (its CTAs must be resident together, one per
 * SM); if the device cannot run it so, the call returns PA_ERR_CUDA.
 *
 * workspace: >= pa_prefill_store_workspace_size() bytes of device memory,
 * 8-byte aligned, zero-filled before first use; the call leaves it as it
 * found it, so it serves any number of calls on one stream (not concurrent
 * calls).  If the grid barrier gives up (PA_DEV_TIMEOUT, where = 440) no
 * attention runs in that CTA; zero the workspace again before the next call.
 */
PA_API size_t pa_prefill_store_workspace_size(void);
PA_API pa_status pa_prefill_store_varlen(void *out, const void *q, int64_t q_row_stride, int32_t total_q,
                                         const void *new_k, int64_t new_k_row_stride, const void *new_v,
                                         int64_t new_v_row_stride, void *k_cache, void *v_cache,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                         int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t num_blocks, float softmax_scale,
                                         int32_t causal, void *workspace, size_t workspace_bytes,
                                         pa_stream_t stream);

/*
 * pa_sample_gumbel -- sample one token per row by the Gumbel-max trick.
 * [NV12 §12.2 "采样器": Sampler.forward and the Gumbel-max derivation]
 *
 *   token[b] = argmax_i softmax(float(logits[b]) / T_b)_i / max(E[b,i], 1e-10)
 *
 * computed in fp32; the lowest index wins among equal maxima.  E ~ Exp(1),
 * one independent draw per (row, vocabulary entry), is drawn by the caller
 * (e.g. torch.empty(...).exponential_(1)), which owns the random state.
 *   out_tokens        int32 [batch].
 *   logits            [batch, vocab] bf16 (logits_is_fp32 = 0) or fp32 (1);
 *                     row b at logits + b*logits_row_stride elements; the
 *                     stride is a multiple of 8 (bf16) or 4 (fp32) elements.
 *   temperatures      fp32 [batch], each > 1e-10; a row whose temperature is
 *                     not gets token -1 and PA_DEV_BAD_TEMPERATURE.
 *   exp_noise         fp32 [batch, vocab], row stride noise_row_stride (a
 *                     multiple of 4 elements).
 *   batch <= 65535.  A row with no finite candidate (all logits -inf or NaN)
 *   gets token 0.  Base pointers 16-byte aligned.  One kernel, a programmatic
 *   dependent launch; each row is read once (HBM-bound).
 */
PA_API pa_status pa_sample_gumbel(int32_t *out_tokens, const void *logits, int64_t logits_row_stride,
                                  int32_t logits_is_fp32, const float *temperatures, const float *exp_noise,
                                  int64_t noise_row_stride, int32_t batch, int32_t vocab, pa_stream_t stream);

/* --------------------------------------------------------------------------
 * Host block manager: the pool's allocator and prefix cache, whose block
 * tables the kernels above consume.  Host code only (no GPU, no CUDA calls).
 * [NV12 §12.8 "BlockManager: 分页 KV Cache + Prefix Caching";
 *  VS §1.1 (the four fields), §1.2.4 (a traced allocation), §1.2.5 (prefix hits)]
 *
 * State: num_blocks blocks of block_size tokens, each with a reference count,
 * the chained hash of its prefix (or none) and its token ids; a FIFO queue of
 * free block ids (taken from the front, returned to the back); the set of
 * used ids; a map from prefix hash to block id.  The chained hash of block i
 * of a sequence is XXH64 (seed 0) of [hash of block i-1 as 8 little-endian
 * bytes, omitted for i = 0] followed by the block's token ids as 64-bit
 * little-endian integers (pa_bm_block_hash).  Sequences are kept in the
 * manager and named by the id pa_bm_seq_add returns.
 *
 * pa_bm_can_allocate  number of leading full blocks (never the last block)
 *                     found in the prefix cache with identical tokens, or -1
 *                     if the free queue is shorter than the blocks still
 *                     needed (cached blocks in use need none); -2: bad args.
 * pa_bm_allocate      give the sequence its blocks: the first
 *                     num_cached_blocks from the cache (one more reference,
 *                     or taken back from the free queue), then fresh ones
 *                     from the front of the queue (a fresh block loses its
 *                     old map entry); num_cached_tokens = cached * block_size.
 * pa_bm_deallocate    drop one reference per block, last block first; blocks
 *                     at zero go to the back of the free queue keeping their
 *                     hash (so a later prefix hit can take them back).
 * pa_bm_can_append    1 if a decode step of the sequence can get the block it
 *                     needs (one exactly when len % block_size == 1), else 0.
 * pa_bm_may_append    take that block if needed.
 * pa_bm_hash_blocks   register the blocks filled by a step of
 *                     num_scheduled_tokens tokens after num_cached_tokens:
 *                     blocks [cached / B, (cached + scheduled) / B).  The
 *                     caller then advances num_cached_tokens
 *                     (pa_bm_seq_set_num_cached_tokens) and appends generated
 *                     tokens (pa_bm_seq_append_token).
 * pa_bm_block_tables  int32 [num_seqs, max_blocks_per_seq] block tables, -1
 *                     past each sequence's blocks (the kernels' format).
 * Queries return counts (or -2 for bad arguments); errors set
 * pa_last_error_message.  A manager is not thread-safe.
 */
typedef struct pa_block_manager pa_block_manager;
PA_API pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, pa_block_manager **out);
PA_API void pa_bm_destroy(pa_block_manager *bm);
PA_API pa_status pa_bm_seq_add(pa_block_manager *bm, const int64_t *token_ids, int32_t num_tokens, int32_t *seq_id);
PA_API pa_status pa_bm_seq_append_token(pa_block_manager *bm, int32_t seq, int64_t token_id);
PA_API pa_status pa_bm_seq_set_num_cached_tokens(pa_block_manager *bm, int32_t seq, int32_t num_cached_tokens);
PA_API pa_status pa_bm_seq_info(const pa_block_manager *bm, int32_t seq, int32_t *num_tokens,
                                int32_t *num_cached_tokens, int32_t *num_table_blocks);
PA_API int32_t pa_bm_can_allocate(const pa_block_manager *bm, int32_t seq);
PA_API pa_status pa_bm_allocate(pa_block_manager *bm, int32_t seq, int32_t num_cached_blocks);
PA_API pa_status pa_bm_deallocate(pa_block_manager *bm, int32_t seq);
PA_API int32_t pa_bm_can_append(const pa_block_manager *bm, int32_t seq);
PA_API pa_status pa_bm_may_append(pa_block_manager *bm, int32_t seq);
PA_API pa_status pa_bm_hash_blocks(pa_block_manager *bm, int32_t seq, int32_t num_scheduled_tokens);
PA_API int32_t pa_bm_seq_block_table(const pa_block_manager *bm, int32_t seq, int32_t *out, int32_t capacity);
PA_API pa_status pa_bm_block_tables(const pa_block_manager *bm, const int32_t *seq_ids, int32_t num_seqs,
                                    int32_t *out, int32_t max_blocks_per_seq);
PA_API int32_t pa_bm_free_block_ids(const pa_block_manager *bm, int32_t *out, int32_t capacity);
PA_API pa_status pa_bm_block_info(const pa_block_manager *bm, int32_t block_id, int32_t *ref_count,
                                  int32_t *has_hash, uint64_t *hash, int32_t *num_token_ids);
PA_API int32_t pa_bm_lookup_hash(const pa_block_manager *bm, uint64_t hash);
PA_API int32_t pa_bm_num_hashes(const pa_block_manager *bm);
PA_API uint64_t pa_bm_block_hash(const int64_t *token_ids, int32_t num_tokens, int32_t has_prefix, uint64_t prefix);
PA_API uint64_t pa_bm_xxh64(const void *data, size_t len, uint64_t seed);

/*
 * pa_set_checked -- enable (1) or disable (0) extra device checks for calls
 * made after it on any thread: block ids outside [0, num_blocks) are then
 * recorded as PA_DEV_BAD_BLOCK (reads of them return zeros either way).
 */
PA_API pa_status pa_set_checked(int32_t enabled);

/*
 * pa_get_device_error -- synchronise `stream`, return the first device-side
 * error recorded on the current device since the last call (code 0 if none)
 * and clear it.  Returns PA_ERR_DEVICE_CHECK if an error was recorded.
 * code and where may be NULL.
 */
PA_API pa_status pa_get_device_error(pa_stream_t stream, int32_t *code, int64_t *where);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
