// pa_store.cu -- store_kvcache scatter and the slot_mapping builders.
//
// store: [NV12 §12.6 "Triton KV Cache Store Kernel"] each token whose slot
// is not negative copies its Hkv*D K values to k_cache[slot*Hkv*D ...] and
// its V values to v_cache.  It is a pure copy: a warp copies one (token,
// K-or-V) row at a time (2 KiB at Hkv=8, D=128) with 16-byte non-allocating
// loads, up to four per lane in flight before their stores, so each row
// moves as fully coalesced 512-byte warp transactions; a grid of at most
// eight CTAs per SM strides over the rows.  HBM-bound at 8 KiB of traffic per
// stored token (2 KiB read + 2 KiB write for each of K and V).
//
// All three kernels are programmatic dependent launches: they start by
// waiting for the preceding work on the stream (griddepcontrol.wait) and
// then release the work queued behind them.
//
// slot mapping: [PA3 §3/§4] the slot of logical position p of a sequence is
// block_table[p / B] * B + p % B; the decode form takes p = ctx - 1, the
// prefill form p = c + i for the uncached suffix of each sequence.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int STORE_THREADS = 256;

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(STORE_THREADS) store_kvcache_kernel(
    const uint4 *__restrict__ key, int64_t key_stride16, const uint4 *__restrict__ value,
    int64_t value_stride16, uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
    const int32_t *__restrict__ slot_mapping, int32_t row16, int64_t num_slots, int32_t num_tokens,
    DevError *err) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int64_t nrows = 2LL * num_tokens;  // row r: token r / 2, K (even) or V (odd)
    const int64_t wstride = (int64_t)gridDim.x * (STORE_THREADS / 32);
    for (int64_t r = (int64_t)blockIdx.x * (STORE_THREADS / 32) + (threadIdx.x >> 5); r < nrows; r += wstride) {
        const int64_t token = r >> 1;
        const bool is_v = (r & 1) != 0;
        const int32_t slot = __ldg(slot_mapping + token);
        if (slot < 0) continue;  // padding
        if (slot >= num_slots) {
            if (lane == 0 && !is_v) record_error(err, PA_DEV_BAD_SLOT, token);
            continue;
        }
        const uint4 *src = is_v ? value + token * value_stride16 : key + token * key_stride16;
        uint4 *dst = (is_v ? v_cache : k_cache) + static_cast<int64_t>(slot) * row16;
        for (int j0 = lane; j0 < row16; j0 += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + 32 * u < row16) v[u] = ld_stream16(src + j0 + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + 32 * u < row16) dst[j0 + 32 * u] = v[u];
        }
    }
}

__global__ void slot_mapping_decode_kernel(int32_t *__restrict__ slot_mapping,
                                           const int32_t *__restrict__ block_tables,
                                           int32_t max_blocks, const int32_t *__restrict__ ctx_lens,
                                           int32_t batch, int32_t block_size, DevError *err) {
    pdl_wait_then_release();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int32_t ctx = ctx_lens[b];
    if (ctx <= 0 || ctx > static_cast<int64_t>(max_blocks) * block_size) {
        if (ctx != 0) record_error(err, PA_DEV_BAD_CONTEXT, b);
        slot_mapping[b] = -1;
        return;
    }
    const int32_t p = ctx - 1;
    slot_mapping[b] = block_tables[static_cast<int64_t>(b) * max_blocks + p / block_size] * block_size +
                      p % block_size;
}

__global__ void slot_mapping_prefill_kernel(int32_t *__restrict__ slot_mapping,
                                            const int32_t *__restrict__ block_tables,
                                            int32_t max_blocks, const int32_t *__restrict__ cu_q,
                                            const int32_t *__restrict__ cu_k, int32_t num_seqs,
                                            int32_t total_q, int32_t block_size, DevError *err) {
    pdl_wait_then_release();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total_q) return;
    // The sequence owning query row t: the last s with cu_q[s] <= t.
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int32_t lq = cu_q[s + 1] - cu_q[s];
    const int32_t lk = cu_k[s + 1] - cu_k[s];
    if (lq < 0 || lk < lq || t >= cu_q[s + 1] ||
        lk > static_cast<int64_t>(max_blocks) * block_size) {
        record_error(err, PA_DEV_BAD_SEQLENS, s);
        slot_mapping[t] = -1;
        return;
    }
    const int32_t p = (lk - lq) + (t - cu_q[s]);
    slot_mapping[t] = block_tables[static_cast<int64_t>(s) * max_blocks + p / block_size] * block_size +
                      p % block_size;
}

}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_store_kvcache(const void *key, int64_t key_row_stride, const void *value,
                           int64_t value_row_stride, void *k_cache, void *v_cache,
                           const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int64_t num_slots, pa_stream_t stream) {
    using namespace pa;
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_kv_heads <= 0 || head_dim <= 0) return fail(PA_ERR_INVALID_ARG, "bad head shape");
    if (head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
    if (num_slots <= 0) return fail(PA_ERR_INVALID_ARG, "num_slots <= 0");
    if (num_tokens > 0x7fffffff / 2) return fail(PA_ERR_INVALID_ARG, "num_tokens too large");
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (key_row_stride < row || value_row_stride < row)
        return fail(PA_ERR_INVALID_ARG, "row stride smaller than num_kv_heads*head_dim");
    if (key_row_stride % 8 || value_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "row strides must be multiples of 8 elements");
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "key/value/cache pointers must be 16-byte aligned");
    const int32_t row16 = static_cast<int32_t>(row / 8);
    const int sms = sm_count();
    if (sms <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    // One warp per row and step; at most 8 CTAs of 8 warps per SM.
    const int64_t rows = 2LL * num_tokens, warps = STORE_THREADS / 32;
    const int64_t grid = std::min<int64_t>((rows + warps - 1) / warps, 8LL * sms);
    return launch_pdl(store_kvcache_kernel, dim3(static_cast<unsigned>(grid)), dim3(STORE_THREADS), 0,
                      reinterpret_cast<cudaStream_t>(stream), "store_kvcache_kernel", static_cast<const uint4 *>(key),
                      (int64_t)(key_row_stride / 8), static_cast<const uint4 *>(value),
                      (int64_t)(value_row_stride / 8), static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                      slot_mapping, row16, num_slots, num_tokens, device_error_ptr());
}

pa_status pa_slot_mapping_decode(int32_t *slot_mapping, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                 int32_t batch, int32_t block_size, pa_stream_t stream) {
    using namespace pa;
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch < 0");
    if (batch == 0) return PA_OK;
    if (!slot_mapping || !block_tables || !context_lens) return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (block_size <= 0 || max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "block_size and max_blocks_per_seq must be positive");
    return launch_pdl(slot_mapping_decode_kernel, dim3((batch + 127) / 128), dim3(128), 0,
                      reinterpret_cast<cudaStream_t>(stream), "slot_mapping_decode_kernel", slot_mapping,
                      block_tables, max_blocks_per_seq, context_lens, batch, block_size, device_error_ptr());
}

pa_status pa_slot_mapping_prefill(int32_t *slot_mapping, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                  const int32_t *cu_seqlens_k, int32_t num_seqs, int32_t total_q,
                                  int32_t block_size, pa_stream_t stream) {
    using namespace pa;
    if (num_seqs < 0 || total_q < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    if (!slot_mapping || !block_tables || !cu_seqlens_q || !cu_seqlens_k)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (block_size <= 0 || max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "block_size and max_blocks_per_seq must be positive");
    return launch_pdl(slot_mapping_prefill_kernel, dim3((total_q + 255) / 256), dim3(256), 0,
                      reinterpret_cast<cudaStream_t>(stream), "slot_mapping_prefill_kernel", slot_mapping,
                      block_tables, max_blocks_per_seq, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                      block_size, device_error_ptr());
}

}  // extern "C"
