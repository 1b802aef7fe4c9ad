// pa_prefill.cu -- varlen causal prefill attention on 5th-generation tensor cores.
//
// What it computes [NV12 §12.6 flash_attn_varlen_func; NV05 prepare_prefill]:
// for sequence s with Lq new rows and Lk keys (c = Lk - Lq of them cached),
// query i at position c + i attends to keys 0..c+i (bottom-right causal;
// all Lk keys when causal == 0), keys read through the block table
// (prefix cache) or from contiguous rows.
//
// How (GB300 design): one CTA per (128-row query tile, sequence, q head).
//  * warp 0 (one thread) issues TMA copies: the Q tile once, then K and V
//    tiles of 128 keys into two-stage rings.  Boxes are {64 dims, 1 head,
//    R rows} with 128-byte swizzle (two boxes per 128-dim row); paged boxes
//    never straddle a block (R = gcd(block_size, 128)).
//  * warp 1 (one thread) owns the tensor cores: S = Q.K^T (M=N=128, K=128,
//    eight tcgen05.mma K=16 steps) into one of two TMEM buffers, then
//    O += P.V with V as an MN-major operand, O accumulating in TMEM.
//    tcgen05.commit arrives on mbarriers to free K/V stages, publish S and
//    release the P buffer.
//  * warps 4..7 (one thread per query row = TMEM lane) read S rows with
//    tcgen05.ld, apply scale and mask, keep the running max/sum in base 2,
//    and write P as bf16 into a 128-byte-swizzled shared-memory tile for
//    the P.V MMA.  O in TMEM is rescaled only when a row's max grows by
//    more than 2^8 (otherwise the stale max keeps P <= 256, exact enough in
//    bf16 and fp32); the final 1/l is applied in the epilogue.
//  * Every mbarrier wait is bounded; a timeout records PA_DEV_TIMEOUT and
//    the roles skip to the CTA-wide teardown.
// TMEM: S0 = columns 0..127, S1 = 128..255, O = 256..383 (512 allocated).
#include <math.h>

#include <algorithm>

#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int D = 128;
constexpr int BM = 128;                   // query rows per tile
constexpr int BN = 128;                   // keys per tile
constexpr int TILE_BYTES = BM * D * 2;    // 32 KiB
constexpr int HALF_BYTES = TILE_BYTES / 2;  // [128 rows][64 dims], 128-byte rows
constexpr int NTHREADS = 256;
constexpr int W_TMA = 0, W_MMA = 1, W_SOFT = 4;  // softmax warps 4..7

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;      // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;  // 2 stages
constexpr int OFF_P = OFF_V + 2 * TILE_BYTES;  // 2 buffers
constexpr int OFF_BAR = OFF_P + 2 * TILE_BYTES;
enum { B_Q = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9, B_SFREE = 11,
       B_PFULL = 13, B_PFREE = 15, NBAR = 17 };
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_FLAGS = OFF_TMEM + 8;
constexpr size_t SMEM_BYTES = OFF_FLAGS + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 256;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);  // Q, K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);   // P K-major, V MN-major
constexpr uint32_t SBO = 1024;  // 8 rows x 128 B between core-matrix groups
constexpr unsigned FULL = 0xffffffffu;

struct PrefillArgs {
    __nv_bfloat16 *out;
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *bt;
    int32_t max_blocks, num_seqs, Hq, group, mtiles;
    int32_t block_size, box_rows, paged, causal, num_blocks, checked;
    float scale_log2;
    DevError *err;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *flags, DevError *err,
                                              int where) {
    if (flags[0]) return false;
    if (mbar_wait(bar, parity)) return true;
    record_error(err, PA_DEV_TIMEOUT, where);
    flags[0] = 1;
    return false;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- which tile: the highest query tiles (the most keys) come first
    const int per = a.num_seqs * a.Hq;
    const int mt = a.mtiles - 1 - (int)(blockIdx.x / per);
    const int rem = (int)(blockIdx.x % per);
    const int s = rem / a.Hq, h = rem % a.Hq, kvh = h / a.group;
    const int q0 = a.cu_q[s], Lq = a.cu_q[s + 1] - q0;
    const int k0 = a.cu_k[s], Lk = a.cu_k[s + 1] - k0;
    if (Lq < 0 || Lk < Lq || (a.paged && Lk > a.max_blocks * a.block_size)) {
        if (threadIdx.x == 0 && mt == 0 && h == 0) record_error(a.err, PA_DEV_BAD_SEQLENS, s);
        return;
    }
    const int m0 = mt * BM;
    if (m0 >= Lq) return;  // the whole CTA leaves together
    const int c = Lk - Lq;
    const int last_row = min(m0 + BM, Lq) - 1;
    const int key_end = a.causal ? min(Lk, c + last_row + 1) : Lk;  // keys [0, key_end) are needed
    const int n_kv = (key_end + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if ((i >= B_SFREE && i < B_SFREE + 2) || (i >= B_PFULL && i < B_PFULL + 2)) cnt = 4;
            mbar_init(&bar[i], cnt);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == W_TMA) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            mbar_arrive_expect_tx(&bar[B_Q], TILE_BYTES);
            tma_load_3d_plain(smem + OFF_Q, &tmq, 0, h, q0 + m0, &bar[B_Q]);
            tma_load_3d_plain(smem + OFF_Q + HALF_BYTES, &tmq, 64, h, q0 + m0, &bar[B_Q]);
            const int R = a.box_rows;
            const int32_t *bt = a.bt + (int64_t)s * a.max_blocks;
            int issued = 0;  // K/V tiles whose copies were issued
            for (int j = 0; j < n_kv; ++j) {
                const int st = j & 1;
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                const int kb = j * BN;
                const int nsub = (min(BN, key_end - kb) + R - 1) / R;
                const uint32_t bytes = (uint32_t)nsub * R * D * 2;
                int rows[BN / 16];
                for (int sub = 0; sub < nsub; ++sub) {
                    const int key = kb + sub * R;
                    if (a.paged) {
                        const int blk = __ldg(bt + key / a.block_size);
                        if (a.checked && (blk < 0 || blk >= a.num_blocks))
                            record_error(a.err, PA_DEV_BAD_BLOCK, (long long)s * a.max_blocks + key / a.block_size);
                        // An invalid block id reads as zeros: TMA fills out-of-range boxes.
                        rows[sub] = (blk < 0 || blk >= a.num_blocks) ? -2 * R : blk * a.block_size + key % a.block_size;
                    } else {
                        rows[sub] = k0 + key;
                    }
                }
                if (!wait_or_abort(&bar[B_KEMPTY + st], ph ^ 1u, flags, a.err, 400)) break;
                mbar_arrive_expect_tx(&bar[B_KFULL + st], bytes);
                uint8_t *kd = smem + OFF_K + st * TILE_BYTES;
                for (int sub = 0; sub < nsub; ++sub) {
                    tma_load_3d_plain(kd + sub * R * 128, &tmk, 0, kvh, rows[sub], &bar[B_KFULL + st]);
                    tma_load_3d_plain(kd + HALF_BYTES + sub * R * 128, &tmk, 64, kvh, rows[sub], &bar[B_KFULL + st]);
                }
                if (!wait_or_abort(&bar[B_VEMPTY + st], ph ^ 1u, flags, a.err, 401)) {
                    issued = j + 1;  // K of tile j is in flight
                    break;
                }
                mbar_arrive_expect_tx(&bar[B_VFULL + st], bytes);
                uint8_t *vd = smem + OFF_V + st * TILE_BYTES;
                for (int sub = 0; sub < nsub; ++sub) {
                    tma_load_3d_plain(vd + sub * R * 128, &tmv, 0, kvh, rows[sub], &bar[B_VFULL + st]);
                    tma_load_3d_plain(vd + HALF_BYTES + sub * R * 128, &tmv, 64, kvh, rows[sub], &bar[B_VFULL + st]);
                }
                issued = j + 1;
            }
            if (flags[0]) {
                // Let issued copies land before the CTA's shared memory is released.
                (void)mbar_wait(&bar[B_Q], 0);
                for (int j = max(0, issued - 2); j < issued; ++j) {
                    (void)mbar_wait(&bar[B_KFULL + (j & 1)], (uint32_t)(j >> 1) & 1u);
                    (void)mbar_wait(&bar[B_VFULL + (j & 1)], (uint32_t)(j >> 1) & 1u);
                }
            }
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t q_addr = smem_addr(smem + OFF_Q);
            int committed_pv = -1;
            auto issue_pv = [&](int jj) -> bool {
                const int pb = jj & 1;
                const uint32_t ph = (uint32_t)(jj >> 1) & 1u;
                if (!wait_or_abort(&bar[B_PFULL + pb], ph, flags, a.err, 410)) return false;
                if (!wait_or_abort(&bar[B_VFULL + pb], ph, flags, a.err, 411)) return false;
                tc_fence_after();
                const uint32_t p_addr = smem_addr(smem + OFF_P + pb * TILE_BYTES);
                const uint32_t v_addr = smem_addr(smem + OFF_V + pb * TILE_BYTES);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint64_t ad = smem_desc_sw128(p_addr + (k >> 2) * HALF_BYTES + (k & 3) * 32, 16, SBO);
                    const uint64_t bd = smem_desc_sw128(v_addr + k * 16 * 128, HALF_BYTES, SBO);
                    mma_bf16_ss(tmem + COL_O, ad, bd, IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&bar[B_PFREE + pb]);
                mma_commit(&bar[B_VEMPTY + pb]);
                committed_pv = jj;
                return true;
            };
            bool ok = wait_or_abort(&bar[B_Q], 0, flags, a.err, 412);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j & 1;
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                ok = wait_or_abort(&bar[B_KFULL + st], ph, flags, a.err, 413);
                if (ok && j >= 2) ok = wait_or_abort(&bar[B_SFREE + st], ph ^ 1u, flags, a.err, 414);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_addr = smem_addr(smem + OFF_K + st * TILE_BYTES);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t ad = smem_desc_sw128(q_addr + (k >> 2) * HALF_BYTES + (k & 3) * 32, 16, SBO);
                    const uint64_t bd = smem_desc_sw128(k_addr + (k >> 2) * HALF_BYTES + (k & 3) * 32, 16, SBO);
                    mma_bf16_ss(tmem + st * BN, ad, bd, IDESC_S, k > 0 ? 1u : 0u);
                }
                mma_commit(&bar[B_KEMPTY + st]);
                mma_commit(&bar[B_SFULL + st]);
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok) ok = issue_pv(n_kv - 1);
            if (!ok && committed_pv >= 0) {
                // Let the issued MMAs finish before TMEM is released.
                (void)mbar_wait(&bar[B_PFREE + (committed_pv & 1)], (uint32_t)(committed_pv >> 1) & 1u);
            }
        }
    } else if (warp >= W_SOFT) {
        // ------------------------------------------------------------ softmax
        const int wq = warp - W_SOFT;
        const int row = wq * 32 + lane;  // tile row == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        const int i = m0 + row;          // query index in the sequence (>= Lq: padding row)
        const int pos = c + i;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            const int sb = j & 1;
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            // Waits in this role are made warp-uniform: tcgen05.ld/st are warp-collective.
            if (!(ok = __all_sync(FULL, wait_or_abort(&bar[B_SFULL + sb], ph, flags, a.err, 420)))) break;
            tc_fence_after();
            float x[BN];
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(t_lane + sb * BN + cc * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) x[cc * 32 + e] = __uint_as_float(r[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SFREE + sb]);

            const int kb = j * BN;
            const int lim = (a.causal ? min(pos, Lk - 1) : Lk - 1) - kb;  // keys kb+k with k <= lim
            float tmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < BN; ++k) {
                x[k] = (k <= lim) ? x[k] * a.scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, x[k]);
            }
            const bool grow = tmax > m_run + 8.f;
            const float m_new = grow ? tmax : m_run;
            const float alpha = grow ? fast_exp2(m_run - m_new) : 1.f;
            if (__any_sync(FULL, grow) && j > 0) {
                // O holds sum_{j' < j} P_j' V_j': wait for the last P.V, then rescale.
                const int pj = j - 1;
                ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + (pj & 1)], (uint32_t)(pj >> 1) & 1u, flags, a.err, 421));
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(t_lane + COL_O + cc * 32, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(t_lane + COL_O + cc * 32, r);
                    }
                    tmem_st_wait();
                }
            }
            l_run *= alpha;
            m_run = m_new;
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            if (ok && j >= 2) ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + sb], ph ^ 1u, flags, a.err, 422));
            if (ok) {
                const uint32_t prow = smem_addr(smem + OFF_P + sb * TILE_BYTES) + row * 128;
                float rs = 0.f;
#pragma unroll
                for (int kc = 0; kc < BN / 8; ++kc) {
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = fast_exp2(x[kc * 8 + e] - m_use);
                        rs += p[e];
                    }
                    const uint32_t addr = prow + (kc >> 3) * HALF_BYTES + (((kc & 7) ^ (row & 7)) << 4);
                    st_shared_v4(addr, pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]), pack_bf16(p[4], p[5]),
                                 pack_bf16(p[6], p[7]));
                }
                l_run += rs;
                if (j == n_kv - 1 && key_end - kb < BN) {
                    // Rows past the last needed key hold stale or unloaded data:
                    // zero them so 0 * garbage cannot reach O.
                    ok = __all_sync(FULL, wait_or_abort(&bar[B_VFULL + sb], ph, flags, a.err, 423));
                    if (ok && row >= key_end - kb) {
                        const uint32_t vrow = smem_addr(smem + OFF_V + sb * TILE_BYTES) + row * 128;
#pragma unroll
                        for (int q16 = 0; q16 < 8; ++q16) {
                            st_shared_v4(vrow + q16 * 16, 0, 0, 0, 0);
                            st_shared_v4(vrow + HALF_BYTES + q16 * 16, 0, 0, 0, 0);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_PFULL + sb]);
        }
        // ---- epilogue: O / l -> bf16 rows of this tile that exist
        const int pj = n_kv - 1;
        if (ok) ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + (pj & 1)], (uint32_t)(pj >> 1) & 1u, flags, a.err, 424));
        if (__all_sync(FULL, ok)) {
            tc_fence_after();
            const float inv = 1.f / l_run;
            const bool valid = i < Lq;
            __nv_bfloat16 *orow = a.out + ((int64_t)(q0 + i) * a.Hq + h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(t_lane + COL_O + cc * 32, r);
                tmem_ld_wait();
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pack_bf16(__uint_as_float(r[8 * e + 0]) * inv, __uint_as_float(r[8 * e + 1]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * e + 2]) * inv, __uint_as_float(r[8 * e + 3]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * e + 4]) * inv, __uint_as_float(r[8 * e + 5]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * e + 6]) * inv, __uint_as_float(r[8 * e + 7]) * inv));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

int g_attr_done[64] = {};

}  // namespace
}  // namespace pa

extern "C" pa_status pa_prefill_varlen(void *out, const void *q, int64_t q_row_stride, int32_t total_q,
                                       const void *k, const void *v, int64_t kv_row_stride, int32_t total_k,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs,
                                       int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t num_blocks, float softmax_scale, int32_t causal,
                                       pa_stream_t stream) {
    using namespace pa;
    (void)max_seqlen_k;
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PA_OK;
    if (!out || !q || !k || !v || !cu_seqlens_q || !cu_seqlens_k) return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
    if (head_dim != D) return fail(PA_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
    if (q_row_stride < (int64_t)num_q_heads * D || q_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "q_row_stride must be >= num_q_heads*head_dim and a multiple of 8");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(PA_ERR_INVALID_ARG, "out/q/k/v pointers must be 16-byte aligned");
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
        return fail(PA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
    const bool paged = block_tables != nullptr;
    int R = 128;
    CUtensorMap tq, tk, tv;
    pa_status st = encode_tensor_map_3d(&tq, q, D, num_q_heads, total_q, D * 2, q_row_stride * 2, 64, BM, true);
    if (st != PA_OK) return st;
    if (paged) {
        if (block_size <= 0 || block_size % 16)
            return fail(PA_ERR_UNSUPPORTED, "block_size %d (must be a positive multiple of 16)", block_size);
        if (max_blocks_per_seq <= 0 || num_blocks <= 0)
            return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq and num_blocks must be positive");
        if ((int64_t)num_blocks * block_size > 0x7fffffffLL ||
            (int64_t)max_blocks_per_seq * block_size > 0x7fffffffLL)
            return fail(PA_ERR_UNSUPPORTED, "pool or table too large for 32-bit slot indices");
        while (block_size % R) R >>= 1;  // gcd(block_size, 128) in {16, 32, 64, 128}
        const int64_t slots = (int64_t)num_blocks * block_size;
        const int64_t rs = (int64_t)num_kv_heads * D * 2;
        st = encode_tensor_map_3d(&tk, k, D, num_kv_heads, slots, D * 2, rs, 64, R, true);
        if (st == PA_OK) st = encode_tensor_map_3d(&tv, v, D, num_kv_heads, slots, D * 2, rs, 64, R, true);
    } else {
        if (total_k <= 0) return fail(PA_ERR_INVALID_ARG, "total_k must be positive for contiguous k/v");
        if (kv_row_stride < (int64_t)num_kv_heads * D || kv_row_stride % 8)
            return fail(PA_ERR_INVALID_ARG, "kv_row_stride must be >= num_kv_heads*head_dim and a multiple of 8");
        st = encode_tensor_map_3d(&tk, k, D, num_kv_heads, total_k, D * 2, kv_row_stride * 2, 64, R, true);
        if (st == PA_OK) st = encode_tensor_map_3d(&tv, v, D, num_kv_heads, total_k, D * 2, kv_row_stride * 2, 64, R, true);
    }
    if (st != PA_OK) return st;

    PrefillArgs A;
    A.out = static_cast<__nv_bfloat16 *>(out);
    A.cu_q = cu_seqlens_q;
    A.cu_k = cu_seqlens_k;
    A.bt = block_tables;
    A.max_blocks = paged ? max_blocks_per_seq : 0;
    A.num_seqs = num_seqs;
    A.Hq = num_q_heads;
    A.group = num_q_heads / num_kv_heads;
    A.mtiles = (max_seqlen_q + BM - 1) / BM;
    A.block_size = paged ? block_size : 1;
    A.box_rows = R;
    A.paged = paged ? 1 : 0;
    A.causal = causal ? 1 : 0;
    A.num_blocks = num_blocks;
    A.checked = checked_mode() ? 1 : 0;
    A.scale_log2 = softmax_scale * 1.4426950408889634f;
    A.err = device_error_ptr();

    const int64_t grid = (int64_t)A.mtiles * num_seqs * num_q_heads;
    if (grid > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "grid too large");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !g_attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_kernel)");
        g_attr_done[dev] = 1;
    }
    prefill_kernel<<<(unsigned)grid, NTHREADS, SMEM_BYTES, reinterpret_cast<cudaStream_t>(stream)>>>(tq, tk, tv, A);
    return check_launch("prefill_kernel");
}
