// pa_decode.cu -- paged split-KV GQA decode attention for sm_103a.
//
// What it computes [NV12 §12.6 flash_attn_with_kvcache; VD §3]: for each
// sequence b and query head h (kv head g = h / G, G = Hq/Hkv),
//   out[b,h] = softmax_p(scale * q[b,h] . K[slot(b,p), g]) V[slot(b,p), g],
// p < context_lens[b], slot(b,p) = block_tables[b][p/B]*B + p%B [PA3 §3].
//
// How (GB300 design):
//  * Work items are (sequence, kv head, chunk of `chunk_tokens` positions).
//    Every CTA rebuilds the per-sequence chunk prefix sum from context_lens
//    in shared memory and walks items blockIdx.x, +gridDim.x, ... (a
//    persistent grid of one CTA per SM).  Items of the 8 kv heads of one
//    chunk are adjacent, so neighbouring CTAs stream the same 2 KiB token
//    rows at the same time.
//  * One producer warp issues TMA tile loads (cp.async.bulk.tensor, 64 rows x
//    256 B per K or V tile; a row is one token of one kv head) into a
//    5-stage shared-memory ring guarded by mbarriers, plus a bulk copy of the
//    item's G query rows.  Tiles never straddle a block: the TMA box is
//    gcd(B, 64) rows, and each box is addressed through the block table.
//  * Four consumer warps each own 16 rows of a tile.  Q.K: 8 lanes per row,
//    16 dims per lane, the whole GQA group's q (G x 16 values) in registers,
//    partial sums combined with a shuffle reduce-scatter (each K byte is read
//    from shared memory once for all G heads).  Online softmax in base 2 per
//    warp, then P.V with each lane owning 4 output dims of all G heads.
//  * Item end: the 4 warp states are merged in shared memory.  A one-chunk
//    sequence writes bf16 output directly; otherwise the chunk's (m, l, o)
//    partial goes to the workspace and the CTA that finishes the last chunk
//    partial goes to the workspace and a small merge kernel, queued behind
//    this one with programmatic dependent launch, combines the partials.
//  * All waits are bounded; a timeout records PA_DEV_TIMEOUT and the warps
//    finish their loops without waiting, keeping every named barrier paired.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int D = 128;
constexpr int ROW_BYTES = D * 2;  // one token row of one kv head
constexpr int TILE = 64;          // rows per pipeline stage
constexpr int WPG = 4;            // consumer warps per group
constexpr int TPW = TILE / WPG;   // rows per consumer warp per tile
constexpr int kMaxBatch = 2048;
constexpr int kMaxSplits = 512;
constexpr unsigned FULL = 0xffffffffu;

template <int G>
struct Cfg {
    static constexpr int NGRP = (G <= 4) ? 2 : 1;  // consumer groups; tiles alternate between them
    static constexpr int NCW = WPG * NGRP;         // consumer warps
    static constexpr int PRODUCER = NCW;           // warp that issues the TMA copies
    static constexpr int MERGER = NCW + 1;         // warp that finishes work items
    static constexpr int NTHREADS = (NCW + 2) * 32;
    // Stage s only ever holds tiles of group s % NGRP, so each full/empty
    // barrier has waiters of one group only and a parity wait can never see a
    // phase two steps old (another group's pending copy) as its own.
    static constexpr int STAGES = 4;
    static_assert(STAGES % NGRP == 0, "a stage must belong to a single consumer group");
    static constexpr int LPT = (G <= 4) ? 8 : 16;  // lanes per row in Q.K
    static constexpr int DPL = D / LPT;            // dims per lane in Q.K
    static constexpr int RPR = 32 / LPT;           // rows per warp per Q.K round
    static constexpr int ROUNDS = TPW / RPR;
    static constexpr int STAGE_BYTES = 2 * TILE * ROW_BYTES;
    static constexpr int Q_BYTES = G * ROW_BYTES;
    static constexpr int SLOT_FLOATS = NCW * G * (D + 2);      // o[NCW][G][D], then (m,l)[NCW][G]
    static constexpr int OFF_Q = STAGES * STAGE_BYTES;          // q slots [2][G][D] bf16
    static constexpr int OFF_S = OFF_Q + 2 * Q_BYTES;           // scores [NCW][TPW][G] f32
    static constexpr int OFF_SLOT = OFF_S + NCW * TPW * G * 4;  // merge slots [2][SLOT_FLOATS] f32
    static constexpr int OFF_BAR = OFF_SLOT + 2 * SLOT_FLOATS * 4;
    static constexpr int NBAR = 2 * STAGES + 8;  // full, empty, qfull[2], qempty[2], done[2], free[2]
    static constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;
    static constexpr int OFF_BID = OFF_FLAGS + 16;  // producer's block ids [2][32] int
    static constexpr int OFF_CUM = OFF_BID + 256;   // [batch+1] int, then clamped ctx [batch] int
    static constexpr size_t smem_bytes(int batch) { return OFF_CUM + 4 * (size_t)(2 * batch + 1) + 1024; }
    static_assert(smem_bytes(kMaxBatch) <= 232448, "shared memory budget");
};

struct DecodeArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    int64_t q_row_stride;
    const int32_t *block_tables;
    const int32_t *ctx_lens;
    int32_t max_blocks;
    int32_t batch, Hq, Hkv, block_size, box_rows, num_blocks;
    float scale_log2;
    int32_t chunk_tokens;
    int32_t max_splits;
    int32_t ctx_limit;  // min(max_blocks*B, max_splits*chunk_tokens)
    float *ws_o;        // [batch][Hq][max_splits][D]
    float2 *ws_ml;      // [batch][Hq][max_splits]  (m, l) in base 2
    DevError *err;
    int32_t checked;
};

__device__ __forceinline__ int clamp_ctx(const DecodeArgs &a, int b, bool report) {
    int ctx = __ldg(a.ctx_lens + b);
    if (ctx < 0 || ctx > a.ctx_limit) {
        if (report) record_error(a.err, PA_DEV_BAD_CONTEXT, b);
        ctx = ctx < 0 ? 0 : a.ctx_limit;
    }
    return ctx;
}

struct Item {
    int b, g, c, nsplit, p_begin, p_end, ntiles;
};

__device__ __forceinline__ Item decode_item(const DecodeArgs &a, const int *cum, const int *ctx_s, int item) {
    Item it;
    const int chunk_id = item / a.Hkv;
    it.g = item - chunk_id * a.Hkv;
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= chunk_id) lo = mid; else hi = mid - 1;
    }
    it.b = lo;
    it.c = chunk_id - cum[lo];
    it.nsplit = cum[lo + 1] - cum[lo];
    const int ctx = ctx_s[lo];
    it.p_begin = it.c * a.chunk_tokens;
    it.p_end = min(ctx, it.p_begin + a.chunk_tokens);
    it.ntiles = (it.p_end - it.p_begin + TILE - 1) / TILE;
    return it;
}

// Sum over the LPT lanes of a row group of v[h], scattered so that lane li
// ends with the total of head li / (LPT / G).
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int li) {
#pragma unroll
    for (int step = 0, off = LPT / 2; off >= 1; ++step, off >>= 1) {
        if ((G >> step) > 1) {
            const int half = G >> (step + 1);
            const bool upper = (li & off) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
                const float send = upper ? v[k] : v[k + half];
                const float keep = upper ? v[k + half] : v[k];
                v[k] = keep + __shfl_xor_sync(FULL, send, off);
            }
        } else {
            v[0] += __shfl_xor_sync(FULL, v[0], off);
        }
    }
    return v[0];
}

// Bounded wait that turns a timeout into a recorded error and a CTA-wide abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *flags,
                                              const DecodeArgs &a, int where) {
    if (flags[0]) return false;
    if (mbar_wait(bar, parity)) return true;
    record_error(a.err, PA_DEV_TIMEOUT, where);
    flags[0] = 1;
    return false;
}

template <int G>
__global__ void __launch_bounds__(Cfg<G>::NTHREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
    using C = Cfg<G>;
    extern __shared__ uint8_t smem_raw[];
    // Align to 1 KiB by pointer arithmetic on the __shared__ array, so every
    // pointer below stays in the shared address space (ld/st.shared).
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    int *cum = reinterpret_cast<int *>(smem + C::OFF_CUM);
    int *ctx_s = cum + a.batch + 1;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    uint64_t *qfull = empty + C::STAGES;
    uint64_t *qempty = qfull + 2;
    uint64_t *done = qempty + 2;
    uint64_t *sfree = done + 2;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WPG);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&qfull[k], 1);
            mbar_init(&qempty[k], C::NCW);
            mbar_init(&done[k], C::NCW);
            mbar_init(&sfree[k], 1);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == C::PRODUCER && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    // Chunk prefix sum: cum[b+1] = sum_{b' <= b} ceil(ctx_b' / chunk_tokens).
    if (warp == 0) {
        int run = 0;
        if (lane == 0) cum[0] = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const int b = base + lane;
            int x = 0;
            if (b < a.batch) {
                const int ctx = clamp_ctx(a, b, blockIdx.x == 0);
                ctx_s[b] = ctx;
                x = (ctx + a.chunk_tokens - 1) / a.chunk_tokens;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, x, o);
                if (lane >= o) x += y;
            }
            if (b < a.batch) cum[b + 1] = run + x;
            run += __shfl_sync(FULL, x, 31);
        }
    }
    __syncthreads();
    // Sequences with no context produce zeros.
    if (warp < C::NCW) {
        for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
            if (ctx_s[b] != 0) continue;
            uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)b * a.Hq * D);
            for (int j = threadIdx.x; j < a.Hq * D / 8; j += C::NCW * 32) o[j] = make_uint4(0, 0, 0, 0);
        }
    }
    __syncthreads();
    const int total_items = cum[a.batch] * a.Hkv;
    // The split-merge kernel queued behind this grid may be scheduled now; it
    // waits (griddepcontrol.wait) until this grid's results are visible.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ------------------------------------------------------------------ producer
    if (warp == C::PRODUCER) {
        // Lane j holds the block id of logical block (p_begin / B + j) of an
        // item; ids of item k+1 are fetched while lane 0 issues item k.
        int *bid_s = reinterpret_cast<int *>(smem + C::OFF_BID);
        auto fetch_ids = [&](int item) -> int {
            if (item >= total_items) return -1;
            const Item I = decode_item(a, cum, ctx_s, item);
            const int first = I.p_begin / a.block_size;
            const int nblk = (I.p_end - 1) / a.block_size - first + 1;
            return lane < nblk ? __ldg(a.block_tables + (int64_t)I.b * a.max_blocks + first + lane) : -1;
        };
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0, k = 0, kq = 0;  // tiles issued, items seen, query copies issued
        bool ok = true;
        int ids = fetch_ids(blockIdx.x);
        for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++k) {
            bid_s[(k & 1) * 32 + lane] = ids;
            __syncwarp();
            ids = fetch_ids(item + gridDim.x);  // consumed next iteration
            if (lane == 0) {
                const Item I = decode_item(a, cum, ctx_s, item);
                const int first = I.p_begin / a.block_size;
                const int nblk = (I.p_end - 1) / a.block_size - first + 1;
                const int *bid = bid_s + (k & 1) * 32;
                if (!wait_or_abort(&qempty[k & 1], ((k >> 1) & 1) ^ 1, flags, a, 100)) ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(&qfull[k & 1], G * ROW_BYTES);
                    bulk_load(smem + C::OFF_Q + (k & 1) * C::Q_BYTES,
                              a.q + (int64_t)I.b * a.q_row_stride + (int64_t)I.g * G * D, G * ROW_BYTES,
                              &qfull[k & 1]);
                    ++kq;
                }
                for (int t = 0; ok && t < I.ntiles; ++t, ++it) {
                    const int stage = it % C::STAGES;
                    if (!wait_or_abort(&empty[stage], ((it / C::STAGES) & 1) ^ 1, flags, a, 101)) {
                        ok = false;
                        break;
                    }
                    const int p0 = I.p_begin + t * TILE;
                    const int rows = min(TILE, I.p_end - p0);
                    const int nsub = (rows + a.box_rows - 1) / a.box_rows;
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)nsub * a.box_rows * ROW_BYTES * 2);
                    uint8_t *ks = smem + stage * C::STAGE_BYTES;
                    uint8_t *vs = ks + TILE * ROW_BYTES;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int ps = p0 + sub * a.box_rows;
                        const int lb = ps / a.block_size - first;
                        const int blk = nblk <= 32 ? bid[lb]
                                                   : __ldg(a.block_tables + (int64_t)I.b * a.max_blocks + first + lb);
                        if (a.checked && (blk < 0 || blk >= a.num_blocks))
                            record_error(a.err, PA_DEV_BAD_BLOCK,
                                         (long long)I.b * a.max_blocks + ps / a.block_size);
                        long long slot = (long long)blk * a.block_size + ps % a.block_size;
                        // An invalid block id reads as zeros: TMA fills out-of-range boxes.
                        if (blk < 0 || blk >= a.num_blocks) slot = -2LL * a.box_rows;
                        tma_load_3d(ks + sub * a.box_rows * ROW_BYTES, &tmk, 0, I.g, (int)slot, &full[stage], pol);
                        tma_load_3d(vs + sub * a.box_rows * ROW_BYTES, &tmv, 0, I.g, (int)slot, &full[stage], pol);
                    }
                }
            }
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (!ok && lane == 0) {
            // Let the copies already issued land before the CTA's shared memory goes away.
            for (uint32_t j = 0; j < C::STAGES && j < it; ++j) {
                const uint32_t x = it - 1 - j;
                (void)mbar_wait(&full[x % C::STAGES], (x / C::STAGES) & 1);
            }
            for (uint32_t j = 0; j < 2 && j < kq; ++j) {
                const uint32_t x = kq - 1 - j;
                (void)mbar_wait(&qfull[x & 1], (x >> 1) & 1);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ merger
    if (warp == C::MERGER) {
        float *slot_base = reinterpret_cast<float *>(smem + C::OFF_SLOT);
        uint32_t k = 0;
        for (int item = blockIdx.x; item < total_items; item += gridDim.x, ++k) {
            const Item I = decode_item(a, cum, ctx_s, item);
            const bool ok = wait_or_abort(&done[k & 1], (k >> 1) & 1, flags, a, 300);
            const float *so = slot_base + (k & 1) * C::SLOT_FLOATS;
            const float *sml = so + C::NCW * G * D;
            float O[G][4], M[G], L[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                M[h] = -INFINITY;
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) M[h] = fmaxf(M[h], sml[(w * G + h) * 2]);
                L[h] = 0.f;
                O[h][0] = O[h][1] = O[h][2] = O[h][3] = 0.f;
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) {
                    const float f = fast_exp2(sml[(w * G + h) * 2] - M[h]);
                    L[h] = fmaf(sml[(w * G + h) * 2 + 1], f, L[h]);
                    const float4 v = *reinterpret_cast<const float4 *>(so + (w * G + h) * D + 4 * lane);
                    O[h][0] = fmaf(v.x, f, O[h][0]);
                    O[h][1] = fmaf(v.y, f, O[h][1]);
                    O[h][2] = fmaf(v.z, f, O[h][2]);
                    O[h][3] = fmaf(v.w, f, O[h][3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[k & 1]);
            if (!ok) continue;
            const int64_t bh0 = (int64_t)I.b * a.Hq + (int64_t)I.g * G;  // first q-head row of (b, g)
            if (I.nsplit == 1) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float inv = 1.f / L[h];
                    __nv_bfloat162 lo = __floats2bfloat162_rn(O[h][0] * inv, O[h][1] * inv);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(O[h][2] * inv, O[h][3] * inv);
                    uint2 pk;
                    pk.x = *reinterpret_cast<uint32_t *>(&lo);
                    pk.y = *reinterpret_cast<uint32_t *>(&hi);
                    *reinterpret_cast<uint2 *>(a.out + (bh0 + h) * D + 4 * lane) = pk;
                }
                continue;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const int64_t pi = (bh0 + h) * a.max_splits + I.c;
                *reinterpret_cast<float4 *>(a.ws_o + pi * D + 4 * lane) =
                    make_float4(O[h][0], O[h][1], O[h][2], O[h][3]);
                if (lane == 0) a.ws_ml[pi] = make_float2(M[h], L[h]);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int grp = warp / WPG, wig = warp % WPG;
    const int rg = lane / C::LPT, li = lane % C::LPT;
    float *sbuf = reinterpret_cast<float *>(smem + C::OFF_S) + warp * TPW * G;  // [TPW][G]
    const uint32_t sbuf_a = smem_addr(sbuf);
    float *slot_base = reinterpret_cast<float *>(smem + C::OFF_SLOT);

    float qf[G][C::DPL];
    float m_run[G], l_run[G], o[G][4];
    uint32_t it = 0, k = 0;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x, ++k) {
        const Item I = decode_item(a, cum, ctx_s, item);
        if (wait_or_abort(&qfull[k & 1], (k >> 1) & 1, flags, a, 200 + warp)) {
            const uint32_t qa = smem_addr(smem + C::OFF_Q + (k & 1) * C::Q_BYTES);
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int part = 0; part < C::DPL / 8; ++part) {
                    const uint4 w = ld_shared_v4(qa + h * ROW_BYTES + part * 128 + 16 * li);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qf[h][part * 8 + 2 * e] = bf16lo(ww[e]) * a.scale_log2;
                        qf[h][part * 8 + 2 * e + 1] = bf16hi(ww[e]) * a.scale_log2;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[k & 1]);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_run[h] = -INFINITY;
            l_run[h] = 0.f;
            o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;
        }
        for (int t = 0; t < I.ntiles; ++t, ++it) {
            if ((int)(it % C::NGRP) != grp) continue;
            const int stage = it % C::STAGES;
            if (wait_or_abort(&full[stage], (it / C::STAGES) & 1, flags, a, 210 + warp)) {
                const uint32_t ks = smem_addr(smem + stage * C::STAGE_BYTES);
                const uint32_t vsa = ks + TILE * ROW_BYTES;
                const int nvalid = min(TILE, I.p_end - (I.p_begin + t * TILE));
                // ---- scores for rows wig*TPW + r*RPR + rg
                uint4 kw[C::ROUNDS][C::DPL / 8];
#pragma unroll
                for (int r = 0; r < C::ROUNDS; ++r)
#pragma unroll
                    for (int part = 0; part < C::DPL / 8; ++part)
                        kw[r][part] = ld_shared_v4(ks + (wig * TPW + r * C::RPR + rg) * ROW_BYTES + part * 128 + 16 * li);
#pragma unroll
                for (int r = 0; r < C::ROUNDS; ++r) {
                    const int row = wig * TPW + r * C::RPR + rg;
                    float acc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
                    for (int part = 0; part < C::DPL / 8; ++part) {
                        const uint32_t ww[4] = {kw[r][part].x, kw[r][part].y, kw[r][part].z, kw[r][part].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float k0 = bf16lo(ww[e]), k1 = bf16hi(ww[e]);
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                acc[h] = fmaf(qf[h][part * 8 + 2 * e], k0, acc[h]);
                                acc[h] = fmaf(qf[h][part * 8 + 2 * e + 1], k1, acc[h]);
                            }
                        }
                    }
                    float s = reduce_scatter<G, C::LPT>(acc, li);
                    if (row >= nvalid) s = -INFINITY;
                    if (li % (C::LPT / G) == 0) sbuf[(r * C::RPR + rg) * G + li / (C::LPT / G)] = s;
                }
                __syncwarp();
                // ---- online softmax over this warp's TPW rows (lanes 16..31 mirror 0..15)
                float alpha[G];
                {
                    const int rr = lane & (TPW - 1);
                    float sc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) sc[h] = sbuf[rr * G + h];
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float mx = sc[h];
#pragma unroll
                        for (int off = TPW / 2; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
                        const float m_new = fmaxf(m_run[h], mx);
                        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                        const float p = fast_exp2(sc[h] - m_use);
                        alpha[h] = fast_exp2(m_run[h] - m_use);
                        float ps = p;
#pragma unroll
                        for (int off = TPW / 2; off >= 1; off >>= 1) ps += __shfl_xor_sync(FULL, ps, off);
                        l_run[h] = l_run[h] * alpha[h] + ps;
                        m_run[h] = m_new;
                        sc[h] = p;
                    }
                    __syncwarp();
                    if (lane < TPW) {
#pragma unroll
                        for (int h = 0; h < G; ++h) sbuf[rr * G + h] = sc[h];
                    }
                    __syncwarp();
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    o[h][0] *= alpha[h];
                    o[h][1] *= alpha[h];
                    o[h][2] *= alpha[h];
                    o[h][3] *= alpha[h];
                }
                // ---- P.V over this warp's valid rows
                const int nv = max(0, min(TPW, nvalid - wig * TPW));
#pragma unroll 4
                for (int rr = 0; rr < nv; ++rr) {
                    const int row = wig * TPW + rr;
                    const uint2 w = ld_shared_v2(vsa + row * ROW_BYTES + 8 * lane);
                    const float v0 = bf16lo(w.x), v1 = bf16hi(w.x), v2 = bf16lo(w.y), v3 = bf16hi(w.y);
                    float p[G];
                    if constexpr (G == 4) {
                        const uint4 pp = ld_shared_v4(sbuf_a + rr * G * 4);
                        p[0] = __uint_as_float(pp.x);
                        p[1] = __uint_as_float(pp.y);
                        p[2] = __uint_as_float(pp.z);
                        p[3] = __uint_as_float(pp.w);
                    } else {
#pragma unroll
                        for (int h = 0; h < G; ++h) p[h] = sbuf[rr * G + h];
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        o[h][0] = fmaf(p[h], v0, o[h][0]);
                        o[h][1] = fmaf(p[h], v1, o[h][1]);
                        o[h][2] = fmaf(p[h], v2, o[h][2]);
                        o[h][3] = fmaf(p[h], v3, o[h][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
        // ---- publish this warp's (m, l, o) for the merge warp
        (void)wait_or_abort(&sfree[k & 1], ((k >> 1) & 1) ^ 1, flags, a, 220 + warp);
        float *so = slot_base + (k & 1) * C::SLOT_FLOATS;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            *reinterpret_cast<float4 *>(so + (warp * G + h) * D + 4 * lane) =
                make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
            if (lane == 0) {
                so[C::NCW * G * D + (warp * G + h) * 2] = m_run[h];
                so[C::NCW * G * D + (warp * G + h) * 2 + 1] = l_run[h];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&done[k & 1]);
    }
}

// Log-sum-exp merge of the split partials of one (sequence, q head):
// M = max_c m_c, L = sum_c l_c 2^(m_c - M), out = sum_c o_c 2^(m_c - M) / L.
// Launched after decode_kernel on the same stream (programmatic dependent
// launch: it may start early and waits for the decode grid's results).
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeArgs a) {
    __shared__ float wts[kMaxSplits];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bh = blockIdx.x;
    const int b = bh / a.Hq;
    const int ctx = clamp_ctx(a, b, false);
    const int nsplit = (ctx + a.chunk_tokens - 1) / a.chunk_tokens;
    if (nsplit <= 1) return;  // written directly by decode_kernel
    const float2 *ml = a.ws_ml + (int64_t)bh * a.max_splits;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float M = -INFINITY;
        for (int c = lane; c < nsplit; c += 32) M = fmaxf(M, ml[c].x);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
        float L = 0.f;
        for (int c = lane; c < nsplit; c += 32) {
            const float2 v = ml[c];
            const float f = fast_exp2(v.x - M);
            wts[c] = f;
            L = fmaf(v.y, f, L);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(FULL, L, off);
        const float invL = 1.f / L;
        __syncwarp();
        for (int c = lane; c < nsplit; c += 32) wts[c] *= invL;
    }
    __syncthreads();
    const float *po = a.ws_o + (int64_t)bh * a.max_splits * D + threadIdx.x;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int c = 0;
    for (; c + 4 <= nsplit; c += 4) {
        acc0 = fmaf(po[(int64_t)(c + 0) * D], wts[c + 0], acc0);
        acc1 = fmaf(po[(int64_t)(c + 1) * D], wts[c + 1], acc1);
        acc2 = fmaf(po[(int64_t)(c + 2) * D], wts[c + 2], acc2);
        acc3 = fmaf(po[(int64_t)(c + 3) * D], wts[c + 3], acc3);
    }
    for (; c < nsplit; ++c) acc0 = fmaf(po[(int64_t)c * D], wts[c], acc0);
    a.out[(int64_t)bh * D + threadIdx.x] = __float2bfloat16_rn((acc0 + acc1) + (acc2 + acc3));
}

int g_attr_done[64][4] = {};

template <int G>
pa_status launch(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                 cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
    if (dev >= 0 && dev < 64 && !g_attr_done[dev][gi]) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Cfg<G>::smem_bytes(kMaxBatch));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_kernel)");
        g_attr_done[dev][gi] = 1;
    }
    decode_kernel<G><<<grid, Cfg<G>::NTHREADS, Cfg<G>::smem_bytes(a.batch), st>>>(tk, tv, a);
    pa_status r = check_launch("decode_kernel");
    if (r != PA_OK || a.max_splits <= 1) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.batch * a.Hq));
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
    if (e != cudaSuccess) return cuda_fail(e, "decode_merge_kernel");
    return check_launch("decode_merge_kernel");
}

int chunk_tokens_for(int max_ctx) {
    int chunk = 4 * TILE;  // 256 positions per work item
    if (max_ctx > 0 && (max_ctx + chunk - 1) / chunk > kMaxSplits) {
        chunk = (max_ctx + kMaxSplits - 1) / kMaxSplits;
        chunk = (chunk + TILE - 1) / TILE * TILE;
    }
    return chunk;
}

struct WsLayout {
    size_t ml_off, o_off, total;
    int max_splits, chunk;
};

WsLayout ws_layout(int batch, int Hq, int max_ctx) {
    WsLayout L;
    L.chunk = chunk_tokens_for(max_ctx);
    L.max_splits = max_ctx > 0 ? (max_ctx + L.chunk - 1) / L.chunk : 1;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    L.ml_off = 0;
    L.o_off = up((size_t)batch * Hq * L.max_splits * 8);
    L.total = L.o_off + (size_t)batch * Hq * L.max_splits * D * 4;
    return L;
}

int effective_max_ctx(int32_t max_context_len, int32_t max_blocks, int32_t block_size) {
    const int64_t cap = (int64_t)max_blocks * block_size;
    if (max_context_len <= 0 || max_context_len > cap) return (int)cap;
    return max_context_len;
}

}  // namespace
}  // namespace pa

extern "C" {

size_t pa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_context_len,
                                int32_t max_blocks_per_seq, int32_t block_size) {
    using namespace pa;
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim != D || block_size <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    (void)num_kv_heads;
    return ws_layout(batch, num_q_heads, effective_max_ctx(max_context_len, max_blocks_per_seq, block_size))
        .total;
}

pa_status pa_decode(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                    float softmax_scale, int32_t max_context_len, void *workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
    using namespace pa;
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch < 0");
    if (batch == 0) return PA_OK;
    if (batch > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "batch %d > %d", batch, kMaxBatch);
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PA_ERR_UNSUPPORTED, "GQA group %d (supported: 1, 2, 4, 8)", G);
    if (head_dim != D) return fail(PA_ERR_UNSUPPORTED, "head_dim %d (only 128)", head_dim);
    if (block_size <= 0 || block_size % 16)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (must be a positive multiple of 16)", block_size);
    if (max_blocks_per_seq <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq and num_blocks must be positive");
    if ((int64_t)num_blocks * block_size > 0x7fffffffLL ||
        (int64_t)max_blocks_per_seq * block_size > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "pool or table too large for 32-bit slot indices");
    if (q_row_stride < (int64_t)num_q_heads * D || q_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "q_row_stride must be >= num_q_heads*head_dim and a multiple of 8");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "out/q/cache pointers must be 16-byte aligned");
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
        return fail(PA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
    const int max_ctx = effective_max_ctx(max_context_len, max_blocks_per_seq, block_size);
    const WsLayout W = ws_layout(batch, num_q_heads, max_ctx);
    if (W.max_splits > 1 && (!workspace || workspace_bytes < W.total))
        return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", W.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (workspace && !aligned16(workspace)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    int box = 64;
    while (block_size % box) box >>= 1;  // gcd(block_size, 64) in {16, 32, 64}
    CUtensorMap tk, tv;
    pa_status st = encode_kv_tensor_map(&tk, k_cache, (int64_t)num_blocks * block_size, num_kv_heads, D, box);
    if (st != PA_OK) return st;
    st = encode_kv_tensor_map(&tv, v_cache, (int64_t)num_blocks * block_size, num_kv_heads, D, box);
    if (st != PA_OK) return st;

    DecodeArgs A;
    A.out = static_cast<__nv_bfloat16 *>(out);
    A.q = static_cast<const __nv_bfloat16 *>(q);
    A.q_row_stride = q_row_stride;
    A.block_tables = block_tables;
    A.ctx_lens = context_lens;
    A.max_blocks = max_blocks_per_seq;
    A.batch = batch;
    A.Hq = num_q_heads;
    A.Hkv = num_kv_heads;
    A.block_size = block_size;
    A.box_rows = box;
    A.num_blocks = num_blocks;
    A.scale_log2 = softmax_scale * 1.4426950408889634f;
    A.chunk_tokens = W.chunk;
    A.max_splits = W.max_splits;
    A.ctx_limit = (int)std::min<int64_t>((int64_t)max_blocks_per_seq * block_size,
                                         (int64_t)W.max_splits * W.chunk);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    A.ws_ml = ws ? reinterpret_cast<float2 *>(ws + W.ml_off) : nullptr;
    A.ws_o = ws ? reinterpret_cast<float *>(ws + W.o_off) : nullptr;
    A.err = device_error_ptr();
    A.checked = checked_mode() ? 1 : 0;

    const int sms = sm_count();
    if (sms <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (G) {
        case 1: return launch<1>(A, tk, tv, sms, s);
        case 2: return launch<2>(A, tk, tv, sms, s);
        case 4: return launch<4>(A, tk, tv, sms, s);
        default: return launch<8>(A, tk, tv, sms, s);
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode_static: decode attention for callers that cannot allocate device
// memory.  The split partials live in a fixed scratch array that is part of
// this library's device image instead of a caller-provided workspace.
// ---------------------------------------------------------------------------

// 32 MiB of split-partial scratch.  It is loaded with the module, so every GPU
// that loads this library holds it until the process exits.
static constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char pa_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void *g_static_scratch_addr[64] = {};  // device address of the array, per device
}  // namespace

extern "C" pa_status pa_decode_static(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float softmax_scale,
                                      int32_t max_context_len, pa_stream_t stream) {
    using namespace pa;
    const size_t need = pa_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                                 max_blocks_per_seq, block_size);
    if (need == 0)  // batch == 0 or arguments pa_decode rejects: let it report
        return pa_decode(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         softmax_scale, max_context_len, nullptr, 0, stream);
    if (need > kStaticScratchBytes)
        return fail(PA_ERR_WORKSPACE,
                    "pa_decode_static: this shape needs %zu bytes of split scratch but the built-in scratch "
                    "holds %zu; lower max_context_len/batch or call pa_decode with a workspace",
                    need, kStaticScratchBytes);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    void *scratch = nullptr;
    {
        // Set-up, once per device, with that device current: the host-side name
        // of the array is not a device address, so ask the runtime for it.
        std::lock_guard<std::mutex> lk(g_static_mu);
        if (g_static_scratch_addr[dev] == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, pa_static_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(pa_static_scratch)");
            g_static_scratch_addr[dev] = p;
        }
        scratch = g_static_scratch_addr[dev];
    }
    return pa_decode(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, softmax_scale,
                     max_context_len, scratch, kStaticScratchBytes, stream);
}
