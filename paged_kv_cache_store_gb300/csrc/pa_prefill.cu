// pa_prefill.cu -- varlen causal prefill attention on 5th-generation tensor cores.
//
// What it computes [NV12 §12.6 flash_attn_varlen_func; NV05 prepare_prefill]:
// for sequence s with Lq new rows and Lk keys (c = Lk - Lq of them cached),
// query i at position c + i attends to keys 0..c+i (bottom-right causal;
// all Lk keys when causal == 0), keys read through the block table
// (prefix cache) or from contiguous rows.
//
// How (GB300 design): persistent CTAs (one per SM) walk work tiles of
// (128-row query tile, sequence, q head), highest query tiles first; all
// roles follow one global KV-tile counter, so the next tile's Q/K/V copies
// overlap the current tile's softmax and epilogue.
//  * warps 0 and 10 (one thread each) issue TMA copies: warp 0 the Q tile
//    and the K tiles of 128 keys, warp 10 the V tiles, into separate rings
//    (Q: 2, K: 3, V: 2 stages) so neither stream waits behind the other.  Boxes are {64 dims, 1 head,
//    R rows} with 128-byte swizzle (two boxes per 128-dim row); paged boxes
//    never straddle a block (R = gcd(block_size, 128)).
//  * warp 1 (one thread) owns the tensor cores: S = Q.K^T (M=N=128, K=128,
//    eight tcgen05.mma K=16 steps) into one of two TMEM buffers, then
//    O += P.V with V as an MN-major operand, O accumulating in TMEM.
//    tcgen05.commit arrives on mbarriers to free K/V stages, publish S and
//    release the P buffer.
//  * warps 2..9: two warps per TMEM lane quarter, one thread per query row
//    and 64 of the 128 key columns each, read S with tcgen05.ld, apply scale
//    and mask, share the row max through shared memory (an mbarrier per
//    warp pair, double-buffered slots), keep running statistics in base 2, and write
//    their half of P as bf16 pairs into TMEM, where the P.V MMA takes it as
//    its A operand (only V is read from shared memory).  O in TMEM is rescaled only when a row's max grows by
//    more than 2^8 (otherwise the stale max keeps P <= 256, exact enough in
//    bf16 and fp32); the final 1/l is applied in the epilogue.
//  * Every mbarrier wait is bounded; a timeout records PA_DEV_TIMEOUT and
//    the roles skip to the CTA-wide teardown.
// TMEM: S0 = columns 0..127, S1 = 128..255, O = 256..383, P0/P1 = 384..511.
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
constexpr int NTHREADS = 352;
constexpr int W_TMA = 0, W_MMA = 1, W_SOFT = 2, W_VTMA = 10;  // softmax warps 2..9
// Softmax warp w reads TMEM lane quarter w % 4 (hardware rule) and key/dim
// columns [64*h, 64*h + 64) with h = (w - 2) / 4: two warps share each row.

constexpr int QST = 2;  // Q tiles (one per work tile in flight)
constexpr int KST = 3;  // K ring stages (K is needed first: deepest prefetch)
constexpr int VST = 2;  // V ring stages (V is needed after the softmax)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QST * TILE_BYTES;
constexpr int OFF_V = OFF_K + KST * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + VST * TILE_BYTES;
enum { B_Q = 0, B_QEMPTY = B_Q + QST, B_KFULL = B_QEMPTY + QST, B_KEMPTY = B_KFULL + KST, B_VFULL = B_KEMPTY + KST,
       B_SFULL = B_VFULL + VST, B_PFULL = B_SFULL + 2, B_PFREE = B_PFULL + 2, B_OFREE = B_PFREE + 2,
       B_XCH = B_OFREE + 1 /* [4 quarters][2 slots] */, NBAR = B_XCH + 8 };
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_FLAGS = OFF_TMEM + 8;
constexpr int OFF_XCH = OFF_FLAGS + 16;  // row-statistics exchange [4 quarters][2 slots][2 halves][32] f32
constexpr int OFF_BID = OFF_XCH + 4 * 2 * 2 * 32 * 4;  // block ids of the current work tile, per producer
constexpr int NBID = 32;
constexpr int SMEM_USED = OFF_BID + 2 * NBID * 4;
// Slack for aligning the dynamic shared-memory base to the 1 KiB the swizzled
// tiles need (the base is normally aligned already; the kernel checks).
constexpr int SMEM_SLACK = 256;
constexpr size_t SMEM_BYTES = SMEM_USED + SMEM_SLACK;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(VST == 2, "V stages are released through the two P buffers' barriers");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 256;  // O accumulator, 128 fp32 columns
constexpr uint32_t COL_P = 384;  // two P buffers, 64 columns each (128 keys as bf16 pairs)
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);  // Q, K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);   // P from TMEM, V MN-major
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

// Tile coordinates of work tile t: the highest query tiles (the most keys)
// come first, then sequence, then q head (the heads of one kv group are
// neighbours, so their K/V tiles are reused from L2).
struct Tile {
    int s, h, m0, q0, Lq, k0, Lk, n_kv, key_end, valid;
};

__device__ __forceinline__ Tile tile_of(const PrefillArgs &a, int t) {
    Tile T;
    const int per = a.num_seqs * a.Hq;
    const int mt = a.mtiles - 1 - t / per;
    const int rem = t % per;
    T.s = rem / a.Hq;
    T.h = rem % a.Hq;
    T.m0 = mt * BM;
    T.q0 = __ldg(a.cu_q + T.s);
    T.Lq = __ldg(a.cu_q + T.s + 1) - T.q0;
    T.k0 = __ldg(a.cu_k + T.s);
    T.Lk = __ldg(a.cu_k + T.s + 1) - T.k0;
    const bool bad = T.Lq < 0 || T.Lk < T.Lq || (a.paged && T.Lk > a.max_blocks * a.block_size);
    T.valid = !bad && T.m0 < T.Lq;
    if (bad && mt == 0 && T.h == 0 && threadIdx.x == 0) record_error(a.err, PA_DEV_BAD_SEQLENS, T.s);
    T.key_end = 0;
    T.n_kv = 0;
    if (T.valid) {
        const int c = T.Lk - T.Lq;
        const int last_row = min(T.m0 + BM, T.Lq) - 1;
        T.key_end = a.causal ? min(T.Lk, c + last_row + 1) : T.Lk;
        T.n_kv = (T.key_end + BN - 1) / BN;
    }
    return T;
}

// First work tile >= t (stepping by gridDim.x) whose query rows exist.  The
// warp tests 32 candidates per round of loads and takes the first by ballot,
// so skipping the many empty high query tiles costs one load latency per 32.
// Every lane must call it; every role gets the same answer.
__device__ __forceinline__ int next_valid_tile(const PrefillArgs &a, int t, int ntiles, int lane) {
    const int per = a.num_seqs * a.Hq;
    for (int base = t; base < ntiles; base += 32 * (int)gridDim.x) {
        const int tt = base + lane * (int)gridDim.x;
        bool v = false;
        if (tt < ntiles) {
            const int mt = a.mtiles - 1 - tt / per;
            const int s = (tt % per) / a.Hq;
            v = mt * BM < __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
        }
        const unsigned m = __ballot_sync(FULL, v);
        if (m) return base + (__ffs(m) - 1) * (int)gridDim.x;
    }
    return ntiles;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    if (pad > (uint32_t)SMEM_SLACK) {  // cannot align the tiles inside the allocation
        if (threadIdx.x == 0) record_error(a.err, PA_DEV_SMEM_ALIGN, (long long)pad);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + OFF_FLAGS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = a.mtiles * a.num_seqs * a.Hq;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if ((i >= B_PFULL && i < B_PFULL + 2) || i == B_OFREE) cnt = 8;
            if (i >= B_XCH) cnt = 64;
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

    // Every role walks the same tiles t = blockIdx.x, +gridDim.x, ... and the
    // same global KV-tile counter g, so ring stages and barrier phases agree.
    if (warp == W_TMA || warp == W_VTMA) {
        // ------------------------------------------------------------ TMA producers
        // Two independent streams: warp W_TMA loads Q and K, warp W_VTMA loads V,
        // each as far ahead as its own ring allows (V is needed after the
        // softmax, K before it, so neither waits behind the other).
        const bool is_k = warp == W_TMA;
        const CUtensorMap *tm = is_k ? &tmk : &tmv;
        const int NS = is_k ? KST : VST;
        const int off = is_k ? OFF_K : OFF_V;
        uint64_t *full = &bar[is_k ? B_KFULL : B_VFULL];
        // A V stage is free once the P.V that read it is complete: with as many V
        // stages as P buffers, the P_FREE barrier of that P.V serves, and the
        // producer waits on its phases in order.  The 3-stage K ring has its
        // own release barriers (one phase per stage use).
        int *bid = reinterpret_cast<int *>(smem + OFF_BID) + (is_k ? 0 : NBID);
        if (lane == 0) {
            if (is_k) prefetch_tensormap(&tmq);
            prefetch_tensormap(tm);
        }
        const int R = a.box_rows;
        uint32_t g = 0, tk = 0;  // KV tiles and Q tiles issued by this warp
        bool ok = true;
        for (int t = next_valid_tile(a, blockIdx.x, ntiles, lane); ok && t < ntiles;
             t = next_valid_tile(a, t + gridDim.x, ntiles, lane)) {
            const Tile T = tile_of(a, t);
            const int32_t *bt = a.bt + (int64_t)T.s * a.max_blocks;
            if (T.valid && a.paged) {
                // The warp fetches the tile's first NBID block ids at once.
                const int nblk = min((T.key_end - 1) / a.block_size + 1, NBID);
                for (int b = lane; b < nblk; b += 32) bid[b] = __ldg(bt + b);
            }
            __syncwarp();
            if (lane == 0 && T.valid) {
                const int kvh = T.h / a.group;
                if (is_k) {
                    const uint32_t qs = tk % QST;
                    ok = wait_or_abort(&bar[B_QEMPTY + qs], ((tk / QST) & 1u) ^ 1u, flags, a.err, 400);
                    if (ok) {
                        mbar_arrive_expect_tx(&bar[B_Q + qs], TILE_BYTES);
                        uint8_t *qd = smem + OFF_Q + qs * TILE_BYTES;
                        tma_load_3d_plain(qd, &tmq, 0, T.h, T.q0 + T.m0, &bar[B_Q + qs]);
                        tma_load_3d_plain(qd + HALF_BYTES, &tmq, 64, T.h, T.q0 + T.m0, &bar[B_Q + qs]);
                        ++tk;
                    }
                }
                for (int j = 0; ok && j < T.n_kv; ++j, ++g) {
                    const int st = g % NS;
                    const int kb = j * BN;
                    const int nsub = (min(BN, T.key_end - kb) + R - 1) / R;
                    if (is_k) {
                        if (!(ok = wait_or_abort(&bar[B_KEMPTY + st], ((g / KST) & 1u) ^ 1u, flags, a.err, 401))) break;
                    } else if (g >= (uint32_t)VST) {  // the P.V of tile g - VST read this stage
                        const uint32_t u = g - VST;
                        if (!(ok = wait_or_abort(&bar[B_PFREE + (u & 1)], (u >> 1) & 1u, flags, a.err, 402))) break;
                    }
                    mbar_arrive_expect_tx(&full[st], (uint32_t)nsub * R * D * 2);
                    uint8_t *dst = smem + off + st * TILE_BYTES;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int key = kb + sub * R;
                        int row;
                        if (a.paged) {
                            const int lb = key / a.block_size;
                            const int blk = lb < NBID ? bid[lb] : __ldg(bt + lb);
                            if (a.checked && is_k && (blk < 0 || blk >= a.num_blocks))
                                record_error(a.err, PA_DEV_BAD_BLOCK, (long long)T.s * a.max_blocks + lb);
                            // An invalid block id reads as zeros: TMA fills out-of-range boxes.
                            row = (blk < 0 || blk >= a.num_blocks) ? -2 * R : blk * a.block_size + key % a.block_size;
                        } else {
                            row = T.k0 + key;
                        }
                        tma_load_3d_plain(dst + sub * R * 128, tm, 0, kvh, row, &full[st]);
                        tma_load_3d_plain(dst + HALF_BYTES + sub * R * 128, tm, 64, kvh, row, &full[st]);
                    }
                }
            }
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0 && !ok) {
            // Let issued copies land before the CTA's shared memory is released.
            for (uint32_t x = (tk >= QST ? tk - QST : 0); x < tk; ++x)
                (void)mbar_wait(&bar[B_Q + x % QST], (x / QST) & 1u);
            for (uint32_t x = (g >= (uint32_t)NS ? g - NS : 0); x < g; ++x) (void)mbar_wait(&full[x % NS], (x / NS) & 1u);
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------ MMA issuer
        // The warp walks the tiles together; lane 0 waits and issues.
        {
            uint32_t g = 0, tk = 0;
            int64_t last_pv = -1;  // global index of the last P.V issued
            bool ok = true;
            // O += P_gg V_gg; `first` overwrites O (first KV tile of a work tile).
            auto issue_pv = [&](uint32_t gg, bool first) -> bool {
                const int pb = gg & 1, vs = gg % VST;
                if (first && tk > 1 &&
                    !wait_or_abort(&bar[B_OFREE], (tk - 2) & 1u, flags, a.err, 410))  // previous epilogue read O
                    return false;
                // (The softmax publishes P only after V of the same tile has landed.)
                if (!wait_or_abort(&bar[B_PFULL + pb], (gg >> 1) & 1u, flags, a.err, 411)) return false;
                tc_fence_after();
                // One descriptor per operand; each K=16 step only moves the start
                // address (low 14 bits, in 16-byte units) by a constant.
                const uint64_t vdesc = smem_desc_sw128(smem_addr(smem + OFF_V + vs * TILE_BYTES), HALF_BYTES, SBO);
                const uint32_t pcol = tmem + COL_P + pb * 64;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)  // 16 keys per step = 8 TMEM columns of P
                    mma_bf16_ts(tmem + COL_O, pcol + k * 8, vdesc + (uint64_t)((k * 16 * 128) >> 4), IDESC_PV,
                                (!first || k > 0) ? 1u : 0u);
                mma_commit(&bar[B_PFREE + pb]);
                last_pv = gg;
                return true;
            };
            // All MMAs of one work tile (lane 0 only); false on a timeout.
            auto mma_tile = [&](const Tile &T) -> bool {
                const uint32_t qs = tk % QST;
                if (!wait_or_abort(&bar[B_Q + qs], (tk / QST) & 1u, flags, a.err, 413)) return false;
                const uint64_t qdesc = smem_desc_sw128(smem_addr(smem + OFF_Q + qs * TILE_BYTES), 16, SBO);
                ++tk;
                for (int j = 0; j < T.n_kv; ++j, ++g) {
                    const int st = g & 1, ks = g % KST;
                    // (S buffer st is free: P of tile g-2 was published, so its S was read.)
                    if (!wait_or_abort(&bar[B_KFULL + ks], (g / KST) & 1u, flags, a.err, 414)) return false;
                    tc_fence_after();
                    const uint64_t kdesc = smem_desc_sw128(smem_addr(smem + OFF_K + ks * TILE_BYTES), 16, SBO);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t off = (uint64_t)(((k >> 2) * HALF_BYTES + (k & 3) * 32) >> 4);
                        mma_bf16_ss(tmem + st * BN, qdesc + off, kdesc + off, IDESC_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit(&bar[B_KEMPTY + ks]);
                    mma_commit(&bar[B_SFULL + st]);
                    if (j == T.n_kv - 1) mma_commit(&bar[B_QEMPTY + qs]);  // this Q tile may be reloaded
                    if (j >= 1 && !issue_pv(g - 1, j == 1)) return false;
                }
                return issue_pv(g - 1, T.n_kv == 1);
            };
            for (int t = next_valid_tile(a, blockIdx.x, ntiles, lane); ok && t < ntiles;
                 t = next_valid_tile(a, t + gridDim.x, ntiles, lane)) {
                if (lane == 0) {
                    const Tile T = tile_of(a, t);
                    if (T.valid) ok = mma_tile(T);
                }
                ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
            }
            if (lane == 0 && !ok && last_pv >= 0) {
                // Let the issued MMAs finish before TMEM is released.
                (void)mbar_wait(&bar[B_PFREE + (last_pv & 1)], (uint32_t)(last_pv >> 1) & 1u);
            }
        }
    } else if (warp >= W_SOFT) {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3, half = (warp - W_SOFT) >> 2;
        const int row = quarter * 32 + lane;  // tile row == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t col0 = half * 64;      // this warp's 64 key columns of S and dim columns of O
        float *xch = reinterpret_cast<float *>(smem + OFF_XCH) + quarter * 128;  // [2 slots][2 halves][32]
        const float sl = a.scale_log2;
        uint32_t g = 0, xc = 0;  // KV tiles consumed; exchanges done with the partner warp
        bool ok = true;
        // Exchange one value per row with the partner warp (same rows, other
        // half): slots alternate, so one bounded mbarrier wait per exchange.
        auto exchange = [&](float v, float &partner) -> bool {
            const uint32_t slot = xc & 1u;
            float *x2 = xch + slot * 64;
            x2[half * 32 + lane] = v;
            mbar_arrive(&bar[B_XCH + quarter * 2 + slot]);
            const bool done = __all_sync(FULL, wait_or_abort(&bar[B_XCH + quarter * 2 + slot], (xc >> 1) & 1u, flags,
                                                              a.err, 425));
            partner = x2[(half ^ 1) * 32 + lane];
            ++xc;
            return done;
        };
        for (int t = next_valid_tile(a, blockIdx.x, ntiles, lane); ok && t < ntiles;
             t = next_valid_tile(a, t + gridDim.x, ntiles, lane)) {
            const Tile T = tile_of(a, t);
            if (!T.valid) continue;
            const int i = T.m0 + row;          // query index in the sequence (>= Lq: padding row)
            const int pos = (T.Lk - T.Lq) + i;
            const int key_last = (a.causal ? min(pos, T.Lk - 1) : T.Lk - 1);  // last key this row sees
            float m_run = -INFINITY;           // running max of raw scores (shared with the partner warp)
            float l_run = 0.f;                 // this half's running sum
            for (int j = 0; j < T.n_kv; ++j, ++g) {
                const int sb = g & 1;
                const uint32_t ph = (g >> 1) & 1u;
                // Waits in this role are warp-uniform: tcgen05.ld/st are warp-collective.
                if (!(ok = __all_sync(FULL, wait_or_abort(&bar[B_SFULL + sb], ph, flags, a.err, 420)))) break;
                tc_fence_after();
                // Each warp reads its 64 columns of the S row; the row max is
                // shared with the partner warp (the other 64 columns).
                uint32_t r[2][32];
                tmem_ld32(t_lane + sb * BN + col0, r[0]);
                tmem_ld32(t_lane + sb * BN + col0 + 32, r[1]);
                tmem_ld_wait();

                const int kb = j * BN + col0;
                const int lim = key_last - kb;  // this warp's keys kb+k with k <= lim are visible
                float x[64];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = __uint_as_float(r[0][e]);
                    x[32 + e] = __uint_as_float(r[1][e]);
                }
                if (__any_sync(FULL, lim < 63)) {
#pragma unroll
                    for (int k = 0; k < 64; ++k)
                        if (k > lim) x[k] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = x[e];
#pragma unroll
                for (int k = 8; k < 64; k += 8)
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], x[k + e]);
                float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                float tpart;
                if (!(ok = exchange(tmax, tpart))) break;
                tmax = fmaxf(tmax, tpart);
                // Lazy rescaling: keep the old max unless this tile's max exceeds it
                // by more than 8 in log2 units (P then stays <= 2^8).
                const bool grow = (tmax - m_run) * sl > 8.f;
                const float m_new = grow ? tmax : m_run;
                const float alpha = grow ? fast_exp2((m_run - m_new) * sl) : 1.f;
                if (__any_sync(FULL, grow) && j > 0) {
                    // O holds the previous tiles' P.V: wait for the last one, then
                    // rescale this warp's 64 columns of O.
                    const uint32_t pg = g - 1;
                    ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + (pg & 1)], (pg >> 1) & 1u, flags, a.err, 421));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + COL_O + col0 + cc * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(t_lane + COL_O + col0 + cc * 32, o);
                    }
                    tmem_st_wait();
                }
                l_run *= alpha;
                m_run = m_new;
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * sl;
                if (g >= 2 && !(ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + sb], ph ^ 1u, flags, a.err, 422))))
                    break;
                // This warp's 64 keys become 32 TMEM columns of bf16 pairs (the A
                // operand of the P.V MMA), in this buffer's half `half`.
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
#pragma unroll
                for (int k2 = 0; k2 < 32; ++k2) {
                    const float p0 = fast_exp2(fmaf(x[2 * k2], sl, neg_m));
                    const float p1 = fast_exp2(fmaf(x[2 * k2 + 1], sl, neg_m));
                    rs[(2 * k2) & 3] += p0;
                    rs[(2 * k2 + 1) & 3] += p1;
                    pk[k2] = pack_bf16(p0, p1);
                }
                tmem_st32(t_lane + COL_P + sb * 64 + half * 32, pk);
                tmem_st_wait();
                l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
                const int kend = T.key_end - j * BN;
                const int vs = g % VST;
                // V of this tile must have landed before P is published (the MMA
                // thread then issues P.V without its own wait).
                if (!(ok = __all_sync(FULL, wait_or_abort(&bar[B_VFULL + vs], (g / VST) & 1u, flags, a.err, 423))))
                    break;
                if (j == T.n_kv - 1 && kend < BN) {
                    // Rows past the last needed key hold stale or unloaded data:
                    // zero them (this warp: one 64-dim half) so 0 * garbage cannot reach O.
                    if (row >= kend) {
                        const uint32_t vrow = smem_addr(smem + OFF_V + vs * TILE_BYTES) + half * HALF_BYTES + row * 128;
#pragma unroll
                        for (int q16 = 0; q16 < 8; ++q16) st_shared_v4(vrow + q16 * 16, 0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_PFULL + sb]);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16; this warp writes its 64 dims of each row
            const uint32_t pg = g - 1;
            if (!(ok = __all_sync(FULL, wait_or_abort(&bar[B_PFREE + (pg & 1)], (pg >> 1) & 1u, flags, a.err, 424))))
                break;
            tc_fence_after();
            uint32_t o[2][32];
            tmem_ld32(t_lane + COL_O + col0, o[0]);
            tmem_ld32(t_lane + COL_O + col0 + 32, o[1]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OFREE]);  // O may be overwritten by the next tile
            float lpart;
            if (!(ok = exchange(l_run, lpart))) break;
            const float l_tot = l_run + lpart;
            if (i < T.Lq) {
                const float inv = 1.f / l_tot;
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((int64_t)(T.q0 + i) * a.Hq + T.h) * D + col0);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t *v = &o[cc][8 * e];
                        dst[cc * 4 + e] = make_uint4(
                            pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                            pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                            pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                            pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
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

    const int64_t ntiles = (int64_t)A.mtiles * num_seqs * num_q_heads;
    if (ntiles > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "too many tiles");
    const int sms = sm_count();
    if (sms <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    const int64_t grid = std::min<int64_t>(ntiles, sms);  // persistent: one CTA per SM
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
