// pa_prefill.cu -- varlen causal prefill attention on 5th-generation tensor cores.
//
// What it computes [NV12 §12.6 flash_attn_varlen_func; NV05 prepare_prefill]:
// for sequence s with Lq new rows and Lk keys (c = Lk - Lq of them cached),
// query i at position c + i attends to keys 0..c+i (bottom-right causal;
// all Lk keys when causal == 0), keys read through the block table
// (prefix cache) or from contiguous rows.
//
// How (GB300 design): persistent CTAs (one per SM) walk work units of
// (128-row query tile, sequence, q head), highest query tiles first.
//  * warp 0 issues the TMA copies of Q and K, warp 2 those of V (rings: Q 2,
//    K 3 and V 2 stages; K/V tiles of 128 keys).  Tiles land 128-byte
//    swizzled as [half][row][64] through 4-D tensor maps that view a
//    [rows][heads][128] tensor as [head][half][row][64]: one copy per tile
//    when blocks hold 128 rows or more.
//  * Two single-thread MMA issuers feed the tensor cores, so one's barrier
//    waits overlap the other's MMAs: warp 1 issues S = Q.K^T (M=N=128, K=128,
//    8 steps; both operands from shared memory) into one of three S buffers,
//    warp 3 issues O += P.V with P read from TMEM (bf16 pairs written over
//    its S buffer) and V as an MN-major operand.  Scores run up to three
//    tiles ahead of P.V; a Q.K waits until the P.V that read its buffer three
//    tiles earlier has completed.
//    tcgen05.commit arrives on mbarriers to free K/V stages and S buffers
//    (which also reports O) and to publish S.
//  * warps 4..7: one thread per query row (its TMEM lane) holds all 128
//    scores of a tile, so row statistics need no exchange.  Online softmax
//    in base 2; P goes back to TMEM as bf16 pairs.  O is rescaled only when a
//    row's max grows by more than 2^8 (P then stays <= 256, exact enough in
//    bf16 and fp32); only a rescale waits for the previous P.V.  The
//    same warps finish the unit: O / l -> bf16 into the unit's Q buffer (no
//    longer read once its last S is in), then one TMA store for a full tile,
//    or coalesced 256-byte row stores for the last, partial tile of a
//    sequence; the buffer is released for a later Q when that store has read
//    it.
//  * On the last KV tile the P.V thread zeroes the V rows between the last
//    needed key and the next multiple of 16 (stale or unloaded data; P is 0
//    there but 0 * NaN is not) and skips the 16-key steps past it.
//  * Fused store (prefill_kernel<true>, pa_prefill_store_varlen): before any
//    tile is loaded, the CTAs of a cooperative launch copy the uncached
//    suffix rows into their cache slots (bulk copies through the unused ring
//    memory) and meet at a grid barrier; then everything runs as above.
//  * Every mbarrier wait is bounded; a timeout records PA_DEV_TIMEOUT and
//    the roles skip to the CTA-wide teardown.
// TMEM: S/P buffers at columns 0, 128 and 256, O = 384..511.
#include <math.h>

#include <algorithm>
#include <atomic>

#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int D = 128;
constexpr int BM = 128;                     // query rows per tile
constexpr int BN = 128;                     // keys per tile
constexpr int TILE_BYTES = BM * D * 2;      // 32 KiB
constexpr int HALF_BYTES = TILE_BYTES / 2;  // [128 rows][64 dims], 128-byte rows
constexpr int NTHREADS = 256;
constexpr int W_QK = 0, W_MMA = 1, W_V = 2, W_PV = 3, W_SOFT = 4;  // softmax warps 4..7
// Softmax warp w reads TMEM lane quarter w % 4 (hardware rule).

constexpr int QST = 2;  // Q buffers (a finished unit's buffer stages its output tile)
constexpr int KST = 3;  // K ring stages
constexpr int VST = 2;  // V ring stages
constexpr int NSB = 3;  // S/P buffers in TMEM
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QST * TILE_BYTES;
constexpr int OFF_V = OFF_K + KST * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + VST * TILE_BYTES;
enum {
    B_QFULL = 0, B_QEMPTY = B_QFULL + QST, B_KFULL = B_QEMPTY + QST, B_KEMPTY = B_KFULL + KST,
    B_VFULL = B_KEMPTY + KST, B_VEMPTY = B_VFULL + VST, B_SFULL = B_VEMPTY + VST, B_PFULL = B_SFULL + NSB,
    B_PDONE = B_PFULL + NSB, B_OEMPTY = B_PDONE + NSB, B_DRAIN, B_DRAIN2, B_SUFFIX /* [2] fused store's loads */,
    B_SUFFIX2,
    B_NU /* [2] next-unit slots, Q.K thread -> softmax */, NBAR = B_NU + 2
};
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_FLAGS = OFF_TMEM + 8;
constexpr int OFF_BID = OFF_FLAGS + 16;  // block ids of the current unit, per producer warp
constexpr int NBID = 32;
constexpr int OFF_NU = OFF_BID + 2 * NBID * 4;  // two Unit slots (the softmax's next unit)
// The CTA-wide unit schedule: (query tile, sequence) groups sorted by their
// number of KV tiles, longest first (used when there are at most SCHED_MAX).
constexpr int SCHED_MAX = 512;
constexpr int OFF_SCHED = OFF_NU + 2 * 48;  // uint16_t [SCHED_MAX]
constexpr int SMEM_USED = OFF_SCHED + SCHED_MAX * 2;
// Slack for aligning the dynamic shared-memory base to the 1 KiB the swizzled
// tiles need (the base is normally aligned already; the kernel checks).
constexpr int SMEM_SLACK = 256;
constexpr size_t SMEM_BYTES = SMEM_USED + SMEM_SLACK;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 384;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false, false);  // Q and K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);   // P from TMEM, V MN-major
constexpr uint32_t SBO = 1024;  // 8 rows x 128 B between core-matrix groups
constexpr int SOFT_BAR = 1;     // named barrier of the softmax warps
constexpr unsigned FULL = 0xffffffffu;

struct PrefillArgs {
    __nv_bfloat16 *out;
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *bt;
    int32_t max_blocks, num_seqs, Hq, group, mtiles;
    int32_t upg;  // work units per (query tile, sequence) group: Hq, or Hq / 2 for paired heads
    int32_t bn;   // keys per KV tile of the kernel (sizes the sort keys)
    int32_t block_size, box_rows, box_halves, paged, causal, num_blocks, checked, sorted;
    float scale_log2;
    DevError *err;
    // Fused store (pa_prefill_store_varlen): the suffix rows to copy into
    // the caches before any tile is loaded, and the grid barrier that
    // separates the copies from the loads.
    const uint4 *new_k, *new_v;
    int64_t new_k_stride16, new_v_stride16;  // rows, in 16-byte units
    uint4 *k_cache, *v_cache;
    int32_t row16, total_q;
    unsigned *gbar;  // [0] arrivals, [1] generation
};

// Every CTA of the (cooperative, hence co-resident) grid arrives; returns
// when all have, or false after kWaitLimitNs.  The last to arrive resets the
// count and moves the generation on, which releases the others; the counter
// is left as it was found, so the next launch can use it.
__device__ bool grid_barrier(unsigned *bar, unsigned n) {
    volatile unsigned *gen = bar + 1;
    const unsigned g = *gen;
    __threadfence();
    if (atomicAdd(bar, 1u) == n - 1) {
        atomicExch(bar, 0u);
        __threadfence();
        atomicAdd(bar + 1, 1u);
        return true;
    }
    const unsigned long long t0 = globaltimer_ns();
    while (*gen == g) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        __nanosleep(64);
    }
    __threadfence();
    return true;
}

// Copies each suffix token's K and V rows (Hkv*D bf16) to its slot.  Row 2t
// is token t's K, 2t+1 its V; CTA b takes a contiguous share of the rows.
// The rows stream through the CTA's shared memory (free until the first
// tile is loaded) with bulk copies: warp 0's lanes each load a few rows of a
// batch (one cp.async.bulk per row, completing on one mbarrier), then store
// them to their slots (one bulk store per row).  The slot of token t of
// sequence s is that of position (Lk - Lq) + (t - cu_q[s]) through the block
// table, as pa_slot_mapping_prefill gives it; a block id outside the pool is
// recorded as PA_DEV_BAD_SLOT and the row is not written, as
// pa_store_kvcache does.  Returns false if a batch's loads did not land in
// time (recorded; the caller skips the rest of the kernel).
__device__ __forceinline__ int64_t suffix_slot(const PrefillArgs &a, int t, bool is_v) {
    int lo = 0, hi = a.num_seqs - 1;  // the sequence of token t: the last s with cu_q[s] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int q0 = __ldg(a.cu_q + lo), Lq = __ldg(a.cu_q + lo + 1) - q0;
    const int Lk = __ldg(a.cu_k + lo + 1) - __ldg(a.cu_k + lo);
    if (Lq < 0 || Lk < Lq || t >= q0 + Lq || Lk > a.max_blocks * a.block_size) return -1;  // recorded by the units
    const int p = (Lk - Lq) + (t - q0);
    const int blk = __ldg(a.bt + (int64_t)lo * a.max_blocks + p / a.block_size);
    if (blk < 0 || blk >= a.num_blocks) {
        if (!is_v) record_error(a.err, PA_DEV_BAD_SLOT, t);
        return -1;
    }
    return (int64_t)blk * a.block_size + p % a.block_size;
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}

constexpr int SUFFIX_ROWS_PER_LANE = 2;  // rows a lane moves per batch

// Two halves of the staging memory alternate: while one batch's rows are
// stored out, the next batch's loads land in the other half.
__device__ bool store_suffix(const PrefillArgs &a, uint8_t *staging, uint32_t staging_bytes, uint64_t *bar,
                             int lane) {
    const uint32_t row_bytes = (uint32_t)a.row16 * 16;
    const int batch = min((int)(staging_bytes / 2 / row_bytes), 32 * SUFFIX_ROWS_PER_LANE);
    const uint32_t half_bytes = (uint32_t)batch * row_bytes;
    const long long nrows = 2LL * a.total_q;
    const long long per = (nrows + gridDim.x - 1) / gridDim.x;
    const long long r_begin = (long long)blockIdx.x * per, r_end = min(nrows, r_begin + per);
    const int nb = (int)((max(0LL, r_end - r_begin) + batch - 1) / batch);
    const uint32_t st0 = smem_addr(staging);
    int64_t slot[2][SUFFIX_ROWS_PER_LANE];
    // Batch k: rows r_begin + k*batch + lane + 32i into half k & 1, completing on bar[k & 1].
    auto load = [&](int k) {
        const long long b0 = r_begin + (long long)k * batch;
        int valid = 0;
#pragma unroll
        for (int i = 0; i < SUFFIX_ROWS_PER_LANE; ++i) {
            const long long r = b0 + lane + 32 * i;
            slot[k & 1][i] = -1;
            if (lane + 32 * i < batch && r < r_end) slot[k & 1][i] = suffix_slot(a, (int)(r >> 1), (r & 1) != 0);
            valid += slot[k & 1][i] >= 0;
        }
        const int total = __reduce_add_sync(0xffffffffu, valid);
        if (lane == 0) mbar_arrive_expect_tx(&bar[k & 1], (uint32_t)total * row_bytes);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < SUFFIX_ROWS_PER_LANE; ++i) {
            if (slot[k & 1][i] < 0) continue;
            const long long r = b0 + lane + 32 * i;
            const int t = (int)(r >> 1);
            const uint4 *src = (r & 1) ? a.new_v + t * a.new_v_stride16 : a.new_k + t * a.new_k_stride16;
            bulk_load(staging + (k & 1) * half_bytes + (lane + 32 * i) * row_bytes, src, row_bytes, &bar[k & 1]);
        }
    };
    bool ok = true;
    if (nb > 0) load(0);
    for (int k = 0; k < nb; ++k) {
        if (k + 1 < nb) {
            bulk_wait_read0();  // batch k-1's stores have read the half batch k+1 is loaded into
            __syncwarp();
            load(k + 1);
        }
        // Every lane waits: the rows it stores were loaded by other lanes' copies too.
        if (!mbar_wait(&bar[k & 1], (k >> 1) & 1u) && !mbar_wait(&bar[k & 1], (k >> 1) & 1u)) {
            record_error(a.err, PA_DEV_TIMEOUT, 441);
            ok = false;
            break;
        }
        const long long b0 = r_begin + (long long)k * batch;
#pragma unroll
        for (int i = 0; i < SUFFIX_ROWS_PER_LANE; ++i) {
            if (slot[k & 1][i] < 0) continue;
            const long long r = b0 + lane + 32 * i;
            bulk_store((((r & 1) ? a.v_cache : a.k_cache) + slot[k & 1][i] * a.row16),
                       st0 + (k & 1) * half_bytes + (lane + 32 * i) * row_bytes, row_bytes);
        }
        bulk_commit_group();
    }
    bulk_wait0();  // the rows are in global memory and the staging memory is free
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait; the abort flag is only read once the barrier is not yet complete.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *flags, DevError *err,
                                              int where) {
    if (mbar_try_wait(smem_addr(bar), parity)) return true;
    if (flags[0]) return false;
    if (mbar_wait(bar, parity)) return true;
    record_error(err, PA_DEV_TIMEOUT, where);
    flags[0] = 1;
    return false;
}

// Softmax arithmetic with fewer instructions per score: a three-input max,
// and fp32x2 (two-lane) fma/add, all native on sm_100-class SMs.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Byte offset of 16-byte chunk c (0..15) of row r in a [half][128 rows][64]
// tile with 128-byte swizzle (the layout TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((c >> 3) * HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Coordinates of work unit t: the highest query tiles (the most keys) come
// first, then sequence, then q head (the heads of one kv head are
// neighbours, so their K/V tiles are reused from L2).
struct Unit {
    int s, h, m0, q0, Lq, k0, Lk, n_kv, key_end, valid;
};
static_assert(sizeof(Unit) <= 48, "next-unit slot");
static_assert(QST == 2, "the next-unit ring reuses a slot with the Q buffer of the same parity");

// A group is (query tile mt, sequence s), numbered (mtiles-1-mt) * num_seqs
// + s: the query tiles from the highest down, then the sequences.
// KV tiles of group (mt, s); 0 when the query tile is empty or the lengths
// are invalid.
__device__ __forceinline__ int group_tiles(const PrefillArgs &a, int mt, int s) {
    const int Lq = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
    const int Lk = __ldg(a.cu_k + s + 1) - __ldg(a.cu_k + s);
    const bool bad = Lq < 0 || Lk < Lq || (a.paged && Lk > a.max_blocks * a.block_size);
    if (bad || mt * BM >= Lq) return 0;
    const int last_row = min(mt * BM + BM, Lq) - 1;
    const int key_end = a.causal ? min(Lk, Lk - Lq + last_row + 1) : Lk;
    return (key_end + a.bn - 1) / a.bn;
}

// Unit t.  Sorted schedule: t = rank * upg + q head, where rank indexes the
// groups sorted longest first.  Otherwise t = ((mtiles-1-mt) * num_seqs + s)
// * upg + q head (empty query tiles included; next_valid_unit skips them).
// (The paired kernel reads U.h as the head pair and recomputes the tiles.)
__device__ __forceinline__ Unit unit_of(const PrefillArgs &a, const uint16_t *sched, int t) {
    Unit U;
    const int grp = a.sorted ? (int)sched[t / a.upg] : t / a.upg;
    const int mt = a.mtiles - 1 - grp / a.num_seqs;
    U.s = grp % a.num_seqs;
    U.h = t % a.upg;
    U.m0 = mt * BM;
    U.q0 = __ldg(a.cu_q + U.s);
    U.Lq = __ldg(a.cu_q + U.s + 1) - U.q0;
    U.k0 = __ldg(a.cu_k + U.s);
    U.Lk = __ldg(a.cu_k + U.s + 1) - U.k0;
    const bool bad = U.Lq < 0 || U.Lk < U.Lq || (a.paged && U.Lk > a.max_blocks * a.block_size);
    U.valid = !bad && U.m0 < U.Lq;
    if (bad && mt == 0 && U.h == 0 && threadIdx.x == 0) record_error(a.err, PA_DEV_BAD_SEQLENS, U.s);
    U.key_end = 0;
    U.n_kv = 0;
    if (U.valid) {
        const int c = U.Lk - U.Lq;
        const int last_row = min(U.m0 + BM, U.Lq) - 1;
        U.key_end = a.causal ? min(U.Lk, c + last_row + 1) : U.Lk;
        U.n_kv = (U.key_end + a.bn - 1) / a.bn;
    }
    return U;
}

// First unit >= t (stepping by gridDim.x) whose query rows exist (unsorted
// schedule).  The warp
// tests 32 candidates per round of loads and takes the first by ballot, so
// skipping the many empty high query tiles costs one load latency per 32.
// Every lane must call it; every role gets the same answer.
__device__ __forceinline__ int next_valid_unit(const PrefillArgs &a, int t, int nunits, int lane) {
    const int per = a.num_seqs * a.upg;
    for (int base = t; base < nunits; base += 32 * (int)gridDim.x) {
        const int tt = base + lane * (int)gridDim.x;
        bool v = false;
        if (tt < nunits) {
            const int mt = a.mtiles - 1 - tt / per;
            const int s = (tt % per) / a.upg;
            v = mt * BM < __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
        }
        const unsigned m = __ballot_sync(FULL, v);
        if (m) return base + (__ffs(m) - 1) * (int)gridDim.x;
    }
    return nunits;
}

// Unit number k of this CTA (prev: its unit number k - 1), nunits after the
// last.  Sorted schedule: round k of gridDim.x consecutive units goes to the
// CTAs in ascending order when k is even and descending when k is odd, so
// every CTA gets a long and a short unit in each pair of rounds.  Warp-
// collective; every role gets the same sequence.
__device__ __forceinline__ int cta_unit(const PrefillArgs &a, int nsorted, int k, int prev, int nunits, int lane) {
    if (a.sorted) {
        const long long t = (long long)k * gridDim.x + ((k & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
        return t < nsorted ? (int)t : nunits;
    }
    return next_valid_unit(a, k == 0 ? (int)blockIdx.x : prev + (int)gridDim.x, nunits, lane);
}

template <bool STORE>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                   const PrefillArgs a) {
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
    const int nunits = a.mtiles * a.num_seqs * a.upg;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) {
            const bool per_warp = (i >= B_PFULL && i < B_PFULL + NSB) || i == B_OEMPTY;
            mbar_init(&bar[i], per_warp ? 4u : 1u);  // softmax warps arrive one each
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    uint16_t *sched = reinterpret_cast<uint16_t *>(smem + OFF_SCHED);
    int nsorted = 0;  // groups of the sorted schedule
    if (a.sorted) {
        // Rank every (query tile, sequence) group by (KV tiles descending,
        // group id ascending); the K ring holds the keys until the copies start.
        const int ng = a.mtiles * a.num_seqs;
        uint64_t *key = reinterpret_cast<uint64_t *>(smem + OFF_K);
        for (int g = threadIdx.x; g < ng; g += NTHREADS) {
            const int mt = a.mtiles - 1 - g / a.num_seqs, s = g % a.num_seqs;
            const int n = group_tiles(a, mt, s);
            key[g] = n > 0 ? ((uint64_t)n << 32) | (uint32_t)(0xffffffffu - (uint32_t)g) : 0ull;
            if (n == 0 && mt == 0 && blockIdx.x == 0) {
                const int Lq = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
                const int Lk = __ldg(a.cu_k + s + 1) - __ldg(a.cu_k + s);
                if (Lq < 0 || Lk < Lq || (a.paged && Lk > a.max_blocks * a.block_size))
                    record_error(a.err, PA_DEV_BAD_SEQLENS, s);
            }
        }
        __syncthreads();
        // Every thread scans all keys at least once (which also counts the
        // non-empty groups); a group's rank is the number of larger keys.
        for (int g = threadIdx.x, first = 1; first || g < ng; g += NTHREADS, first = 0) {
            const uint64_t mine = g < ng ? key[g] : 0ull;
            int rank = 0, nz = 0;
            for (int j = 0; j < ng; ++j) {
                const uint64_t kj = key[j];
                rank += kj > mine;
                nz += kj != 0ull;
            }
            if (first) nsorted = nz;
            if (mine != 0ull) sched[rank] = (uint16_t)g;
        }
        // The K ring's first bytes are written by TMA next: order these
        // generic-proxy accesses before them.
        fence_proxy_async_smem();
    }
    if (STORE) {
        // Fused store: the suffix rows go to the caches first; the grid
        // barrier makes every CTA's copies visible before any tile is loaded
        // (proxy fences on both sides of it).
        if (warp == 0 && !store_suffix(a, smem + OFF_Q, OFF_BAR - OFF_Q, &bar[B_SUFFIX], lane) && lane == 0)
            flags[0] = 1;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0 && !grid_barrier(a.gbar, gridDim.x)) {
            record_error(a.err, PA_DEV_TIMEOUT, 440);
            flags[0] = 1;  // every role skips its work
        }
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    nsorted *= a.upg;  // units of the sorted schedule
    // Unit i goes to slot i & 1; a slot is rewritten only after the softmax read
    // it (the Q.K thread cannot start unit i+2 before the softmax has released
    // the Q buffer of unit i), so a reader is never two phases behind.
    Unit *nu = reinterpret_cast<Unit *>(smem + OFF_NU);

    // Every role walks the same units (cta_unit) and the
    // same global KV-tile counter g, so ring stages and barrier phases agree.
    if (STORE && flags[0]) {
        // The grid barrier gave up: no role starts (nothing was issued yet).
    } else if (warp == W_QK || warp == W_V) {
        // ------------------------------------------------------------ TMA producers
        const bool is_k = warp == W_QK;
        const CUtensorMap *tm = is_k ? &tmk : &tmv;
        const int NS = is_k ? KST : VST;
        const int off = is_k ? OFF_K : OFF_V;
        uint64_t *full = &bar[is_k ? B_KFULL : B_VFULL];
        uint64_t *empty = &bar[is_k ? B_KEMPTY : B_VEMPTY];
        int *bid = reinterpret_cast<int *>(smem + OFF_BID) + (is_k ? 0 : NBID);
        if (lane == 0) {
            if (is_k) prefetch_tensormap(&tmq);
            prefetch_tensormap(tm);
        }
        const int R = a.box_rows;
        uint32_t g = 0, u = 0, nq = 0;  // KV tiles, units and Q copies issued by this warp
        bool ok = true;
        for (int k = 0, t = cta_unit(a, nsorted, 0, 0, nunits, lane); ok && t < nunits;
             ++k, t = cta_unit(a, nsorted, k, t, nunits, lane)) {
            const Unit U = unit_of(a, sched, t);
            const int32_t *bt = a.bt + (int64_t)U.s * a.max_blocks;
            if (U.valid && a.paged) {
                // The warp fetches the unit's first NBID block ids at once.
                const int nblk = min((U.key_end - 1) / a.block_size + 1, NBID);
                for (int b = lane; b < nblk; b += 32) bid[b] = __ldg(bt + b);
            }
            __syncwarp();
            if (lane == 0 && U.valid) {
                const int kvh = U.h / a.group;
                if (is_k) {
                    const int qb = u % QST;
                    ok = wait_or_abort(&bar[B_QEMPTY + qb], ((u / QST) & 1u) ^ 1u, flags, a.err, 400);
                    if (ok) {
                        mbar_arrive_expect_tx(&bar[B_QFULL + qb], TILE_BYTES);
                        tma_load_4d_plain(smem + OFF_Q + qb * TILE_BYTES, &tmq, 0, U.q0 + U.m0, 0, U.h,
                                          &bar[B_QFULL + qb]);
                        ++nq;
                    }
                }
                for (int j = 0; ok && j < U.n_kv; ++j, ++g) {
                    const int st = g % NS;
                    const int kb = j * BN;
                    const int nsub = (min(BN, U.key_end - kb) + R - 1) / R;
                    if (!(ok = wait_or_abort(&empty[st], ((g / NS) & 1u) ^ 1u, flags, a.err, 401))) break;
                    mbar_arrive_expect_tx(&full[st], (uint32_t)nsub * R * D * 2);
                    uint8_t *dst = smem + off + st * TILE_BYTES;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int key = kb + sub * R;
                        int row;
                        if (a.paged) {
                            const int lb = key / a.block_size;
                            const int blk = lb < NBID ? bid[lb] : __ldg(bt + lb);
                            if (a.checked && is_k && (blk < 0 || blk >= a.num_blocks))
                                record_error(a.err, PA_DEV_BAD_BLOCK, (long long)U.s * a.max_blocks + lb);
                            // An invalid block id reads as zeros: TMA fills out-of-range boxes.
                            row = (blk < 0 || blk >= a.num_blocks) ? -2 * R : blk * a.block_size + key % a.block_size;
                        } else {
                            row = U.k0 + key;
                        }
                        if (a.box_halves == 2) {
                            tma_load_4d_plain(dst, tm, 0, row, 0, kvh, &full[st]);
                        } else {
                            tma_load_4d_plain(dst + sub * R * 128, tm, 0, row, 0, kvh, &full[st]);
                            tma_load_4d_plain(dst + HALF_BYTES + sub * R * 128, tm, 0, row, 1, kvh, &full[st]);
                        }
                    }
                }
                ++u;
            }
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0 && !ok) {
            // Let issued copies land before the CTA's shared memory is released.
            for (uint32_t x = (nq >= (uint32_t)QST ? nq - QST : 0); is_k && x < nq; ++x)
                (void)mbar_wait(&bar[B_QFULL + x % QST], (x / QST) & 1u);
            for (uint32_t x = (g >= (uint32_t)NS ? g - NS : 0); x < g; ++x) (void)mbar_wait(&full[x % NS], (x / NS) & 1u);
        }
    } else if (warp == W_MMA || warp == W_PV) {
        // ------------------------------------------------------------ MMA issuers (lane 0)
        const bool is_qk = warp == W_MMA;
        uint32_t g = 0, u = 0;  // KV tiles and units
        bool ok = true, issued = false;
        // S[buffer gk & 1] = Q K(gk)^T, Q from TMEM.
        uint64_t qdesc = 0;
        auto qk = [&](uint32_t gk) -> bool {
            const int ks = gk % KST, sb = gk % NSB;
            if (!wait_or_abort(&bar[B_KFULL + ks], (gk / KST) & 1u, flags, a.err, 418)) return false;
            // The P.V that read this buffer NSB tiles ago must be complete.
            if (!wait_or_abort(&bar[B_PDONE + sb], ((gk / NSB) & 1u) ^ 1u, flags, a.err, 419)) return false;
            tc_fence_after();
            const uint64_t kdesc = smem_desc_sw128(smem_addr(smem + OFF_K + ks * TILE_BYTES), 16, SBO);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t o = (uint64_t)(((k >> 2) * HALF_BYTES + (k & 3) * 32) >> 4);
                mma_bf16_ss(tmem + COL_S + sb * BN, qdesc + o, kdesc + o, IDESC_S, k > 0 ? 1u : 0u);
            }
            mma_commit(&bar[B_SFULL + sb]);
            mma_commit(&bar[B_KEMPTY + ks]);
            issued = true;
            return true;
        };
        // O += P V for KV tile gv = g + jj of the current unit.
        auto pv = [&](const Unit &U, int jj) -> bool {
            const uint32_t gv = g + jj;
            const int vs = gv % VST, sb = gv % NSB;
            if (jj == 0 && !wait_or_abort(&bar[B_OEMPTY], (u & 1u) ^ 1u, flags, a.err, 410)) return false;
            if (!wait_or_abort(&bar[B_PFULL + sb], (gv / NSB) & 1u, flags, a.err, 412)) return false;
            if (!wait_or_abort(&bar[B_VFULL + vs], (gv / VST) & 1u, flags, a.err, 414)) return false;
            const int kend = min(BN, U.key_end - jj * BN);  // keys of this tile that are needed
            const int kpad = (kend + 15) & ~15;
            if (kend < kpad) {
                // Rows kend..kpad-1 are read by the last 16-key step: zero them.
                const uint32_t vb = smem_addr(smem + OFF_V + vs * TILE_BYTES);
                for (int r = kend; r < kpad; ++r)
                    for (int c = 0; c < 16; ++c) st_shared_v4(vb + sw128_off(r, c), 0, 0, 0, 0);
                fence_proxy_async_smem();
            }
            tc_fence_after();
            const uint64_t vdesc = smem_desc_sw128(smem_addr(smem + OFF_V + vs * TILE_BYTES), HALF_BYTES, SBO);
            for (int k = 0; k < kpad / 16; ++k)  // 16 keys per step = 8 TMEM columns of P
                mma_bf16_ts(tmem + COL_O, tmem + COL_S + sb * BN + k * 8, vdesc + (uint64_t)((k * 16 * 128) >> 4),
                            IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bar[B_VEMPTY + vs]);
            mma_commit(&bar[B_PDONE + sb]);
            issued = true;
            return true;
        };
        // Unit i goes to slot i & 1 of the softmax's next-unit ring once the Q
        // buffer of unit i - 2 is released.  The softmax releases that buffer
        // only after all its threads passed unit i - 2's epilogue barrier and
        // after it published the first P of unit i - 1, so every thread has
        // read slot i & 1 (unit i - 2) before it is rewritten, and a waiter is
        // never two phases behind.
        auto post_unit = [&](uint32_t i, const Unit &V) -> bool {
            if (!wait_or_abort(&bar[B_QEMPTY + i % QST], ((i / QST) & 1u) ^ 1u, flags, a.err, 417)) return false;
            nu[i & 1] = V;
            mbar_arrive(&bar[B_NU + (i & 1)]);
            return true;
        };
        // All lanes walk the units (cta_unit is warp-collective); lane 0
        // waits and issues.
        for (int k = 0, t = cta_unit(a, nsorted, 0, 0, nunits, lane); ok && t < nunits;
             ++k, t = cta_unit(a, nsorted, k, t, nunits, lane)) {
            const Unit U = unit_of(a, sched, t);
            if (!U.valid) continue;
            if (lane == 0) {
                if (is_qk) {
                    // The softmax warps learn their next unit here, off their critical path.
                    ok = post_unit(u, U);
                    ok = ok && wait_or_abort(&bar[B_QFULL + u % QST], (u / QST) & 1u, flags, a.err, 416);
                    qdesc = smem_desc_sw128(smem_addr(smem + OFF_Q + (u % QST) * TILE_BYTES), 16, SBO);
                    for (int j = 0; ok && j < U.n_kv; ++j) ok = qk(g + j);
                } else {
                    for (int j = 0; ok && j < U.n_kv; ++j) ok = pv(U, j);
                }
            }
            g += U.n_kv;
            ++u;
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0 && ok && is_qk) {  // the end of the CTA's units
            Unit end = {};
            end.valid = 0;
            (void)post_unit(u, end);
        }
        if (lane == 0 && !ok && issued) {
            // Let the issued MMAs finish before TMEM is released.
            uint64_t *dr = &bar[is_qk ? B_DRAIN : B_DRAIN2];
            mma_commit(dr);
            (void)mbar_wait(dr, 0);
        }
    } else if (warp >= W_SOFT) {
        // ------------------------------------------------------------ softmax, epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // tile row == TMEM lane
        const int tid = threadIdx.x - W_SOFT * 32;  // 0..127
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl = a.scale_log2;
        uint32_t gs = 0, u = 0;  // S tiles consumed, units finished
        bool ok = true;
        // Waits in this role are warp-uniform: tcgen05.ld/st are warp-collective.
        auto wwait = [&](uint64_t *b, uint32_t parity, int where) -> bool {
            return __all_sync(FULL, wait_or_abort(b, parity, flags, a.err, where));
        };
        // P.V number x (global tile count) and all before it have completed:
        // wait for its commit on PDONE[x % NSB].  Called only after S(x) was
        // waited for: the Q.K that wrote S(x) had waited for this barrier's
        // previous phase (P.V x - NSB), so the phase awaited is the next to
        // complete, never one further (a parity wait would pass at once); and
        // P.V x + NSB needs a P this warpgroup has not published yet.
        auto wait_o = [&](uint32_t x) -> bool { return wwait(&bar[B_PDONE + x % NSB], (x / NSB) & 1u, 421); };
        auto take_unit = [&](uint32_t i, Unit &U) -> bool {
            if (!wwait(&bar[B_NU + (i & 1)], (i >> 1) & 1u, 430)) return false;
            U = nu[i & 1];
            return U.valid != 0;
        };
        Unit U;
        bool have = take_unit(0, U);
        int pend_q = -1;  // Q buffer whose output store still has to be read out (thread 0)
        while (ok && have) {
            const int i = U.m0 + row;  // query index in the sequence (>= Lq: padding row)
            const int pos = (U.Lk - U.Lq) + i;
            const int key_last = (a.causal ? min(pos, U.Lk - 1) : U.Lk - 1);  // last key this row sees
            float m_run = -INFINITY;  // running reference max of raw scores
            float l_run = 0.f;        // running sum of P relative to it
            for (int j = 0; j < U.n_kv; ++j, ++gs) {
                const int sb = gs % NSB;
                const uint32_t cs = t_lane + COL_S + sb * BN;
                if (!(ok = wwait(&bar[B_SFULL + sb], (gs / NSB) & 1u, 420))) break;
                tc_fence_after();
                uint32_t r[128];
                tmem_ld32(cs, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(cs + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_ld32(cs + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
                tmem_ld32(cs + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
                tmem_ld_wait();
                const int lim = key_last - j * BN;  // keys j*BN + k with k <= lim are visible
                if (__any_sync(FULL, lim < BN - 1)) {
#pragma unroll
                    for (int k = 0; k < BN; ++k)
                        if (k > lim) r[k] = __float_as_uint(-INFINITY);
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k2 = 0; k2 < BN / 2; ++k2)
                    m4[k2 & 3] = max3f(m4[k2 & 3], __uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1]));
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                // Lazy rescaling: keep the old max unless this tile's max exceeds it
                // by more than 8 in log2 units (P then stays <= 2^8).
                const bool grow = (mx - m_run) * sl > 8.f;
                const float m_new = grow ? mx : m_run;
                const float alpha = grow ? fast_exp2((m_run - m_new) * sl) : 1.f;
                if (j > 0 && __any_sync(FULL, grow)) {
                    // O must hold P.V up to tile j-1 before it is rescaled.
                    if (!(ok = wait_o(gs - 1))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + COL_O + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(t_lane + COL_O + c * 32, o);
                    }
                }
                l_run *= alpha;
                m_run = m_new;
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * sl;
                // P = 2^(s*scale - m) as bf16 pairs over the first 64 columns of the buffer.
                float2 rs[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
                const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(neg_m, neg_m);
                uint32_t pk[64];
#pragma unroll
                for (int k2 = 0; k2 < 64; ++k2) {
                    const float2 xx =
                        fma2(make_float2(__uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1])), sl2, nm2);
                    const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                    rs[k2 & 3] = add2(rs[k2 & 3], pp);
                    pk[k2] = pack_bf16(pp.x, pp.y);
                }
                tmem_st32(cs, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
                tmem_st32(cs + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
                tmem_st_wait();
                l_run += ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_PFULL + sb]);
                if (tid == 0 && pend_q >= 0) {
                    // The previous unit's tile store has read its staging buffer by
                    // now: release the buffer for a later Q.
                    bulk_wait_read0();
                    mbar_arrive(&bar[B_QEMPTY + pend_q]);
                    pend_q = -1;
                }
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 tile in shared memory -> global memory
            if (!(ok = wait_o(gs - 1))) break;
            tc_fence_after();
            uint32_t o[128];
            tmem_ld32(t_lane + COL_O, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            tmem_ld32(t_lane + COL_O + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
            tmem_ld32(t_lane + COL_O + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[64]));
            tmem_ld32(t_lane + COL_O + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[96]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OEMPTY]);  // O may be overwritten by the next unit
            // This unit's Q buffer stages the output tile: every Q.K that read it
            // is complete (this warp waited for the unit's last S).
            const uint32_t os = smem_addr(smem + OFF_Q + (u % QST) * TILE_BYTES);
            const float inv = 1.f / l_run;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t *v = &o[8 * c];
                st_shared_v4(os + sw128_off(row, c),
                             pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                             pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                             pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                             pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            }
            const int nrows = min(BM, U.Lq - U.m0);
            if (nrows == BM) {
                fence_proxy_async_smem();  // the tile store reads the staging tile through the async proxy
                named_bar_sync(SOFT_BAR, 128);
                if (tid == 0) {
                    tma_store_4d(&tmo, smem + OFF_Q + (u % QST) * TILE_BYTES, 0, U.q0 + U.m0, 0, U.h);
                    bulk_commit_group();
                    pend_q = u % QST;  // released after the next tile (or below, at the end)
                }
            } else {
                // The last tile of a sequence: rows past Lq belong to the next
                // sequence, so only the valid rows are written, 16 threads per row.
                named_bar_sync(SOFT_BAR, 128);
#pragma unroll 4
                for (int it = 0; it < BM * 16 / 128; ++it) {
                    const int q = it * 128 + tid, rr = q >> 4, c = q & 15;
                    if (rr < nrows) {
                        const uint4 v = ld_shared_v4(os + sw128_off(rr, c));
                        *reinterpret_cast<uint4 *>(a.out + ((int64_t)(U.q0 + U.m0 + rr) * a.Hq + U.h) * D + c * 8) = v;
                    }
                }
                named_bar_sync(SOFT_BAR, 128);  // the staging tile was read
                if (tid == 0) pend_q = u % QST;   // released with the next unit's first P, like a tile store
            }
            ++u;
            have = ok && take_unit(u, U);
        }
        if (tid == 0 && pend_q >= 0) {
            bulk_wait_read0();
            mbar_arrive(&bar[B_QEMPTY + pend_q]);
        }
        if (tid == 0) bulk_wait0();  // tile stores complete before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ===========================================================================
// Paired-head prefill (GQA groups of even size).
//
// A work unit is one 128-row query tile of one sequence for two q heads of
// the same kv head (A = head 2p, B = head 2p+1), so each K/V tile is loaded
// once for both.  The keys come in tiles of 64.  TMEM (512 columns) holds,
// per head, two S/P buffers of 64 columns and the 128-column O: S(A,0..1) at
// 0 and 64, S(B,0..1) at 128 and 192, O(A) at 256, O(B) at 384.  Each head has
// its own softmax warpgroup, so the two heads' exponentials run side by side,
// and with two S buffers per head the tensor cores compute the scores of the
// next tile while the softmax works on the current one.
//  * warp 0 loads Q (both heads' tiles into the unit's pair of Q slots; the
//    next unit's pair is loaded while this one runs) and the K tiles, warp 2
//    the V tiles (rings of three 16 KiB stages).
//  * warp 1 issues S(h, b) = Q(h).K^T (M = 128, N = 64, K = 128: 8 MMAs)
//    for both heads into buffer b = tile & 1, once the P.V that last read the
//    buffer has completed; warp 3 issues O(h) += P(h).V (M = 128, N = 128,
//    K = 64: 4 MMAs, P from TMEM) for both heads once P is published.
//  * warps 4..7 (head A) and 8..11 (head B): one thread per query row, online
//    softmax in base 2 over the 64 scores of a tile, lazy rescaling of O (only
//    when a row max grows by more than 2^8), P as bf16 pairs over the first
//    32 columns of the S buffer; at the end of a unit O / l -> bf16 into the
//    head's Q slot (no longer read) -> TMA store (full tiles) or row stores.
// ===========================================================================
constexpr int P2_BN = 64;                      // keys per KV tile
constexpr int P2_KV_BYTES = P2_BN * D * 2;     // 16 KiB
constexpr int P2_KV_HALF = P2_KV_BYTES / 2;    // [64 rows][64 dims]
constexpr int P2_NTHREADS = 384;
constexpr int P2_W_QLK = 0, P2_W_QK = 1, P2_W_V = 2, P2_W_PV = 3, P2_W_SOFT = 4;  // softmax warps 4..11
constexpr int P2_QS = 4;  // Q slots: unit u uses 2 * (u & 1) (head A) and 2 * (u & 1) + 1 (head B)
constexpr int P2_KS = 3, P2_VS = 3;
constexpr int P2_OFF_Q = 0;
constexpr int P2_OFF_K = P2_OFF_Q + P2_QS * TILE_BYTES;
constexpr int P2_OFF_V = P2_OFF_K + P2_KS * P2_KV_BYTES;
constexpr int P2_OFF_BAR = P2_OFF_V + P2_VS * P2_KV_BYTES;
enum {
    C_QFULL = 0, C_QEMPTY = C_QFULL + P2_QS, C_KFULL = C_QEMPTY + P2_QS, C_KEMPTY = C_KFULL + P2_KS,
    C_VFULL = C_KEMPTY + P2_KS, C_VEMPTY = C_VFULL + P2_VS,
    C_SFULL = C_VEMPTY + P2_VS /* [head][buffer] */, C_PFULL = C_SFULL + 4 /* [head][buffer] */,
    C_PDONE = C_PFULL + 4 /* [head][buffer] */, C_OEMPTY = C_PDONE + 4 /* [head] */, C_DRAIN = C_OEMPTY + 2,
    C_DRAIN2, C_SUFFIX /* [2] */, P2_NBAR = C_SUFFIX + 2
};
constexpr int P2_OFF_TMEM = P2_OFF_BAR + P2_NBAR * 8;
constexpr int P2_OFF_FLAGS = P2_OFF_TMEM + 8;
constexpr int P2_OFF_BID = P2_OFF_FLAGS + 16;         // block ids of the current unit, per loader warp
constexpr int P2_OFF_SCHED = P2_OFF_BID + 2 * NBID * 4;
constexpr int P2_SMEM_USED = P2_OFF_SCHED + SCHED_MAX * 2;
constexpr size_t P2_SMEM_BYTES = P2_SMEM_USED + SMEM_SLACK;
static_assert(P2_SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SCHED_MAX * 8 <= P2_KS * P2_KV_BYTES, "the sort keys fit in the K ring");
constexpr uint32_t P2_COL_S = 0, P2_COL_O = 256;  // S(h, b) at h * 128 + b * 64; O(h) at 256 + h * 128
constexpr uint32_t P2_IDESC_S = idesc_bf16_f32(BM, P2_BN, false, false);

template <bool STORE>
__global__ void __launch_bounds__(P2_NTHREADS, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                        const PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    if (pad > (uint32_t)SMEM_SLACK) {
        if (threadIdx.x == 0) record_error(a.err, PA_DEV_SMEM_ALIGN, (long long)pad);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P2_OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P2_OFF_TMEM);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + P2_OFF_FLAGS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nunits = a.mtiles * a.num_seqs * a.upg;

    if (threadIdx.x == 0) {
        for (int i = 0; i < P2_NBAR; ++i) {
            const bool per_warp = (i >= C_PFULL && i < C_PFULL + 4) || i == C_OEMPTY || i == C_OEMPTY + 1;
            mbar_init(&bar[i], per_warp ? 4u : 1u);  // the softmax warps of a head arrive one each
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == P2_W_QK) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    uint16_t *sched = reinterpret_cast<uint16_t *>(smem + P2_OFF_SCHED);
    int nsorted = 0;
    if (a.sorted) {
        // Rank the (query tile, sequence) groups by (KV tiles descending, group
        // id ascending); the K ring holds the keys until the copies start.
        const int ng = a.mtiles * a.num_seqs;
        uint64_t *key = reinterpret_cast<uint64_t *>(smem + P2_OFF_K);
        for (int g = threadIdx.x; g < ng; g += P2_NTHREADS) {
            const int mt = a.mtiles - 1 - g / a.num_seqs, s = g % a.num_seqs;
            const int n = group_tiles(a, mt, s);
            key[g] = n > 0 ? ((uint64_t)n << 32) | (uint32_t)(0xffffffffu - (uint32_t)g) : 0ull;
            if (n == 0 && mt == 0 && blockIdx.x == 0) {
                const int Lq = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
                const int Lk = __ldg(a.cu_k + s + 1) - __ldg(a.cu_k + s);
                if (Lq < 0 || Lk < Lq || (a.paged && Lk > a.max_blocks * a.block_size))
                    record_error(a.err, PA_DEV_BAD_SEQLENS, s);
            }
        }
        __syncthreads();
        for (int g = threadIdx.x, first = 1; first || g < ng; g += P2_NTHREADS, first = 0) {
            const uint64_t mine = g < ng ? key[g] : 0ull;
            int rank = 0, nz = 0;
            for (int j = 0; j < ng; ++j) {
                const uint64_t kj = key[j];
                rank += kj > mine;
                nz += kj != 0ull;
            }
            if (first) nsorted = nz;
            if (mine != 0ull) sched[rank] = (uint16_t)g;
        }
        fence_proxy_async_smem();
    }
    if (STORE) {
        if (warp == 0 && !store_suffix(a, smem + P2_OFF_Q, P2_OFF_BAR - P2_OFF_Q, &bar[C_SUFFIX], lane) && lane == 0)
            flags[0] = 1;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0 && !grid_barrier(a.gbar, gridDim.x)) {
            record_error(a.err, PA_DEV_TIMEOUT, 440);
            flags[0] = 1;
        }
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    nsorted *= a.upg;

    // Every role walks the same units and the same KV-tile counter g, so the
    // ring stages, S buffers and barrier phases agree.
    if (STORE && flags[0]) {
        // The grid barrier gave up: no role starts.
    } else if (warp == P2_W_QLK || warp == P2_W_V) {
        // ------------------------------------------------------------ TMA loads
        const bool is_k = warp == P2_W_QLK;
        const CUtensorMap *tm = is_k ? &tmk : &tmv;
        const int off = is_k ? P2_OFF_K : P2_OFF_V;
        uint64_t *full = &bar[is_k ? C_KFULL : C_VFULL];
        uint64_t *empty = &bar[is_k ? C_KEMPTY : C_VEMPTY];
        int *bid = reinterpret_cast<int *>(smem + P2_OFF_BID) + (is_k ? 0 : NBID);
        if (lane == 0) {
            if (is_k) prefetch_tensormap(&tmq);
            prefetch_tensormap(tm);
        }
        const int R = a.box_rows;  // rows per box: gcd(block_size, 64)
        uint32_t g = 0, u = 0, nq = 0;
        bool ok = true;
        for (int k = 0, t = cta_unit(a, nsorted, 0, 0, nunits, lane); ok && t < nunits;
             ++k, t = cta_unit(a, nsorted, k, t, nunits, lane)) {
            const Unit U = unit_of(a, sched, t);
            const int32_t *bt = a.bt + (int64_t)U.s * a.max_blocks;
            if (U.valid && a.paged) {
                const int nblk = min((U.key_end - 1) / a.block_size + 1, NBID);
                for (int b = lane; b < nblk; b += 32) bid[b] = __ldg(bt + b);
            }
            __syncwarp();
            if (lane == 0 && U.valid) {
                const int h0 = 2 * U.h, kvh = h0 / a.group;
                if (is_k) {
                    for (int x = 0; ok && x < 2; ++x) {
                        const int qs = 2 * (u & 1) + x;
                        ok = wait_or_abort(&bar[C_QEMPTY + qs], ((u >> 1) & 1u) ^ 1u, flags, a.err, 500);
                        if (ok) {
                            mbar_arrive_expect_tx(&bar[C_QFULL + qs], TILE_BYTES);
                            tma_load_4d_plain(smem + P2_OFF_Q + qs * TILE_BYTES, &tmq, 0, U.q0 + U.m0, 0, h0 + x,
                                              &bar[C_QFULL + qs]);
                            ++nq;
                        }
                    }
                }
                for (int j = 0; ok && j < U.n_kv; ++j, ++g) {
                    const int st = g % P2_KS;
                    const int kb = j * P2_BN;
                    const int nsub = (min(P2_BN, U.key_end - kb) + R - 1) / R;
                    if (!(ok = wait_or_abort(&empty[st], ((g / P2_KS) & 1u) ^ 1u, flags, a.err, 501))) break;
                    mbar_arrive_expect_tx(&full[st], (uint32_t)nsub * R * D * 2);
                    uint8_t *dst = smem + off + st * P2_KV_BYTES;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int key = kb + sub * R;
                        int row;
                        if (a.paged) {
                            const int lb = key / a.block_size;
                            const int blk = lb < NBID ? bid[lb] : __ldg(bt + lb);
                            if (a.checked && is_k && (blk < 0 || blk >= a.num_blocks))
                                record_error(a.err, PA_DEV_BAD_BLOCK, (long long)U.s * a.max_blocks + lb);
                            row = (blk < 0 || blk >= a.num_blocks) ? -2 * R : blk * a.block_size + key % a.block_size;
                        } else {
                            row = U.k0 + key;
                        }
                        if (a.box_halves == 2) {
                            tma_load_4d_plain(dst, tm, 0, row, 0, kvh, &full[st]);
                        } else {
                            tma_load_4d_plain(dst + sub * R * 128, tm, 0, row, 0, kvh, &full[st]);
                            tma_load_4d_plain(dst + P2_KV_HALF + sub * R * 128, tm, 0, row, 1, kvh, &full[st]);
                        }
                    }
                }
                ++u;
            }
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0 && !ok) {
            // Let issued copies land before the CTA's shared memory is released.
            for (uint32_t x = (nq >= (uint32_t)P2_QS ? nq - P2_QS : 0); is_k && x < nq; ++x) {
                const uint32_t uu = x >> 1, qs = 2 * (uu & 1) + (x & 1);
                (void)mbar_wait(&bar[C_QFULL + qs], (uu >> 1) & 1u);
            }
            for (uint32_t x = (g >= (uint32_t)P2_KS ? g - P2_KS : 0); x < g; ++x)
                (void)mbar_wait(&full[x % P2_KS], (x / P2_KS) & 1u);
        }
    } else if (warp == P2_W_QK || warp == P2_W_PV) {
        // ------------------------------------------------------------ MMA issuers (lane 0)
        const bool is_qk = warp == P2_W_QK;
        uint32_t g = 0, u = 0;
        bool ok = true, issued = false;
        for (int k = 0, t = cta_unit(a, nsorted, 0, 0, nunits, lane); ok && t < nunits;
             ++k, t = cta_unit(a, nsorted, k, t, nunits, lane)) {
            const Unit U = unit_of(a, sched, t);
            if (!U.valid) continue;
            if (lane == 0 && is_qk) {
                uint64_t qdesc[2];
                for (int x = 0; x < 2; ++x) {
                    const int qs = 2 * (u & 1) + x;
                    ok = ok && wait_or_abort(&bar[C_QFULL + qs], (u >> 1) & 1u, flags, a.err, 510);
                    qdesc[x] = smem_desc_sw128(smem_addr(smem + P2_OFF_Q + qs * TILE_BYTES), 16, SBO);
                }
                for (int j = 0; ok && j < U.n_kv; ++j) {
                    const uint32_t gg = g + j;
                    const int ks = gg % P2_KS, b = gg & 1;
                    if (!(ok = wait_or_abort(&bar[C_KFULL + ks], (gg / P2_KS) & 1u, flags, a.err, 511))) break;
                    const uint64_t kdesc = smem_desc_sw128(smem_addr(smem + P2_OFF_K + ks * P2_KV_BYTES), 16, SBO);
                    for (int x = 0; ok && x < 2; ++x) {
                        // S(x, b) is free once the P.V that read it two tiles ago has completed.
                        if (!(ok = wait_or_abort(&bar[C_PDONE + 2 * x + b], ((gg >> 1) & 1u) ^ 1u, flags, a.err,
                                                 512)))
                            break;
                        tc_fence_after();
                        const uint32_t d = tmem + P2_COL_S + x * 128 + b * 64;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t qo = (uint64_t)(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
                            const uint64_t ko = (uint64_t)(((kk >> 2) * P2_KV_HALF + (kk & 3) * 32) >> 4);
                            mma_bf16_ss(d, qdesc[x] + qo, kdesc + ko, P2_IDESC_S, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&bar[C_SFULL + 2 * x + b]);
                        issued = true;
                    }
                    if (ok) mma_commit(&bar[C_KEMPTY + ks]);
                }
            } else if (lane == 0) {
                for (int j = 0; ok && j < U.n_kv; ++j) {
                    const uint32_t gg = g + j;
                    const int vs = gg % P2_VS, b = gg & 1;
                    if (!(ok = wait_or_abort(&bar[C_VFULL + vs], (gg / P2_VS) & 1u, flags, a.err, 520))) break;
                    const int kend = min(P2_BN, U.key_end - j * P2_BN);  // keys of this tile that are needed
                    const int kpad = (kend + 15) & ~15;
                    const uint32_t vb = smem_addr(smem + P2_OFF_V + vs * P2_KV_BYTES);
                    if (kend < kpad) {
                        // Rows kend..kpad-1 are read by the last 16-key step: zero them
                        // (stale or unloaded data; P is 0 there but 0 * NaN is not 0).
                        for (int r = kend; r < kpad; ++r)
                            for (int c = 0; c < 16; ++c)
                                st_shared_v4(vb + (uint32_t)((c >> 3) * P2_KV_HALF + r * 128 + (((c & 7) ^ (r & 7)) << 4)),
                                             0, 0, 0, 0);
                        fence_proxy_async_smem();
                    }
                    const uint64_t vdesc = smem_desc_sw128(vb, P2_KV_HALF, SBO);
                    for (int x = 0; ok && x < 2; ++x) {
                        if (j == 0 && !(ok = wait_or_abort(&bar[C_OEMPTY + x], (u & 1u) ^ 1u, flags, a.err, 521)))
                            break;
                        if (!(ok = wait_or_abort(&bar[C_PFULL + 2 * x + b], (gg >> 1) & 1u, flags, a.err, 522))) break;
                        tc_fence_after();
                        const uint32_t pcol = tmem + P2_COL_S + x * 128 + b * 64;
                        for (int kk = 0; kk < kpad / 16; ++kk)  // 16 keys per step = 8 TMEM columns of P
                            mma_bf16_ts(tmem + P2_COL_O + x * 128, pcol + kk * 8,
                                        vdesc + (uint64_t)((kk * 16 * 128) >> 4), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bar[C_PDONE + 2 * x + b]);
                        issued = true;
                    }
                    if (ok) mma_commit(&bar[C_VEMPTY + vs]);
                }
            }
            g += U.n_kv;
            ++u;
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0 && !ok && issued) {
            // Let the issued MMAs finish before TMEM is released.
            uint64_t *dr = &bar[is_qk ? C_DRAIN : C_DRAIN2];
            mma_commit(dr);
            (void)mbar_wait(dr, 0);
        }
    } else if (warp >= P2_W_SOFT) {
        // ------------------------------------------------------------ softmax, epilogue (one head each)
        const int x = (warp - P2_W_SOFT) >> 2;  // 0: head A, 1: head B
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // tile row == TMEM lane
        const int tid = threadIdx.x - (P2_W_SOFT + 4 * x) * 32;  // 0..127
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t col_s = P2_COL_S + x * 128, col_o = P2_COL_O + x * 128;
        const float sl = a.scale_log2;
        uint32_t g = 0, u = 0;
        bool ok = true;
        auto wwait = [&](uint64_t *b, uint32_t parity, int where) -> bool {
            return __all_sync(FULL, wait_or_abort(b, parity, flags, a.err, where));
        };
        int pend_q = -1;  // Q slot whose output store still has to be read out (tid 0)
        for (int k = 0, t = cta_unit(a, nsorted, 0, 0, nunits, lane); ok && t < nunits;
             ++k, t = cta_unit(a, nsorted, k, t, nunits, lane)) {
            const Unit U = unit_of(a, sched, t);
            if (!U.valid) continue;
            const int i = U.m0 + row;  // query index in the sequence (>= Lq: padding row)
            const int pos = (U.Lk - U.Lq) + i;
            const int key_last = (a.causal ? min(pos, U.Lk - 1) : U.Lk - 1);
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < U.n_kv; ++j) {
                const uint32_t gg = g + j;
                const int b = gg & 1;
                const uint32_t cs = t_lane + col_s + b * 64;
                if (!(ok = wwait(&bar[C_SFULL + 2 * x + b], (gg >> 1) & 1u, 530))) break;
                tc_fence_after();
                uint32_t r[64];
                tmem_ld32(cs, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(cs + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_ld_wait();
                const int lim = key_last - j * P2_BN;  // keys j*64 + kk with kk <= lim are visible
                if (__any_sync(FULL, lim < P2_BN - 1)) {
#pragma unroll
                    for (int kk = 0; kk < P2_BN; ++kk)
                        if (kk > lim) r[kk] = __float_as_uint(-INFINITY);
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k2 = 0; k2 < P2_BN / 2; ++k2)
                    m4[k2 & 3] = max3f(m4[k2 & 3], __uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1]));
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const bool grow = (mx - m_run) * sl > 8.f;
                const float m_new = grow ? mx : m_run;
                const float alpha = grow ? fast_exp2((m_run - m_new) * sl) : 1.f;
                if (j > 0 && __any_sync(FULL, grow)) {
                    // O must hold P.V up to tile gg-1 before it is rescaled (the one
                    // before that has completed: the Q.K that wrote this S waited for it).
                    if (!(ok = wwait(&bar[C_PDONE + 2 * x + ((gg - 1) & 1)], ((gg - 1) >> 1) & 1u, 531))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + col_o + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(t_lane + col_o + c * 32, o);
                    }
                }
                l_run *= alpha;
                m_run = m_new;
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * sl;
                float2 rs[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
                const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(neg_m, neg_m);
                uint32_t pk[32];
#pragma unroll
                for (int k2 = 0; k2 < 32; ++k2) {
                    const float2 xx =
                        fma2(make_float2(__uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1])), sl2, nm2);
                    const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                    rs[k2 & 3] = add2(rs[k2 & 3], pp);
                    pk[k2] = pack_bf16(pp.x, pp.y);
                }
                tmem_st32(cs, pk);
                tmem_st_wait();
                l_run += ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[C_PFULL + 2 * x + b]);
                if (tid == 0 && pend_q >= 0) {
                    // The previous unit's output store has read its staging slot by now.
                    bulk_wait_read0();
                    mbar_arrive(&bar[C_QEMPTY + pend_q]);
                    pend_q = -1;
                }
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 tile in this head's Q slot -> global memory
            const uint32_t gl = g + U.n_kv - 1;  // the unit's last tile
            if (!(ok = wwait(&bar[C_PDONE + 2 * x + (gl & 1)], (gl >> 1) & 1u, 532))) break;
            tc_fence_after();
            uint32_t o[128];
            tmem_ld32(t_lane + col_o, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            tmem_ld32(t_lane + col_o + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
            tmem_ld32(t_lane + col_o + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[64]));
            tmem_ld32(t_lane + col_o + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[96]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[C_OEMPTY + x]);  // O may be overwritten by the next unit
            const int qs = 2 * (u & 1) + x;
            const uint32_t os = smem_addr(smem + P2_OFF_Q + qs * TILE_BYTES);
            const float inv = 1.f / l_run;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t *v = &o[8 * c];
                st_shared_v4(os + sw128_off(row, c),
                             pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                             pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                             pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                             pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            }
            const int head = 2 * U.h + x;
            const int nrows = min(BM, U.Lq - U.m0);
            if (nrows == BM) {
                fence_proxy_async_smem();
                named_bar_sync(1 + x, 128);
                if (tid == 0) {
                    tma_store_4d(&tmo, smem + P2_OFF_Q + qs * TILE_BYTES, 0, U.q0 + U.m0, 0, head);
                    bulk_commit_group();
                    pend_q = qs;
                }
            } else {
                named_bar_sync(1 + x, 128);
#pragma unroll 4
                for (int it = 0; it < BM * 16 / 128; ++it) {
                    const int q = it * 128 + tid, rr = q >> 4, c = q & 15;
                    if (rr < nrows) {
                        const uint4 v = ld_shared_v4(os + sw128_off(rr, c));
                        *reinterpret_cast<uint4 *>(a.out + ((int64_t)(U.q0 + U.m0 + rr) * a.Hq + head) * D + c * 8) = v;
                    }
                }
                fence_proxy_async_smem();  // the slot's next Q arrives by TMA (async proxy)
                named_bar_sync(1 + x, 128);
                if (tid == 0) pend_q = qs;
            }
            g += U.n_kv;
            ++u;
        }
        if (tid == 0 && pend_q >= 0) {
            bulk_wait_read0();
            mbar_arrive(&bar[C_QEMPTY + pend_q]);
        }
        if (tid == 0) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == P2_W_QK) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Per (device, instantiation): the shared-memory attribute has been set
// (an atomic flag; concurrent first calls may both set the idempotent attribute).
std::atomic<int> g_attr_done[64][4];

// The fused store's inputs (null: plain prefill).
struct SuffixStore {
    const void *new_k, *new_v;
    int64_t new_k_row_stride, new_v_row_stride;  // elements
    unsigned *gbar;
};

pa_status prefill_impl(void *out, const void *q, int64_t q_row_stride, int32_t total_q, const void *k,
                       const void *v, int64_t kv_row_stride, int32_t total_k, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                       int32_t num_seqs, int32_t max_seqlen_q, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, float softmax_scale,
                       int32_t causal, const SuffixStore *store, pa_stream_t stream) {
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
    if (((int64_t)max_seqlen_q + BM - 1) / BM * num_seqs * num_q_heads > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "too many tiles");
    const bool paged = block_tables != nullptr;
    // Even GQA groups run the paired-head kernel (two q heads of one kv head
    // per unit, 64-key tiles); other groups the one-head kernel (128-key tiles).
    const int group = num_q_heads / num_kv_heads;
    const bool paired = group % 2 == 0;
    const int tile_keys = paired ? P2_BN : BN;
    int R = tile_keys;
    if (paged) {
        if (block_size <= 0 || block_size % 16)
            return fail(PA_ERR_UNSUPPORTED, "block_size %d (must be a positive multiple of 16)", block_size);
        if (max_blocks_per_seq <= 0 || num_blocks <= 0)
            return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq and num_blocks must be positive");
        if ((int64_t)num_blocks * block_size > 0x7fffffffLL ||
            (int64_t)max_blocks_per_seq * block_size > 0x7fffffffLL)
            return fail(PA_ERR_UNSUPPORTED, "pool or table too large for 32-bit slot indices");
        while (block_size % R) R >>= 1;  // gcd(block_size, tile_keys) in {16, 32, 64(, 128)}
    } else {
        if (total_k <= 0) return fail(PA_ERR_INVALID_ARG, "total_k must be positive for contiguous k/v");
        if (kv_row_stride < (int64_t)num_kv_heads * D || kv_row_stride % 8)
            return fail(PA_ERR_INVALID_ARG, "kv_row_stride must be >= num_kv_heads*head_dim and a multiple of 8");
    }
    // A box of tile_keys rows holds a whole K/V tile in [half][row][64] order;
    // shorter boxes (small blocks) are fetched one 64-dim half at a time.
    const int halves = R == tile_keys ? 2 : 1;
    CUtensorMap tq, tk, tv;
    pa_status st = encode_halves_map(&tq, q, total_q, q_row_stride * 2, num_q_heads, BM, 2);
    if (st != PA_OK) return st;
    const int64_t kv_rows = paged ? (int64_t)num_blocks * block_size : (int64_t)total_k;
    const int64_t kv_stride = paged ? (int64_t)num_kv_heads * D * 2 : kv_row_stride * 2;
    st = encode_halves_map(&tk, k, kv_rows, kv_stride, num_kv_heads, R, halves);
    if (st == PA_OK) st = encode_halves_map(&tv, v, kv_rows, kv_stride, num_kv_heads, R, halves);
    // Output tiles of 128 full rows go out by TMA store.
    CUtensorMap to;
    if (st == PA_OK) st = encode_halves_map(&to, out, total_q, (int64_t)num_q_heads * D * 2, num_q_heads, BM, 2);
    if (st != PA_OK) return st;

    PrefillArgs A;
    A.out = static_cast<__nv_bfloat16 *>(out);
    A.cu_q = cu_seqlens_q;
    A.cu_k = cu_seqlens_k;
    A.bt = block_tables;
    A.max_blocks = paged ? max_blocks_per_seq : 0;
    A.num_seqs = num_seqs;
    A.Hq = num_q_heads;
    A.group = group;
    A.mtiles = (max_seqlen_q + BM - 1) / BM;
    A.upg = paired ? num_q_heads / 2 : num_q_heads;
    A.bn = tile_keys;
    A.block_size = paged ? block_size : 1;
    A.box_rows = R;
    A.box_halves = halves;
    A.paged = paged ? 1 : 0;
    A.causal = causal ? 1 : 0;
    A.num_blocks = num_blocks;
    A.checked = checked_mode() ? 1 : 0;
    A.sorted = (int64_t)A.mtiles * num_seqs <= SCHED_MAX ? 1 : 0;
    A.scale_log2 = softmax_scale * 1.4426950408889634f;
    A.err = device_error_ptr();
    A.new_k = store ? static_cast<const uint4 *>(store->new_k) : nullptr;
    A.new_v = store ? static_cast<const uint4 *>(store->new_v) : nullptr;
    A.new_k_stride16 = store ? store->new_k_row_stride / 8 : 0;
    A.new_v_stride16 = store ? store->new_v_row_stride / 8 : 0;
    A.k_cache = store ? static_cast<uint4 *>(const_cast<void *>(k)) : nullptr;
    A.v_cache = store ? static_cast<uint4 *>(const_cast<void *>(v)) : nullptr;
    A.row16 = num_kv_heads * D / 8;
    A.total_q = total_q;
    A.gbar = store ? store->gbar : nullptr;

    const int64_t nunits = (int64_t)A.mtiles * num_seqs * A.upg;
    const int sms = sm_count();
    if (sms <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    const int64_t grid = std::min<int64_t>(nunits, sms);  // persistent: one CTA per SM
    int dev = 0;
    cudaGetDevice(&dev);
    using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, PrefillArgs);
    const KernelFn kern = paired ? (store ? prefill_pair_kernel<true> : prefill_pair_kernel<false>)
                                 : (store ? prefill_kernel<true> : prefill_kernel<false>);
    const size_t smem_bytes = paired ? P2_SMEM_BYTES : SMEM_BYTES;
    const int threads = paired ? P2_NTHREADS : NTHREADS;
    const int fi = (store ? 1 : 0) + (paired ? 2 : 0);
    if (dev >= 0 && dev < 64 && !g_attr_done[dev][fi].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_kernel)");
        g_attr_done[dev][fi].store(1, std::memory_order_release);
    }
    if (!store) {
        kern<<<(unsigned)grid, threads, smem_bytes, reinterpret_cast<cudaStream_t>(stream)>>>(tq, tk, tv, to, A);
        return check_launch("prefill_kernel");
    }
    // The fused store's CTAs wait on one another at the grid barrier: a
    // cooperative launch guarantees they are resident together (one per SM).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, A);
    if (e != cudaSuccess) return cuda_fail(e, "prefill_kernel (cooperative)");
    return check_launch("prefill_kernel");
}

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
    (void)max_seqlen_k;
    return pa::prefill_impl(out, q, q_row_stride, total_q, k, v, kv_row_stride, total_k, block_tables,
                            max_blocks_per_seq, cu_seqlens_q, cu_seqlens_k, num_seqs, max_seqlen_q, num_q_heads,
                            num_kv_heads, head_dim, block_size, num_blocks, softmax_scale, causal, nullptr, stream);
}

extern "C" size_t pa_prefill_store_workspace_size(void) { return 256; }

extern "C" pa_status pa_prefill_store_varlen(void *out, const void *q, int64_t q_row_stride, int32_t total_q,
                                             const void *new_k, int64_t new_k_row_stride, const void *new_v,
                                             int64_t new_v_row_stride, void *k_cache, void *v_cache,
                                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                                             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                             int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                             int32_t block_size, int32_t num_blocks, float softmax_scale,
                                             int32_t causal, void *workspace, size_t workspace_bytes,
                                             pa_stream_t stream) {
    using namespace pa;
    (void)max_seqlen_k;
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PA_OK;
    if (!block_tables) return fail(PA_ERR_INVALID_ARG, "the fused store needs block_tables (a paged pool)");
    if (!new_k || !new_v) return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_kv_heads <= 0) return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be positive");
    const int64_t row = (int64_t)num_kv_heads * D;
    if (new_k_row_stride < row || new_v_row_stride < row || new_k_row_stride % 8 || new_v_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "new K/V row strides must be >= num_kv_heads*head_dim and multiples of 8");
    if (!aligned16(new_k) || !aligned16(new_v)) return fail(PA_ERR_INVALID_ARG, "new_k/new_v must be 16-byte aligned");
    if (!workspace || workspace_bytes < pa_prefill_store_workspace_size())
        return fail(PA_ERR_WORKSPACE, "workspace missing or smaller than pa_prefill_store_workspace_size()");
    if (reinterpret_cast<uintptr_t>(workspace) % 8) return fail(PA_ERR_INVALID_ARG, "workspace must be 8-byte aligned");
    SuffixStore st{new_k, new_v, new_k_row_stride, new_v_row_stride, static_cast<unsigned *>(workspace)};
    return prefill_impl(out, q, q_row_stride, total_q, k_cache, v_cache, 0, 0, block_tables, max_blocks_per_seq,
                        cu_seqlens_q, cu_seqlens_k, num_seqs, max_seqlen_q, num_q_heads, num_kv_heads, head_dim,
                        block_size, num_blocks, softmax_scale, causal, &st, stream);
}
