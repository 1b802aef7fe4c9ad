// pa_decode.cu -- paged split-KV GQA decode attention for sm_103a.
//
// What it computes [NV12 §12.6 flash_attn_with_kvcache; VD §3]: for each
// sequence b and query head h (kv head g = h / G, G = Hq/Hkv),
//   out[b,h] = softmax_p(scale * q[b,h] . K[slot(b,p), g]) V[slot(b,p), g],
// p < context_lens[b], slot(b,p) = block_tables[b][p/B]*B + p%B [PA3 §3].
//
// How (GB300 design):
//  * Work is a flat list of 64-position tiles ordered (sequence, kv head,
//    tile), cut into one contiguous share per CTA of a persistent grid (one
//    CTA per SM).  The shares are equal in cost, not in tiles: a (sequence,
//    kv head) pair costs 1.5 tiles' worth on top of its tiles (its q rows,
//    block-id fetch and merge), so a CTA whose share holds many short pairs
//    streams fewer tiles.  The first 15/16 of each share is the CTA's own
//    range; the last 1/16 a tail range that CTAs take from an atomic counter
//    once their own range is done, so the CTAs that stream faster absorb the
//    tail.  A range holds whole (sequence, kv head) segments in its middle
//    and at most one part-segment at each end.  Every CTA rebuilds the
//    per-sequence tile counts, their costs and both prefix sums from
//    context_lens in shared memory, then the table of range starts.  Launches
//    with fewer than 16 tiles per CTA are split by tiles alone (closed form),
//    as their time is latency, not their slowest share.
//  * Two producer warps issue TMA tile loads (cp.async.bulk.tensor, 64 rows x
//    256 B per K or V tile; a row is one token of one kv head) into a
//    4-stage shared-memory ring guarded by mbarriers: one warp the K tiles
//    and the segment's G query rows (a bulk copy), the other the V tiles.
//    Split this way, each warp's issue latency is paid in parallel.  The K
//    warp also takes the chunk ranges and hands each range to the other
//    warps through a small ring of tickets.  Tiles never straddle a block:
//    the TMA box is gcd(B, 64) rows, and each box is addressed through the
//    block table, whose entries the producers' lanes prefetch 32 at a time.
//  * K and V tiles land 128-byte swizzled, split into the two 64-dim halves
//    of each row ([half][row][64]; the tensor map views a pool as
//    [kv head][half][slot][64]), so that 8 consecutive rows at one 16-byte
//    column sit in 8 different banks.
//  * Eight consumer warps in two groups of four; tiles alternate between the
//    groups and each warp owns 16 keys of a tile.  Q.K and P.V run on the
//    tensor cores as mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the
//    GQA group's G query rows as the M side (rows G..15 are zero): the whole
//    group shares each K and V byte, operands come by ldmatrix, and the S
//    fragment of Q.K is already the A fragment of P.V.  This is not about
//    tensor throughput (decode moves ~2 flops per byte) but about issue and
//    shared-memory traffic: one MMA replaces 64 FMAs and the scores need no
//    shuffle reduction.  Online softmax in base 2 with a lazy reference max:
//    the running max only moves (rescaling O and l) when a score exceeds it
//    by more than 2^8, which a warp vote detects.
//  * Segment end: a merge warp combines the consumer warps' states.  A whole
//    segment writes bf16 output directly.  A part-segment writes its (m, l, o)
//    partial to the workspace and counts itself on the pair's arrival
//    counter; the CTA whose count completes the pair merges the parts
//    (log-sum-exp) and resets the counter.
//  * Every global read or write comes after griddepcontrol.wait, so the
//    kernel can be launched early behind the kernel that produces its inputs
//    (programmatic dependent launch).
//  * All waits are bounded; a timeout records PA_DEV_TIMEOUT and the warps
//    finish their loops without waiting, keeping every barrier paired.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pa_internal.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int D = 128;
constexpr int ROW_BYTES = D * 2;  // one token row of one kv head
constexpr int TILE = 64;          // rows per pipeline stage
constexpr int WPG = 4;            // consumer warps per group
constexpr int KPW = TILE / WPG;   // keys per consumer warp per tile (one MMA n-pair)
constexpr float kLazyRescale = 8.f;  // log2 headroom before the running max must move
constexpr int kMaxBatch = 2048;
constexpr int kMaxBatchCascade = 1024;   // pa_decode_shared_prefix
constexpr int kMaxPrefixRows = 8192;     // (member, q head) rows with prefix partials in a workspace
constexpr int kPrefixSplits = 2;         // the shared prefix's tiles are cut in this many parts
constexpr int kMaxGrid = 256;     // CTAs of the persistent grid (min(SMs, this))
constexpr int kMaxRanges = 2 * kMaxGrid;  // a head and a tail range per CTA
constexpr int kTailShift = 4;  // a CTA's tail range is 1/16 of its share
// The work is split by cost, not by tiles: a (sequence, kv head) pair costs
// kCostTile per tile plus kCostPair for the work it carries whatever its
// length (its q rows, its block-id fetch, the merge of its result and, for
// a member of a shared prefix, the fold of the prefix partial).
#ifndef PA_PAIR_COST
#define PA_PAIR_COST 6
#endif
constexpr int kCostTile = 4;
constexpr int kCostPair = PA_PAIR_COST;
// Below this many tiles per CTA a launch is bound by latency, not by its
// slowest share, and the pairs cost nothing extra (an even split by tiles).
constexpr int kCostMinTilesPerCta = 16;
constexpr int NTK = 4;            // tickets in flight (ranges handed from the K warp to the others)
constexpr int kMinTilesPerCta = 8;  // grid = min(SMs, tile bound / this)
constexpr unsigned FULL = 0xffffffffu;

template <int G>
struct Cfg {
    static constexpr int NGRP = 2;                 // consumer groups; tiles alternate between them
    static constexpr int NCW = WPG * NGRP;         // consumer warps
    static constexpr int PRODUCER_K = NCW;         // warp that issues the K tile (and q) copies
    static constexpr int PRODUCER_V = NCW + 1;     // warp that issues the V tile copies
    static constexpr int MERGER = NCW + 2;         // warp that finishes segments
    static constexpr int NWARPS = NCW + 3;
    static constexpr int NTHREADS = NWARPS * 32;
    // Tile x of the flat list goes to consumer group x % NGRP, so the split of
    // a segment between the groups (and the summation order) does not depend
    // on which CTA runs it.  Group g uses stages g, g + NGRP, ... in turn,
    // counted by its own tile counter; each full/empty barrier therefore has
    // waiters of one group only and a parity wait can never see a phase two
    // steps old as its own.
    static constexpr int STAGES = 4;
    static_assert(STAGES % NGRP == 0, "a stage must belong to a single consumer group");
    static constexpr int SPG = STAGES / NGRP;  // stages per group
    static_assert(NGRP == 2, "the producers keep one tile counter per group");
    static constexpr int NSLOT = 2;  // merge slots (consumer warps -> merge warp), used round-robin
    static constexpr int STAGE_BYTES = 2 * TILE * ROW_BYTES;
    static constexpr int Q_BYTES = G * ROW_BYTES;
    static constexpr int SLOT_FLOATS = NCW * G * (D + 2);      // o[NCW][G][D], then (m,l)[NCW][G]
    static constexpr int OFF_Q = STAGES * STAGE_BYTES;          // q slots [2][G][D] bf16
    static constexpr int OFF_SLOT = OFF_Q + 2 * Q_BYTES;        // merge slots [NSLOT][SLOT_FLOATS] f32
    static constexpr int OFF_BAR = OFF_SLOT + NSLOT * SLOT_FLOATS * 4;
    // kfull, vfull, empty (the V half), kempty (the K half) [STAGES]; qfull,
    // qempty, done, sfree [2]; tfull, tempty [NTK]
    static constexpr int NBAR = 4 * STAGES + 8 + 2 * NTK;
    static constexpr int OFF_FLAGS = OFF_BAR + NBAR * 8;   // [0]: abort
    static constexpr int OFF_TK = OFF_FLAGS + 16;          // Ticket [NTK]
    static constexpr int OFF_WSUM = OFF_TK + NTK * 32;     // scan scratch [NWARPS] uint32
    // Rows the consumers' ldmatrix reads instead of a tile row: per consumer
    // warp the new token's K and V rows (fused store), then one zero row for
    // keys past the context.  Never written by TMA.
    static constexpr int OFF_SIDE = OFF_WSUM + 64;
    static constexpr int OFF_ZERO = OFF_SIDE + 2 * NCW * ROW_BYTES;
    static constexpr int OFF_RT = OFF_ZERO + ROW_BYTES;    // range starts [2 * kMaxGrid + 1] int64
    static constexpr int OFF_CUM = OFF_RT + (8 * (2 * kMaxGrid + 1) + 15) / 16 * 16;  // per-head tile prefix sum [batch + 1] uint32
    static_assert(OFF_SIDE % 16 == 0 && OFF_ZERO % 16 == 0, "ldmatrix reads these rows: 16-byte aligned");
    static_assert(OFF_Q % 16 == 0 && OFF_SLOT % 16 == 0, "vector accesses: 16-byte aligned");
    __host__ __device__ static constexpr size_t off_ctx(int batch) { return OFF_CUM + 4 * (size_t)(batch + 1); }  // [batch] int
    // With shared prefixes: per sequence its first streamed position and its
    // prefix-partial entry ([batch] int each).
    __host__ __device__ static constexpr size_t off_ps(int batch) { return off_ctx(batch) + 4 * (size_t)batch; }
    __host__ __device__ static constexpr size_t off_pe(int batch) { return off_ps(batch) + 4 * (size_t)batch; }
    __host__ __device__ static constexpr size_t smem_bytes(int batch, bool cascade = false) {
        return (cascade ? off_pe(batch) + 4 * (size_t)batch : off_ps(batch)) + 1024;
    }
    static_assert(smem_bytes(kMaxBatch) <= 232448, "shared memory budget");
    static_assert(smem_bytes(kMaxBatchCascade, true) <= 232448, "shared memory budget (shared prefixes)");
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
    int32_t ctx_limit;  // max_blocks * block_size
    float *ws_o;        // [2 * kMaxRanges][G][D]  partials: slot 2r is range r's first segment, 2r+1 its last
    float2 *ws_ml;      // [2 * kMaxRanges][G]     (m, l) in base 2
    int *ws_cnt;        // [kMaxRanges]            arrivals of the parts of the pair that starts in range r
    int *ws_ctr;        // [2]                     chunk ranges taken, CTAs done taking
    DevError *err;
    int32_t checked;
    // Fused store (pa_decode_store): the new token's K and V rows, patched into
    // the landed tile and written to their slots by the consumer warp that
    // owns the token's key in the sequence's last tile.
    const uint2 *new_k, *new_v;  // null: plain decode
    int64_t new_k_stride, new_v_stride;  // in 8-byte units
    uint2 *k_cache, *v_cache;
    // Shared prefixes (pa_decode_shared_prefix): sequences whose leading full
    // blocks are the same physical blocks stream only their own suffix; the
    // attention over the shared prefix was computed for all of them by the
    // prefix kernel, whose (m, l, o) partial per (member, q head) the merge
    // folds in.
    int32_t cascade;
    int32_t max_prefix_seqs;  // members that get a prefix partial (entries in pfx_*)
    const float *pfx_o;       // [kPrefixSplits][kMaxPrefixRows][D]
    const float2 *pfx_ml;     // [kPrefixSplits][kMaxPrefixRows]  (m, l) in base 2
    int *grp;                 // [2][kMaxBatchCascade]: ps and pe of every sequence, written by the prefix kernel
};

__device__ __forceinline__ int clamp_ctx(const DecodeArgs &a, int b, bool report) {
    int ctx = __ldg(a.ctx_lens + b);
    if (ctx < 0 || ctx > a.ctx_limit) {
        if (report) record_error(a.err, PA_DEV_BAD_CONTEXT, b);
        ctx = ctx < 0 ? 0 : a.ctx_limit;
    }
    return ctx;
}

// The tiles of pair (b, g) are [Hkv*CT_b + g*nt_b, ... + nt_b) in the flat
// list, nt_b = ceil(ctx_b / TILE), CT_b = sum_{b' < b} nt_b'.  The list is
// cut into 2 * grid ranges that follow the flat order: range 2j is CTA j's
// head, 2j+1 its tail, a separate range that any CTA may take from the tail
// counter once its own head range is done (a range may be empty).  The cuts
// divide the list's cost (kCostTile per tile, kCostPair per pair) into equal
// shares, a tail being 1/16 of its CTA's share; st[r] is the first tile of
// range r and st[2 * grid] the number of tiles.
struct Ranges {
    const long long *st;  // null: the closed form below (equal shares of tiles)
    int grid;
    long long base, rem;  // closed form: CTA j's share is base + (j < rem) tiles
    __device__ long long cta_start(int j) const { return (long long)j * base + min((long long)j, rem); }
    __device__ long long cta_len(int j) const { return base + (j < rem ? 1 : 0); }
    __device__ long long start(int r) const {
        if (st) return st[r];
        const int j = r >> 1;
        const long long cl = cta_len(j);
        return cta_start(j) + ((r & 1) ? cl - (cl >> kTailShift) : 0);
    }
    __device__ long long len(int r) const {
        if (st) return st[r + 1] - st[r];
        const long long cl = cta_len(r >> 1);
        return (r & 1) ? (cl >> kTailShift) : cl - (cl >> kTailShift);
    }
    __device__ int owner(long long x) const {  // the (non-empty) range holding tile x
        if (!st) {
            const long long cut = rem * (base + 1);
            const int j = (int)(x < cut ? x / (base + 1) : rem + (x - cut) / base);
            const long long cl = cta_len(j);
            return 2 * j + (x >= cta_start(j) + cl - (cl >> kTailShift) ? 1 : 0);
        }
        int lo = 0, hi = 2 * grid - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (st[mid] <= x) lo = mid; else hi = mid - 1;
        }
        return lo;
    }
};

// A range handed from the K producer warp to the other warps.
struct Ticket {
    long long pos;  // flat index of the first tile
    int len;        // tiles; 0 ends the CTA's work
    int r;          // range index
    int b, g, t;    // (sequence, kv head, tile) of tile pos
    int pad;
};

// One (sequence, kv head) part of a range.
struct Seg {
    int b, g, t_begin, t_end, nt, p_begin, p_end;
    int p0;         // position of the pair's tile 0 (after a shared prefix; 0 otherwise)
    long long pos;  // flat index of tile t_begin
};

// Walks a range segment by segment.  Every role of the CTA runs its own copy
// and sees the same sequence of segments.
struct Walker {
    int b, g, t;
    long long pos, left;
    const int *ps_s;  // per-sequence first streamed position (null: all 0)
    __device__ Walker(const Ticket &k, const int *ps) : b(k.b), g(k.g), t(k.t), pos(k.pos), left(k.len), ps_s(ps) {}
    __device__ bool next(const int *ctx_s, int Hkv, int batch, Seg &s) {
        if (left <= 0) return false;
        const int ctx = ctx_s[b];
        const int p0 = ps_s ? ps_s[b] : 0;
        const int nt = (ctx - p0 + TILE - 1) / TILE;
        const int take = (int)min((long long)(nt - t), left);
        s.b = b;
        s.g = g;
        s.t_begin = t;
        s.t_end = t + take;
        s.nt = nt;
        s.p0 = p0;
        s.p_begin = p0 + t * TILE;
        s.p_end = min(ctx, p0 + s.t_end * TILE);
        s.pos = pos;
        left -= take;
        pos += take;
        t = 0;
        if (++g == Hkv) {
            g = 0;
            do ++b; while (b < batch && ctx_s[b] == 0);
        }
        return true;
    }
};

// Shared prefixes [NV12 §12.8 prefix caching: sequences whose prompts begin
// with the same full blocks hold the same physical blocks, ref_count > 1].
// Sequence b may share its first nfull_b = (ctx_b - 1) / B blocks (every block
// before the one holding its newest token).  Sequences are grouped by the id
// of their first block; the group's leader is its lowest sequence index, and
// its shared length is the longest run of leading block ids on which every
// member agrees with the leader, capped by every member's nfull.  Members of
// groups with two or more sequences and a shared length of at least one block
// get ps[b] = shared blocks * B (the first position they stream themselves)
// and a dense entry index pe[b] (batch order, below max_prefix_seqs); every
// other sequence gets ps = 0, pe = -1.  lead[b] is the leader (or -1) and
// nmem[L] the number of leader L's members that have an entry.
// Every thread of the CTA calls it (it synchronises the CTA).  Scratch:
// (2 * H + batch) ints, H = the smallest power of two >= 2 * batch; lead and
// nmem are [batch] ints outside the scratch.  The result depends only on the
// inputs, not on timing: every CTA and kernel that runs it agrees.
__device__ void find_prefix_groups(int batch, const int32_t *bt, int max_blocks, int block_size,
                                   int max_prefix_seqs, const int *ctx_s, int *ps_s, int *pe_s, int *lead,
                                   int *nmem, int *scr, uint32_t *wsum) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    int H = 64;
    while (H < 2 * batch) H <<= 1;
    int *hkey = scr, *hmin = scr + H, *pmin = scr + 2 * H;  // hash: first block id -> lowest sequence
    for (int i = tid; i < H; i += nthr) {
        hkey[i] = -1;
        hmin[i] = 0x7fffffff;
    }
    for (int b = tid; b < batch; b += nthr) {
        pmin[b] = 0x7fffffff;
        nmem[b] = 0;
    }
    __syncthreads();
    for (int b = tid; b < batch; b += nthr) {
        const int nfull = ctx_s[b] > 0 ? (ctx_s[b] - 1) / block_size : 0;
        const int key = nfull >= 1 ? __ldg(bt + (int64_t)b * max_blocks) : -1;
        lead[b] = -1;
        if (key < 0) continue;  // nothing to share, or a padding id
        uint32_t slot = ((uint32_t)key * 2654435761u) & (uint32_t)(H - 1);
        for (int probe = 0; probe < H; ++probe) {
            const int k = atomicCAS(&hkey[slot], -1, key);
            if (k == -1 || k == key) {
                atomicMin(&hmin[slot], b);
                lead[b] = (int)slot;  // the slot for now; the leader after the next step
                break;
            }
            slot = (slot + 1) & (uint32_t)(H - 1);
        }
    }
    __syncthreads();
    for (int b = tid; b < batch; b += nthr) {
        if (lead[b] < 0) continue;
        const int L = hmin[lead[b]];
        const int nb = (ctx_s[b] - 1) / block_size, nl = (ctx_s[L] - 1) / block_size;
        int j = min(nb, nl);
        if (b != L) {
            // Block 0 agrees by construction; compare four ids per round (loads in flight together).
            const int n = j;
            const int32_t *tb = bt + (int64_t)b * max_blocks, *tl = bt + (int64_t)L * max_blocks;
            for (j = 1; j < n; j += 4) {
                int d = 4;
#pragma unroll
                for (int u = 3; u >= 0; --u)
                    if (j + u < n && __ldg(tb + j + u) != __ldg(tl + j + u)) d = u;
                if (d < 4) {
                    j += d;
                    break;
                }
            }
            j = min(j, n);
        }
        lead[b] = L;
        atomicMin(&pmin[L], j);
    }
    __syncthreads();
    // Membership needs the group's size: count the sequences per leader.
    for (int b = tid; b < batch; b += nthr)
        if (lead[b] >= 0) atomicAdd(&nmem[lead[b]], 1);
    __syncthreads();
    // Dense entries in batch order: a block-wide exclusive scan of the member flags.
    const int per = (batch + nthr - 1) / nthr;
    const int b0 = tid * per, b1 = min(batch, b0 + per);
    auto member = [&](int b) -> bool {
        const int L = lead[b];
        return L >= 0 && nmem[L] >= 2 && pmin[L] >= 1;
    };
    uint32_t run = 0;
    for (int b = b0; b < b1; ++b) run += member(b) ? 1u : 0u;
    uint32_t x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += wsum[w2];
    uint32_t e = before + x - run;
    __syncthreads();
    for (int b = b0; b < b1; ++b) {
        const bool m = member(b) && (int)e < max_prefix_seqs;
        e += member(b) ? 1u : 0u;
        ps_s[b] = m ? pmin[lead[b]] * block_size : 0;
        pe_s[b] = m ? (int)(e - 1) : -1;
    }
    __syncthreads();
    // Entries per leader (the members the prefix kernel computes).
    for (int b = tid; b < batch; b += nthr) nmem[b] = 0;
    __syncthreads();
    for (int b = tid; b < batch; b += nthr)
        if (pe_s[b] >= 0) atomicAdd(&nmem[lead[b]], 1);
    fence_proxy_async_smem();  // the scratch is ring memory that TMA writes next
    __syncthreads();
}

// D += A.B for one m16n8k16 tile: A 16x16 bf16 (row-major fragments),
// B 16x8 bf16 (column fragments), D 16x8 fp32.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 bf16 matrices from shared memory; lanes 8i..8i+7 give the row
// addresses of matrix i.  The .trans form delivers them transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
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

// STORE: the fused store of pa_decode_store (a separate instantiation, so the
// plain decode carries none of it).
template <int G, bool STORE>
__global__ void __launch_bounds__(Cfg<G>::NTHREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
    using C = Cfg<G>;
    extern __shared__ uint8_t smem_raw[];
    // Align to 1 KiB by pointer arithmetic on the __shared__ array, so every
    // pointer below stays in the shared address space (ld/st.shared).
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint32_t *cum = reinterpret_cast<uint32_t *>(smem + C::OFF_CUM);
    int *ctx_s = reinterpret_cast<int *>(smem + C::off_ctx(a.batch));
    int *ps_s = a.cascade ? reinterpret_cast<int *>(smem + C::off_ps(a.batch)) : nullptr;
    int *pe_s = a.cascade ? reinterpret_cast<int *>(smem + C::off_pe(a.batch)) : nullptr;
    uint32_t *wsum = reinterpret_cast<uint32_t *>(smem + C::OFF_WSUM);
    Ticket *tks = reinterpret_cast<Ticket *>(smem + C::OFF_TK);
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *vfull = kfull + C::STAGES;
    uint64_t *empty = vfull + C::STAGES;   // the stage's V half was read
    uint64_t *kempty = empty + C::STAGES;  // the stage's K half was read (after Q.K, before P.V)
    uint64_t *qfull = kempty + C::STAGES;
    uint64_t *qempty = qfull + 2;
    uint64_t *done = qempty + 2;
    uint64_t *sfree = done + 2;
    uint64_t *tfull = sfree + 2;
    uint64_t *tempty = tfull + NTK;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::OFF_FLAGS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&vfull[s], 1);
            mbar_init(&empty[s], WPG);
            mbar_init(&kempty[s], WPG);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&qfull[k], 1);
            mbar_init(&qempty[k], C::NCW);
            mbar_init(&done[k], C::NCW);
            mbar_init(&sfree[k], 1);
        }
        for (int k = 0; k < NTK; ++k) {
            mbar_init(&tfull[k], 1);
            mbar_init(&tempty[k], C::NWARPS - 1);  // every warp but the K producer reads a ticket
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == C::PRODUCER_K && lane == 0) prefetch_tensormap(&tmk);
    if (warp == C::PRODUCER_V && lane == 0) prefetch_tensormap(&tmv);
    // Inputs may come from the kernel this one was launched behind.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (threadIdx.x < ROW_BYTES / 16) st_shared_zero16(smem_addr(smem + C::OFF_ZERO) + 16 * threadIdx.x);
    // Per-sequence tile counts and their exclusive prefix sum, and the same
    // for the sequences' costs (per kv head): each thread takes a run of `per`
    // sequences, then a block-wide scan of the run sums.  The cost sums live
    // in the first ring stage, which no copy writes before the set-up ends.
    unsigned long long *ccum = reinterpret_cast<unsigned long long *>(smem);  // [batch + 1]
    unsigned long long *wsum_c = ccum + kMaxBatch + 1;                         // [NWARPS]
    {
        const int per = (a.batch + C::NTHREADS - 1) / C::NTHREADS;
        const int b0 = threadIdx.x * per, b1 = min(a.batch, b0 + per);
        for (int b = b0; b < b1; ++b) {
            ctx_s[b] = clamp_ctx(a, b, blockIdx.x == 0);
            if (a.cascade) {
                // Shared prefixes: the groups the prefix kernel found (it completed
                // before griddepcontrol.wait returned).
                ps_s[b] = __ldcg(a.grp + b);
                pe_s[b] = __ldcg(a.grp + kMaxBatchCascade + b);
            }
        }
        // Tiles of each sequence: its context after the shared prefix.
        auto ntiles = [&](int b) -> uint32_t {
            return (uint32_t)((ctx_s[b] - (ps_s ? ps_s[b] : 0) + TILE - 1) / TILE);
        };
        auto cost = [&](uint32_t n) -> unsigned long long {
            return n ? (unsigned long long)kCostTile * n + kCostPair : 0ull;
        };
        uint32_t run = 0;
        unsigned long long runc = 0;
        for (int b = b0; b < b1; ++b) {
            const uint32_t n = ntiles(b);
            run += n;
            runc += cost(n);
        }
        uint32_t x = run;
        unsigned long long xc = runc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(FULL, x, o);
            const unsigned long long yc = __shfl_up_sync(FULL, xc, o);
            if (lane >= o) {
                x += y;
                xc += yc;
            }
        }
        if (lane == 31) {
            wsum[warp] = x;
            wsum_c[warp] = xc;
        }
        __syncthreads();
        uint32_t before = 0;
        unsigned long long before_c = 0;
        for (int w2 = 0; w2 < warp; ++w2) {
            before += wsum[w2];
            before_c += wsum_c[w2];
        }
        uint32_t excl = before + x - run;
        unsigned long long excl_c = before_c + xc - runc;
        for (int b = b0; b < b1; ++b) {
            cum[b] = excl;
            ccum[b] = excl_c;
            const uint32_t n = ntiles(b);
            excl += n;
            excl_c += cost(n);
        }
        if (threadIdx.x == C::NTHREADS - 1) {
            cum[a.batch] = before + x;
            ccum[a.batch] = before_c + xc;
        }
    }
    __syncthreads();
    // The range starts: cut the cost into gridDim.x equal shares (the last 1/16
    // of each a tail) and map every cut to the first tile at or after it.  A
    // cut inside a pair's fixed cost goes to the pair's first tile; one inside
    // a tile's cost to the nearer tile boundary.
    long long *rt = reinterpret_cast<long long *>(smem + C::OFF_RT);
    const long long ntot = (long long)a.Hkv * cum[a.batch];
    // Small launches are split by tiles alone, in closed form.
    const bool by_cost = ntot >= (long long)kCostMinTilesPerCta * (long long)gridDim.x;
    if (by_cost) {
        const int grid = (int)gridDim.x;
        const long long ctot = (long long)a.Hkv * (long long)ccum[a.batch];
        // One cut per thread; in 32-bit arithmetic when the costs fit (64-bit
        // division is a long software sequence).
        auto fill = [&](auto zero) {
            using I = decltype(zero);
            const I hkv = (I)a.Hkv, wt = (I)kCostTile, wp = (I)kCostPair;
            const I total = (I)ctot, base = total / (I)grid, rem = total % (I)grid;
            for (int r = threadIdx.x; r <= 2 * grid; r += C::NTHREADS) {
                I xr = total;
                if (r < 2 * grid) {
                    // Share j: base units, one more for the first rem CTAs.
                    const I j = (I)(r >> 1);
                    const I x0 = j * base + (j < rem ? j : rem), len = base + (j < rem ? (I)1 : (I)0);
                    xr = (r & 1) ? x0 + len - (len >> kTailShift) : x0;
                }
                long long pos = ntot;
                if (xr < total) {
                    int lo = 0, hi = a.batch - 1;  // the last sequence whose costs start at or before xr
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (hkv * (I)ccum[mid] <= xr) lo = mid; else hi = mid - 1;
                    }
                    const I nt = (I)(cum[lo + 1] - cum[lo]);
                    const I pc = wt * nt + wp;  // one pair of sequence lo
                    const I rm = xr - hkv * (I)ccum[lo];
                    const I g = rm / pc, r2 = rm - g * pc;
                    I t = 0;
                    if (r2 > wp) {
                        t = (r2 - wp + wt / 2) / wt;
                        if (t > nt) t = nt;
                    }
                    pos = (long long)a.Hkv * cum[lo] + (long long)(g * nt + t);
                }
                rt[r] = pos;
            }
        };
        if (ctot < (1ll << 31)) fill(0u); else fill(0ll);
    }
    fence_proxy_async_smem();  // the ring's first stage is written by TMA from here on
    __syncthreads();
    const Ranges sp{by_cost ? rt : nullptr, (int)gridDim.x, ntot / (long long)gridDim.x, ntot % (long long)gridDim.x};
    // Sequences with no context produce zeros.
    if (warp < C::NCW) {
        for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
            if (ctx_s[b] != 0) continue;
            uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)b * a.Hq * D);
            for (int j = threadIdx.x; j < a.Hq * D / 8; j += C::NCW * 32) o[j] = make_uint4(0, 0, 0, 0);
        }
    }
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Ticket i is read by every warp but the K producer; parities follow i / NTK.
    auto take_ticket = [&](uint32_t i, Ticket &k) -> bool {
        const bool ok = wait_or_abort(&tfull[i % NTK], (i / NTK) & 1, flags, a, 400 + warp);
        k = tks[i % NTK];
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[i % NTK]);
        return ok && k.len > 0;
    };

    // ------------------------------------------------------------------ producers
    // Two warps on different SM sub-partitions: one issues the K tiles (and
    // the segment's q rows), the other the V tiles, each completing on its own
    // barrier of the stage.  Both wait on the stage's empty barrier; neither
    // can fall two phases behind, since a stage is only released again after
    // both of its copies landed.
    if (warp == C::PRODUCER_K || warp == C::PRODUCER_V) {
        const bool isk = warp == C::PRODUCER_K;
        const CUtensorMap *tm = isk ? &tmk : &tmv;
        uint64_t *fullb = isk ? kfull : vfull;
        const uint64_t pol = policy_evict_first();
        uint32_t n0 = 0, n1 = 0, k = 0, kq = 0, ti = 0;  // tiles issued per group, segments, q copies, tickets
        bool ok = true;
        // The K warp's lane 0 picks the ranges: its own head range, then tail
        // ranges from the counter.  The next tail is taken two tiles before
        // the current range ends, so the atomic's latency is hidden.
        int next_tail = -1;
        bool taken = false;
        bool first = true;
        while (ok) {
            Ticket tk;
            if (isk) {
                int r = -1;
                if (lane == 0) {
                    if (first && sp.len(2 * (int)blockIdx.x) > 0) {
                        r = 2 * (int)blockIdx.x;
                    } else {
                        if (!taken) next_tail = atomicAdd(&a.ws_ctr[0], 1);
                        taken = false;
                        while (next_tail < sp.grid && sp.len(2 * next_tail + 1) == 0)
                            next_tail = atomicAdd(&a.ws_ctr[0], 1);
                        if (next_tail < sp.grid) r = 2 * next_tail + 1;
                    }
                    tk.len = 0;
                    tk.r = r;
                    if (r >= 0) {
                        tk.pos = sp.start(r);
                        tk.len = (int)sp.len(r);
                        // Locate tile pos: the last sequence with Hkv * cum[b] <= pos.
                        const uint32_t qv = (uint32_t)(tk.pos / a.Hkv);
                        int lo = 0, hi = a.batch - 1;
                        while (lo < hi) {
                            const int mid = (lo + hi + 1) >> 1;
                            if (cum[mid] <= qv) lo = mid; else hi = mid - 1;
                        }
                        const long long off = tk.pos - (long long)a.Hkv * cum[lo];
                        const int nt = (int)(cum[lo + 1] - cum[lo]);
                        tk.b = lo;
                        tk.g = (int)(off / nt);
                        tk.t = (int)(off % nt);
                    }
                    ok = wait_or_abort(&tempty[ti % NTK], ((ti / NTK) & 1) ^ 1, flags, a, 102);
                    if (ok) {
                        tks[ti % NTK] = tk;
                        mbar_arrive(&tfull[ti % NTK]);  // release: the ticket is visible to its readers
                    }
                }
                first = false;
                ++ti;
                ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                tk.len = __shfl_sync(FULL, tk.len, 0);
                tk.pos = __shfl_sync(FULL, tk.pos, 0);
                tk.b = __shfl_sync(FULL, tk.b, 0);
                tk.g = __shfl_sync(FULL, tk.g, 0);
                tk.t = __shfl_sync(FULL, tk.t, 0);
                if (!ok || tk.len <= 0) break;
            } else {
                const bool got = take_ticket(ti++, tk);
                if (!got) break;
            }
            // Lane l holds the block id of logical block wbase + l of the current
            // segment's sequence; the next segment's first window is fetched while
            // the current one is issued.
            auto fetch = [&](const Seg &s, int lb) -> int {
                const int nblk = (s.p_end - 1) / a.block_size + 1;  // logical blocks of the sequence in use
                return lb + lane < nblk ? __ldg(a.block_tables + (int64_t)s.b * a.max_blocks + lb + lane) : -1;
            };
            Walker w(tk, ps_s);
            int range_left = tk.len;  // tiles of this range not yet issued
            Seg cur, nxt;
            bool have = w.next(ctx_s, a.Hkv, a.batch, cur);
            int wbase = have ? cur.p_begin / a.block_size : 0;
            int win = have ? fetch(cur, wbase) : -1;
            bool have_n = have && w.next(ctx_s, a.Hkv, a.batch, nxt);
            int win_n = have_n ? fetch(nxt, nxt.p_begin / a.block_size) : -1;
            for (; ok && have; ++k) {
                if (isk) {
                    if (lane == 0) {
                        ok = wait_or_abort(&qempty[k & 1], ((k >> 1) & 1) ^ 1, flags, a, 100);
                        if (ok) {
                            mbar_arrive_expect_tx(&qfull[k & 1], G * ROW_BYTES);
                            bulk_load(smem + C::OFF_Q + (k & 1) * C::Q_BYTES,
                                      a.q + (int64_t)cur.b * a.q_row_stride + (int64_t)cur.g * G * D,
                                      G * ROW_BYTES, &qfull[k & 1]);
                            ++kq;
                        }
                    }
                    ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                }
                for (int t = cur.t_begin; ok && t < cur.t_end; ++t) {
                    const int tg = (int)((cur.pos + (t - cur.t_begin)) % C::NGRP);  // consumer group of the tile
                    const uint32_t n = tg ? n1++ : n0++;
                    const int stage = tg + C::NGRP * (int)(n % C::SPG);
                    // Each half of a stage is refilled once the consumers read it: K after
                    // their Q.K, V after their P.V.
                    if (lane == 0)
                        ok = wait_or_abort(isk ? &kempty[stage] : &empty[stage], ((n / C::SPG) & 1) ^ 1, flags, a, 101);
                    ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (isk && lane == 0 && !taken && range_left <= 2) {
                        next_tail = atomicAdd(&a.ws_ctr[0], 1);
                        taken = true;
                    }
                    --range_left;
                    const int p0 = cur.p0 + t * TILE;
                    const int rows = min(TILE, cur.p_end - p0);
                    const int nsub = (rows + a.box_rows - 1) / a.box_rows;
                    if (lane == 0) mbar_arrive_expect_tx(&fullb[stage], (uint32_t)nsub * a.box_rows * ROW_BYTES);
                    uint8_t *dst = smem + stage * C::STAGE_BYTES + (isk ? 0 : TILE * ROW_BYTES);
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int ps = p0 + sub * a.box_rows;
                        const int lb = ps / a.block_size;
                        if (lb - wbase >= 32) {  // warp-uniform; only sequences with > 32 blocks in a segment
                            wbase = lb;
                            win = fetch(cur, lb);
                        }
                        const int blk = __shfl_sync(FULL, win, lb - wbase);
                        if (lane == 0) {
                            if (isk && a.checked && (blk < 0 || blk >= a.num_blocks))
                                record_error(a.err, PA_DEV_BAD_BLOCK, (long long)cur.b * a.max_blocks + lb);
                            long long slot = (long long)blk * a.block_size + ps % a.block_size;
                            // An invalid block id reads as zeros: TMA fills out-of-range boxes.
                            if (blk < 0 || blk >= a.num_blocks) slot = -2LL * a.box_rows;
                            tma_load_4d(dst + sub * a.box_rows * ROW_BYTES, tm, 0, (int)slot, 0, cur.g, &fullb[stage],
                                        pol);
                        }
                    }
                }
                cur = nxt;
                have = have_n;
                win = win_n;
                wbase = have ? cur.p_begin / a.block_size : 0;
                have_n = have && w.next(ctx_s, a.Hkv, a.batch, nxt);
                win_n = have_n ? fetch(nxt, nxt.p_begin / a.block_size) : -1;
            }
        }
        if (isk && lane == 0) {
            // This CTA takes no more tail ranges.  The last CTA to get here
            // resets both counters for the next launch.
            __threadfence();
            if (atomicAdd(&a.ws_ctr[1], 1) == (int)gridDim.x - 1) {
                a.ws_ctr[0] = 0;
                a.ws_ctr[1] = 0;
            }
        }
        if (!ok && lane == 0) {
            // Let the copies already issued land before the CTA's shared memory goes away.
            for (int g2 = 0; g2 < C::NGRP; ++g2) {
                const uint32_t n = g2 ? n1 : n0;
                for (uint32_t j = 0; j < C::SPG && j < n; ++j) {
                    const uint32_t x = n - 1 - j;
                    (void)mbar_wait(&fullb[g2 + C::NGRP * (x % C::SPG)], (x / C::SPG) & 1);
                }
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
        uint32_t k = 0, ti = 0;
        Ticket tk;
        while (take_ticket(ti++, tk)) {
            Walker w(tk, ps_s);
            Seg sg;
            for (int si = 0; w.next(ctx_s, a.Hkv, a.batch, sg); ++si, ++k) {
                const bool ok = wait_or_abort(&done[k % C::NSLOT], (k / C::NSLOT) & 1, flags, a, 300);
                const float *so = slot_base + (k % C::NSLOT) * C::SLOT_FLOATS;
                const float *sml = so + C::NCW * G * D;
                float O[G][4], M[G], L[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    M[h] = -INFINITY;
#pragma unroll
                    for (int w2 = 0; w2 < C::NCW; ++w2) M[h] = fmaxf(M[h], sml[(w2 * G + h) * 2]);
                    L[h] = 0.f;
                    O[h][0] = O[h][1] = O[h][2] = O[h][3] = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < C::NCW; ++w2) {
                        const float f = fast_exp2(sml[(w2 * G + h) * 2] - M[h]);
                        L[h] = fmaf(sml[(w2 * G + h) * 2 + 1], f, L[h]);
                        const float4 v = *reinterpret_cast<const float4 *>(so + (w2 * G + h) * D + 4 * lane);
                        O[h][0] = fmaf(v.x, f, O[h][0]);
                        O[h][1] = fmaf(v.y, f, O[h][1]);
                        O[h][2] = fmaf(v.z, f, O[h][2]);
                        O[h][3] = fmaf(v.w, f, O[h][3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfree[k % C::NSLOT]);
                if (pe_s && sg.t_begin == 0 && pe_s[sg.b] >= 0) {
                    // The pair's first part also carries the attention over the
                    // shared prefix, computed for all members by the prefix kernel.
                    const int64_t row0 = (int64_t)pe_s[sg.b] * a.Hq + (int64_t)sg.g * G;
#pragma unroll
                    for (int sp2 = 0; sp2 < kPrefixSplits; ++sp2)
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const int64_t row = (int64_t)sp2 * kMaxPrefixRows + row0 + h;
                        const float2 ml = __ldcg(a.pfx_ml + row);
                        const float4 po = __ldcg(reinterpret_cast<const float4 *>(a.pfx_o + row * D) + lane);
                        const float mn = fmaxf(M[h], ml.x);
                        const float f0 = M[h] == -INFINITY ? 0.f : fast_exp2(M[h] - mn);
                        const float f1 = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mn);
                        L[h] = fmaf(L[h], f0, ml.y * f1);
                        O[h][0] = fmaf(O[h][0], f0, po.x * f1);
                        O[h][1] = fmaf(O[h][1], f0, po.y * f1);
                        O[h][2] = fmaf(O[h][2], f0, po.z * f1);
                        O[h][3] = fmaf(O[h][3], f0, po.w * f1);
                        M[h] = mn;
                    }
                }
                const int64_t bh0 = (int64_t)sg.b * a.Hq + (int64_t)sg.g * G;  // first q-head row of (b, g)
                if (sg.t_begin == 0 && sg.t_end == sg.nt) {  // the whole pair: final output
                    if (!ok) continue;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float inv = 1.f / L[h];
                        uint2 pk;
                        pk.x = pack_bf16(O[h][0] * inv, O[h][1] * inv);
                        pk.y = pack_bf16(O[h][2] * inv, O[h][3] * inv);
                        *reinterpret_cast<uint2 *>(a.out + (bh0 + h) * D + 4 * lane) = pk;
                    }
                    continue;
                }
                // A part of the pair (only a range's first and last segments can be):
                // write the partial, then count it on the pair's arrival counter.
                const int slot = 2 * tk.r + (si == 0 ? 0 : 1);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    *reinterpret_cast<float4 *>(a.ws_o + ((int64_t)slot * G + h) * D + 4 * lane) =
                        make_float4(O[h][0], O[h][1], O[h][2], O[h][3]);
                    if (lane == 0) a.ws_ml[slot * G + h] = make_float2(M[h], L[h]);
                }
                const long long p0 = sg.pos - sg.t_begin;  // the pair's first tile
                const int r0 = sp.owner(p0), r1 = sp.owner(p0 + sg.nt - 1);
                // The pair's parts: the non-empty ranges r0..r1.
                int nparts = 0;
                for (int r = r0 + lane; r <= r1; r += 32) nparts += sp.len(r) > 0 ? 1 : 0;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) nparts += __shfl_xor_sync(FULL, nparts, off);
                __threadfence();
                __syncwarp();
                int arrived = 0;
                if (lane == 0) arrived = atomicAdd(&a.ws_cnt[r0], 1);
                arrived = __shfl_sync(FULL, arrived, 0);
                if (arrived != nparts - 1) continue;
                // Every part has landed: merge them.  The pair's part in range r0
                // is that range's first segment when the pair starts the range,
                // else its last; in each later range it is the first segment.
                __threadfence();
                const int slot0 = 2 * r0 + (p0 == sp.start(r0) ? 0 : 1);
                auto part_slot = [&](int r) { return r == r0 ? slot0 : 2 * r; };
                // (m, l) of up to 32 ranges at a time, one range per lane.
                float Mx[G], Lx[G], acc[G][4];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    Mx[h] = -INFINITY;
                    Lx[h] = 0.f;
                    acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
                }
                for (int rb = r0; rb <= r1; rb += 32) {
                    const int r = rb + lane;
                    if (r <= r1 && sp.len(r) > 0) {
#pragma unroll
                        for (int h = 0; h < G; ++h) Mx[h] = fmaxf(Mx[h], __ldcg(&a.ws_ml[part_slot(r) * G + h]).x);
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) Mx[h] = fmaxf(Mx[h], __shfl_xor_sync(FULL, Mx[h], off));
                constexpr int PB = G >= 8 ? 1 : 8 / G;  // parts whose loads are in flight together
                for (int rb = r0; rb <= r1; rb += 32) {
                    const int r = rb + lane;
                    const bool valid = r <= r1 && sp.len(r) > 0;
                    float f[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        f[h] = 0.f;
                        if (valid) {
                            const float2 ml = __ldcg(&a.ws_ml[part_slot(r) * G + h]);
                            f[h] = fast_exp2(ml.x - Mx[h]);
                            Lx[h] = fmaf(ml.y, f[h], Lx[h]);
                        }
                    }
                    unsigned mask = __ballot_sync(FULL, valid);
                    while (mask) {
                        int c[PB];
#pragma unroll
                        for (int q = 0; q < PB; ++q) {
                            c[q] = mask ? __ffs(mask) - 1 : -1;
                            mask &= mask - 1;
                        }
                        float4 v[PB][G];
#pragma unroll
                        for (int q = 0; q < PB; ++q)
#pragma unroll
                            for (int h = 0; h < G; ++h)
                                if (c[q] >= 0)
                                    v[q][h] = __ldcg(reinterpret_cast<const float4 *>(
                                                         a.ws_o + ((int64_t)part_slot(rb + c[q]) * G + h) * D) +
                                                     lane);
#pragma unroll
                        for (int q = 0; q < PB; ++q)
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                if (c[q] < 0) continue;
                                const float fc = __shfl_sync(FULL, f[h], c[q]);
                                acc[h][0] = fmaf(v[q][h].x, fc, acc[h][0]);
                                acc[h][1] = fmaf(v[q][h].y, fc, acc[h][1]);
                                acc[h][2] = fmaf(v[q][h].z, fc, acc[h][2]);
                                acc[h][3] = fmaf(v[q][h].w, fc, acc[h][3]);
                            }
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) Lx[h] += __shfl_xor_sync(FULL, Lx[h], off);
                    const float inv = 1.f / Lx[h];
                    uint2 pk;
                    pk.x = pack_bf16(acc[h][0] * inv, acc[h][1] * inv);
                    pk.y = pack_bf16(acc[h][2] * inv, acc[h][3] * inv);
                    *reinterpret_cast<uint2 *>(a.out + (bh0 + h) * D + 4 * lane) = pk;
                }
                if (lane == 0) a.ws_cnt[r0] = 0;  // ready for the next launch
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    // Fragment coordinates (m16n8k16): row g4 of A/C is query head g4 of the
    // group (valid when g4 < G), columns 2*t4, 2*t4+1 (and +8) are keys or
    // dims.  Each warp owns keys [wig*KPW, wig*KPW + 16) of a tile.
    const int grp = warp / WPG, wig = warp % WPG;
    const int g4 = lane >> 2, t4 = lane & 3;
    const bool hvalid = g4 < G;
    const int mi = lane >> 3, r8 = lane & 7;
    // Byte offset of key row k inside a K or V tile region: boxes of box_rows
    // keys, each [2 halves][box_rows][128 B]; 128 B swizzle by (k & 7).
    const int br = a.box_rows;
    auto key_off = [&](int kk) -> uint32_t {
        return (uint32_t)((kk / br) * (br * ROW_BYTES) + (kk % br) * 128);
    };
    const uint32_t half_stride = (uint32_t)br * 128;
    const int qk_key = wig * KPW + (mi >> 1) * 8 + r8;  // tile key whose row this lane addresses in Q.K
    const int pv_key = wig * KPW + (mi & 1) * 8 + r8;   // ... and in P.V
    const uint32_t qk_row = key_off(qk_key);
    const uint32_t pv_row = key_off(pv_key);
    // Unswizzled 256-byte rows outside the tiles (16-byte column c at 16c).
    const uint32_t side_k = smem_addr(smem + C::OFF_SIDE) + 2 * warp * ROW_BYTES;
    const uint32_t side_v = side_k + ROW_BYTES;
    const uint32_t zero_row = smem_addr(smem + C::OFF_ZERO);
    float *slot_base = reinterpret_cast<float *>(smem + C::OFF_SLOT);

    uint32_t qa[8][2];  // A fragments of q: [k step][cols 2*t4.. and 2*t4+8..] of row g4
    float o[16][4];     // O fragments: [dim tile j] rows g4 (and g4+8, unused), dims 8j + 2*t4, +1
    uint32_t nt_mine = 0, k = 0, ti = 0;  // tiles of this warp's group, segments, tickets
    Ticket tk;
    while (take_ticket(ti++, tk)) {
        Walker w(tk, ps_s);
        Seg sg;
        for (; w.next(ctx_s, a.Hkv, a.batch, sg); ++k) {
            if (wait_or_abort(&qfull[k & 1], (k >> 1) & 1, flags, a, 200 + warp)) {
                const uint32_t qrow = smem_addr(smem + C::OFF_Q + (k & 1) * C::Q_BYTES) + g4 * ROW_BYTES + 4 * t4;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    qa[kk][0] = hvalid ? ld_shared_u32(qrow + 32 * kk) : 0u;
                    qa[kk][1] = hvalid ? ld_shared_u32(qrow + 32 * kk + 16) : 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[k & 1]);
            // Fused store: the new token (position ctx-1) is key kn of the
            // sequence's last tile, owned by one warp of one group.  That warp
            // loads its K and V rows now; at that tile it puts them in its side
            // rows, where its ldmatrix reads them in place of the cache's
            // (stale) rows, and writes them to the cache slot.  Nothing in this
            // launch copies that slot, so no proxy fence is needed.
            int st_t = -1, st_kn = 0;
            long long st_slot = 0;
            uint2 st_k = make_uint2(0, 0), st_v = make_uint2(0, 0);
            if (STORE && sg.t_end == sg.nt) {
                const int pn = sg.p_end - 1, tn = (pn - sg.p0) / TILE, kn = (pn - sg.p0) % TILE;
                if ((int)((sg.pos + (tn - sg.t_begin)) % C::NGRP) == grp && kn / KPW == wig) {
                    const int blk = __ldg(a.block_tables + (int64_t)sg.b * a.max_blocks + pn / a.block_size);
                    if (blk >= 0 && blk < a.num_blocks) {  // else the box reads as zeros, as unfused
                        st_t = tn;
                        st_kn = kn;
                        st_slot = (long long)blk * a.block_size + pn % a.block_size;
                        st_k = __ldg(a.new_k + sg.b * a.new_k_stride + sg.g * (D / 4) + lane);
                        st_v = __ldg(a.new_v + sg.b * a.new_v_stride + sg.g * (D / 4) + lane);
                    }
                }
            }
            float m_ref = -INFINITY, l_part = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

            for (int t = sg.t_begin; t < sg.t_end; ++t) {
                if ((int)((sg.pos + (t - sg.t_begin)) % C::NGRP) != grp) continue;
                const uint32_t n = nt_mine++;
                const int stage = grp + C::NGRP * (int)(n % C::SPG);
                const uint32_t ph = (n / C::SPG) & 1;
                if (wait_or_abort(&kfull[stage], ph, flags, a, 210 + warp)) {
                    const uint32_t ks = smem_addr(smem + stage * C::STAGE_BYTES);
                    const uint32_t vs = ks + TILE * ROW_BYTES;
                    const int nvalid = min(TILE, sg.p_end - (sg.p0 + t * TILE));
                    const bool st_here = STORE && t == st_t;
                    if (st_here) {  // lane l holds bytes 8l..8l+7 of each row
                        st_shared_v2(side_k + 8 * lane, st_k);
                        st_shared_v2(side_v + 8 * lane, st_v);
                        a.k_cache[(st_slot * a.Hkv + sg.g) * (D / 4) + lane] = st_k;
                        a.v_cache[(st_slot * a.Hkv + sg.g) * (D / 4) + lane] = st_v;
                        __syncwarp();
                    }
                    const bool k_side = st_here && qk_key == st_kn;
                    // ---- S = Q.K^T for this warp's 16 keys: two n-tiles of 8 keys
                    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    #pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int chunk = 2 * kk + (mi & 1);  // 16-byte column of the row
                        const uint32_t ad =
                            k_side ? side_k + 16 * chunk
                                   : ks + qk_row + (chunk >> 3) * half_stride + ((uint32_t)((chunk & 7) ^ r8) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(ad, b0, b1, b2, b3);
                        mma16816(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                        mma16816(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
                    }
                    // The K half is no longer read: let the K producer refill it now.
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&kempty[stage]);
                    // ---- online softmax (base 2) with a lazy reference max
                    const int key0 = wig * KPW + 2 * t4;
                    float x[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + (e >> 1) * 8 + (e & 1);
                        x[e] = key < nvalid ? sc[e >> 1][e & 1] * a.scale_log2 : -INFINITY;
                    }
                    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                    if (__any_sync(FULL, hvalid && mx > m_ref + kLazyRescale)) {
                        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
                        const float m_new = fmaxf(m_ref, mx);
                        const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m_ref - m_new);
                        l_part *= alpha;
    #pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            o[j][0] *= alpha;
                            o[j][1] *= alpha;
                        }
                        m_ref = m_new;
                    }
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                    float p[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) p[e] = fast_exp2(x[e] - m_use);
                    l_part += (p[0] + p[1]) + (p[2] + p[3]);
                    const uint32_t pa0 = pack_bf16(p[0], p[1]), pa2 = pack_bf16(p[2], p[3]);
                    // ---- O += P.V once the V tile has landed
                    if (wait_or_abort(&vfull[stage], ph, flags, a, 230 + warp)) {
                        // Rows past the context may hold anything (NaN included) and
                        // 0 * NaN is not 0: their lanes read the zero row instead.
                        const bool v_alt = pv_key >= nvalid || (st_here && pv_key == st_kn);
                        const uint32_t v_alt_row = pv_key >= nvalid ? zero_row : side_v;
    #pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const int chunk = j + (mi >> 1);
                            const uint32_t ad =
                                v_alt ? v_alt_row + 16 * chunk
                                      : vs + pv_row + (chunk >> 3) * half_stride + ((uint32_t)((chunk & 7) ^ r8) << 4);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(ad, b0, b1, b2, b3);
                            mma16816(o[j], pa0, 0u, pa2, 0u, b0, b1);
                            mma16816(o[j + 1], pa0, 0u, pa2, 0u, b2, b3);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
            }
            // ---- publish this warp's (m, l, o) for the merge warp
            l_part += __shfl_xor_sync(FULL, l_part, 1);
            l_part += __shfl_xor_sync(FULL, l_part, 2);
            (void)wait_or_abort(&sfree[k % C::NSLOT], ((k / C::NSLOT) & 1) ^ 1, flags, a, 220 + warp);
            float *so = slot_base + (k % C::NSLOT) * C::SLOT_FLOATS;
            if (hvalid) {
                float *row = so + (warp * G + g4) * D + 2 * t4;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<float2 *>(row + 8 * j) = make_float2(o[j][0], o[j][1]);
                if (t4 == 0) {
                    so[C::NCW * G * D + (warp * G + g4) * 2] = m_ref;
                    so[C::NCW * G * D + (warp * G + g4) * 2 + 1] = l_part;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&done[k % C::NSLOT]);
        }
    }
}

// ---------------------------------------------------------------------------
// Prefix kernel (pa_decode_shared_prefix).  For every group of sequences that
// share leading blocks (find_prefix_groups), the attention of all members'
// query heads over the shared prefix, as fp32 (m, l, o) partials that the
// decode kernel's merge folds into each member's result.  A work item is one
// kv head and a chunk of up to 64 query rows (64 / G members with their G
// heads); its CTA reads each K/V tile of the prefix once (TMA, 3-stage ring)
// and each of its 4 consumer warps runs one m16 row tile over every key
// (mma.sync m16n8k16, online softmax in base 2, exact running max).
// ---------------------------------------------------------------------------
// Set-up shared by both prefix kernels (every thread of the CTA calls it):
// context lengths, the groups (CTA 0 also publishes them for the decode
// kernel) and the chunks of `mpi` members per group, numbered in leader
// order (cbase[L] = first chunk of leader L, cbase[batch] = all chunks).
// Returns the number of chunks.
__device__ int prefix_setup(const DecodeArgs &a, int mpi, int *scr, int *ctx_s, int *ps_s, int *pe_s, int *lead,
                            int *nmem, int *cbase, uint32_t *wsum) {
    const int nthr = blockDim.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int b = threadIdx.x; b < a.batch; b += nthr) ctx_s[b] = clamp_ctx(a, b, false);
    __syncthreads();
    find_prefix_groups(a.batch, a.block_tables, a.max_blocks, a.block_size, a.max_prefix_seqs, ctx_s, ps_s, pe_s,
                       lead, nmem, scr, wsum);
    if (blockIdx.x == 0)
        for (int b = threadIdx.x; b < a.batch; b += nthr) {
            a.grp[b] = ps_s[b];
            a.grp[kMaxBatchCascade + b] = pe_s[b];
        }
    // nmem is 0 for sequences that lead no group: a block-wide exclusive scan.
    const int per = (a.batch + nthr - 1) / nthr;
    const int b0 = threadIdx.x * per, b1 = min(a.batch, b0 + per);
    int run = 0;
    for (int b = b0; b < b1; ++b) run += (nmem[b] + mpi - 1) / mpi;
    int x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = (uint32_t)x;
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += (int)wsum[w2];
    int c = before + x - run;
    for (int b = b0; b < b1; ++b) {
        cbase[b] = c;
        c += (nmem[b] + mpi - 1) / mpi;
    }
    if (threadIdx.x == nthr - 1) cbase[a.batch] = before + x;
    __syncthreads();
    return cbase[a.batch];
}

// The group of chunk ci: the last leader whose chunk base is <= ci.
__device__ __forceinline__ int chunk_leader(const int *cbase, int batch, int ci) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cbase[mid] <= ci) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// One warp: the members of leader L that have an entry, in batch order;
// chunk c's `mpi` of them go to mem[0..).  Returns how many (all lanes).
__device__ int chunk_members(int L, int c, int mpi, int batch, const int *lead, const int *pe_s, int *mem) {
    const int lane = threadIdx.x & 31;
    int seen = 0;
    for (int b0 = L; b0 < batch; b0 += 32) {
        const int b = b0 + lane;
        const bool m = b < batch && lead[b] == L && pe_s[b] >= 0;
        const unsigned bal = __ballot_sync(FULL, m);
        const int r = seen + __popc(bal & ((1u << lane) - 1u));
        if (m && r >= c * mpi && r < (c + 1) * mpi) mem[r - c * mpi] = b;
        seen += __popc(bal);
        if (seen >= (c + 1) * mpi) break;
    }
    return min(mpi, seen - c * mpi);
}

constexpr int PFX_WARPS = 4;                       // consumer warps, one m16 row tile each
constexpr int PFX_ROWS = 16 * PFX_WARPS;           // query rows per work item
constexpr int PFX_STAGES = 3;
constexpr int PFX_THREADS = 32 * (PFX_WARPS + 1);  // + the TMA warp (the last)
constexpr int PFX_STAGE_BYTES = 2 * TILE * ROW_BYTES;
constexpr int PFX_OFF_BAR = PFX_STAGES * PFX_STAGE_BYTES;  // full, empty [PFX_STAGES] each
constexpr int PFX_OFF_ZERO = PFX_OFF_BAR + 64;             // one zero row (keys past the prefix)
constexpr int PFX_OFF_MEM = PFX_OFF_ZERO + ROW_BYTES;      // the item's members [PFX_ROWS] int
constexpr int PFX_OFF_WSUM = PFX_OFF_MEM + 4 * PFX_ROWS;   // scan scratch [PFX_THREADS / 32] uint32
constexpr int PFX_OFF_ARR = PFX_OFF_WSUM + 64;             // ctx, ps, pe, lead, nmem, chunk base [batch + 1]
__host__ __device__ constexpr size_t pfx_smem_bytes(int batch) { return PFX_OFF_ARR + 24 * (size_t)(batch + 1) + 1024; }
static_assert(pfx_smem_bytes(kMaxBatchCascade) <= 232448, "prefix kernel shared memory");

template <int G>
__global__ void __launch_bounds__(PFX_THREADS, 1)
    decode_prefix_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const DecodeArgs a, float *pfx_o, float2 *pfx_ml) {
    constexpr int MPI = PFX_ROWS / G;  // members per work item
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + PFX_OFF_BAR);
    uint64_t *empty = full + PFX_STAGES;
    int *mem = reinterpret_cast<int *>(smem + PFX_OFF_MEM);
    uint32_t *wsum = reinterpret_cast<uint32_t *>(smem + PFX_OFF_WSUM);
    int *ctx_s = reinterpret_cast<int *>(smem + PFX_OFF_ARR);
    int *ps_s = ctx_s + (a.batch + 1), *pe_s = ps_s + (a.batch + 1), *lead = pe_s + (a.batch + 1);
    int *nmem = lead + (a.batch + 1), *cbase = nmem + (a.batch + 1);
    __shared__ int s_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == PFX_WARPS;
    if (threadIdx.x == 0) {
        for (int i = 0; i < PFX_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], PFX_WARPS);
        }
        s_flag = 0;
        fence_mbar_init();
    }
    if (producer && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The decode kernel launched behind this one may start its set-up; it
    // reads the partials only after this grid has completed.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x < ROW_BYTES / 16) st_shared_zero16(smem_addr(smem + PFX_OFF_ZERO) + 16 * threadIdx.x);
    const int nchunks =
        prefix_setup(a, MPI, reinterpret_cast<int *>(smem), ctx_s, ps_s, pe_s, lead, nmem, cbase, wsum);
    const int nitems = nchunks * a.Hkv * kPrefixSplits;  // (split, kv head, chunk)
    const uint64_t pol = policy_evict_first();
    uint32_t tc = 0;  // tiles through the ring (every role counts the same)
    bool ok = true;
    for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
        const int split = it / (nchunks * a.Hkv), g = (it / nchunks) % a.Hkv, ci = it % nchunks;
        const int L = chunk_leader(cbase, a.batch, ci);
        const int c = ci - cbase[L];
        __syncthreads();  // the previous item's member list is no longer read
        if (warp == 0) {
            const int n = chunk_members(L, c, MPI, a.batch, lead, pe_s, mem);
            if (lane == 0) s_flag = n;  // members in this chunk
        }
        __syncthreads();
        const int nm = s_flag;
        const int P = ps_s[L];  // shared positions (a multiple of the block size)
        const int ntall = (P + TILE - 1) / TILE;
        // This split's tiles: [t0, t0 + nt) of the prefix (possibly none).
        const int t0 = (int)((int64_t)ntall * split / kPrefixSplits);
        const int nt = (int)((int64_t)ntall * (split + 1) / kPrefixSplits) - t0;
        if (producer) {
            if (lane == 0) {
                for (int t = t0; ok && t < t0 + nt; ++t, ++tc) {
                    const int st = tc % PFX_STAGES;
                    ok = mbar_wait(&empty[st], ((tc / PFX_STAGES) & 1u) ^ 1u);
                    if (!ok) {
                        record_error(a.err, PA_DEV_TIMEOUT, 150);
                        break;
                    }
                    const int p0 = t * TILE, rows = min(TILE, P - p0);
                    const int nsub = (rows + a.box_rows - 1) / a.box_rows;
                    mbar_arrive_expect_tx(&full[st], 2u * nsub * a.box_rows * ROW_BYTES);
                    uint8_t *dst = smem + st * PFX_STAGE_BYTES;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const int ps = p0 + sub * a.box_rows;
                        const int blk = __ldg(a.block_tables + (int64_t)L * a.max_blocks + ps / a.block_size);
                        long long slot = (long long)blk * a.block_size + ps % a.block_size;
                        if (blk < 0 || blk >= a.num_blocks) slot = -2LL * a.box_rows;  // reads as zeros
                        tma_load_4d(dst + sub * a.box_rows * ROW_BYTES, &tmk, 0, (int)slot, 0, g, &full[st], pol);
                        tma_load_4d(dst + TILE * ROW_BYTES + sub * a.box_rows * ROW_BYTES, &tmv, 0, (int)slot, 0, g,
                                    &full[st], pol);
                    }
                }
            }
            tc = __shfl_sync(FULL, tc, 0);
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
            continue;
        }
        // ---- consumer warp: rows 16 * warp + (g4, g4 + 8) of the item
        const int g4 = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
        int rb[2], rh[2];  // member sequence (or -1) and q head of the two rows this thread holds
        for (int i = 0; i < 2; ++i) {
            const int r = 16 * warp + g4 + 8 * i;
            rb[i] = r / G < nm ? mem[r / G] : -1;
            rh[i] = g * G + r % G;
        }
        uint32_t qa[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t *qr = reinterpret_cast<const uint32_t *>(a.q + (int64_t)max(rb[i], 0) * a.q_row_stride +
                                                                       (int64_t)rh[i] * D);
                qa[kk][i] = rb[i] >= 0 ? __ldg(qr + 8 * kk + t4) : 0u;          // cols 16kk + 2t4, +1
                qa[kk][i + 2] = rb[i] >= 0 ? __ldg(qr + 8 * kk + 4 + t4) : 0u;  // cols 16kk + 8 + 2t4, +1
            }
        float o[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        const int br = a.box_rows;
        auto key_off = [&](int kk) -> uint32_t { return (uint32_t)((kk / br) * (br * ROW_BYTES) + (kk % br) * 128); };
        const uint32_t half_stride = (uint32_t)br * 128;
        const uint32_t zero_row = smem_addr(smem + PFX_OFF_ZERO);
        for (int t = t0; t < t0 + nt; ++t, ++tc) {
            const int st = tc % PFX_STAGES;
            if (ok && !mbar_wait(&full[st], (tc / PFX_STAGES) & 1u)) {
                record_error(a.err, PA_DEV_TIMEOUT, 151);
                ok = false;
            }
            ok = __all_sync(FULL, ok);
            if (ok) {
                const uint32_t ks = smem_addr(smem + st * PFX_STAGE_BYTES), vs = ks + TILE * ROW_BYTES;
                const int nvalid = min(TILE, P - t * TILE);
                float sc[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
                for (int kg = 0; kg < 4; ++kg) {  // 16 keys at a time: n-tiles 2kg, 2kg+1
                    const uint32_t krow = key_off(16 * kg + (mi >> 1) * 8 + r8);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int chunk = 2 * kk + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(ks + krow + (chunk >> 3) * half_stride + ((uint32_t)((chunk & 7) ^ r8) << 4), b0, b1, b2,
                                b3);
                        mma16816(sc[2 * kg], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                        mma16816(sc[2 * kg + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                    }
                }
                // Online softmax (base 2) of the two rows; keys past the prefix are masked.
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = 8 * j + 2 * t4 + (e & 1);
                        sc[j][e] = key < nvalid ? sc[j][e] * a.scale_log2 : -INFINITY;
                        mx[e >> 1] = fmaxf(mx[e >> 1], sc[j][e]);
                    }
                float alpha[2], mu[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    mx[i] = fmaxf(mx[i], __shfl_xor_sync(FULL, mx[i], 1));
                    mx[i] = fmaxf(mx[i], __shfl_xor_sync(FULL, mx[i], 2));
                    const float mn = fmaxf(m_run[i], mx[i]);
                    alpha[i] = m_run[i] == -INFINITY ? 0.f : fast_exp2(m_run[i] - mn);
                    m_run[i] = mn;
                    mu[i] = mn == -INFINITY ? 0.f : mn;
                    l_run[i] *= alpha[i];
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    o[j][0] *= alpha[0];
                    o[j][1] *= alpha[0];
                    o[j][2] *= alpha[1];
                    o[j][3] *= alpha[1];
                }
                uint32_t pa[4][4];  // A fragments of P for the 4 16-key steps
#pragma unroll
                for (int kg = 0; kg < 4; ++kg)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const float *v = sc[2 * kg + h2];
                        const float p0 = fast_exp2(v[0] - mu[0]), p1 = fast_exp2(v[1] - mu[0]);
                        const float p2 = fast_exp2(v[2] - mu[1]), p3 = fast_exp2(v[3] - mu[1]);
                        l_run[0] += p0 + p1;
                        l_run[1] += p2 + p3;
                        pa[kg][2 * h2] = pack_bf16(p0, p1);      // row g4
                        pa[kg][2 * h2 + 1] = pack_bf16(p2, p3);  // row g4 + 8
                    }
#pragma unroll
                for (int kg = 0; kg < 4; ++kg) {
                    const int vkey = 16 * kg + (mi & 1) * 8 + r8;
                    const bool zero = vkey >= nvalid;  // stale rows may hold NaN; P is 0 there
                    const uint32_t vrow = key_off(vkey);
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const int chunk = j + (mi >> 1);
                        const uint32_t ad = zero ? zero_row + 16 * chunk
                                                 : vs + vrow + (chunk >> 3) * half_stride +
                                                       ((uint32_t)((chunk & 7) ^ r8) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(ad, b0, b1, b2, b3);
                        mma16816(o[j], pa[kg][0], pa[kg][1], pa[kg][2], pa[kg][3], b0, b1);
                        mma16816(o[j + 1], pa[kg][0], pa[kg][1], pa[kg][2], pa[kg][3], b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (!ok) continue;
        // ---- the rows' partials: (m, l) and unnormalised o
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            l_run[i] += __shfl_xor_sync(FULL, l_run[i], 1);
            l_run[i] += __shfl_xor_sync(FULL, l_run[i], 2);
            if (rb[i] < 0) continue;
            // A split with no tile leaves (-inf, 0, 0): the merge skips it.
            const int64_t row = (int64_t)split * kMaxPrefixRows + (int64_t)pe_s[rb[i]] * a.Hq + rh[i];
            if (t4 == 0) pfx_ml[row] = make_float2(m_run[i], l_run[i]);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<float2 *>(pfx_o + row * D + 8 * j + 2 * t4) = make_float2(o[j][2 * i], o[j][2 * i + 1]);
        }
    }
    if (producer && lane == 0 && !ok) {
        // Let issued copies land before the CTA's shared memory goes away.
        for (uint32_t x = (tc >= (uint32_t)PFX_STAGES ? tc - PFX_STAGES : 0); x < tc; ++x)
            (void)mbar_wait(&full[x % PFX_STAGES], (x / PFX_STAGES) & 1u);
    }
}

// ---------------------------------------------------------------------------
// Prefix kernel on the 5th-generation tensor cores (block sizes that are a
// multiple of 64, so the shared prefix is whole 64-key tiles and a K or V
// tile is one TMA box [2 halves][64 rows][128 B]).  A work item is 128 rows
// -- 128 / G members x the G q heads of one kv head -- against one key
// split of the group's prefix: S = Q.K^T (M = 128, N = 64, K = 128) into one
// of two TMEM buffers, a row-per-thread online softmax (base 2, lazy
// rescaling of O), P written back over S as bf16, O += P.V (P from TMEM).
// Roles: warp 0 loads K and V tiles, warp 1 issues Q.K (and owns TMEM),
// warp 2 issues P.V, warp 3 lists the item's members, warps 4..7 (TMEM lane
// quarters 0..3) load Q, run the softmax and write the (m, l, o) partials.
// ---------------------------------------------------------------------------
constexpr int TCP_THREADS = 256;
constexpr int TCP_W_LOAD = 0, TCP_W_QK = 1, TCP_W_PV = 2, TCP_W_MEM = 3, TCP_W_SOFT = 4;
constexpr int TCP_ROWS = 128;
constexpr int TCP_ST = 3;                               // K/V ring stages
constexpr int TCP_KV = TILE * ROW_BYTES;                // one K or V tile: 16 KiB
constexpr int TCP_QHALF = TCP_ROWS * 128;               // [128 rows][64 dims] of Q
constexpr int TCP_OFF_Q = 0;                            // Q [2 halves][128 rows][128 B]
constexpr int TCP_OFF_K = TCP_OFF_Q + 2 * TCP_QHALF;
constexpr int TCP_OFF_V = TCP_OFF_K + TCP_ST * TCP_KV;
constexpr int TCP_OFF_BAR = TCP_OFF_V + TCP_ST * TCP_KV;
enum {
    T_KFULL = 0, T_KEMPTY = T_KFULL + TCP_ST, T_VFULL = T_KEMPTY + TCP_ST, T_VEMPTY = T_VFULL + TCP_ST,
    T_SFULL = T_VEMPTY + TCP_ST /* [2] */, T_PFULL = T_SFULL + 2 /* [2] */, T_PDONE = T_PFULL + 2 /* [2] */,
    T_QFULL = T_PDONE + 2, T_QEMPTY, T_OEMPTY, T_DRAIN, T_DRAIN2, TCP_NBAR
};
constexpr int TCP_OFF_TMEM = TCP_OFF_BAR + TCP_NBAR * 8;
constexpr int TCP_OFF_FLAGS = TCP_OFF_TMEM + 16;          // [0]: abort, [1]: members in the item
constexpr int TCP_OFF_MEM = TCP_OFF_FLAGS + 16;           // the item's members [TCP_ROWS] int
constexpr int TCP_OFF_WSUM = TCP_OFF_MEM + 4 * TCP_ROWS;  // scan scratch [8] uint32
constexpr int TCP_OFF_ARR = TCP_OFF_WSUM + 64;            // ctx, ps, pe, lead, nmem, chunk base [batch + 1]
__host__ __device__ constexpr size_t tcp_smem_bytes(int batch) { return TCP_OFF_ARR + 24 * (size_t)(batch + 1) + 1024; }
static_assert(tcp_smem_bytes(kMaxBatchCascade) <= 232448, "tcgen05 prefix kernel shared memory");
// The grouping scratch (a hash of 2 * 2048 ints for 1024 sequences, then
// batch ints) lives in the K and V rings before the first copy.
static_assert(4 * (2 * 2048 + kMaxBatchCascade) <= 2 * TCP_ST * TCP_KV, "grouping scratch fits in the rings");
constexpr uint32_t TCP_TMEM_COLS = 256;                   // S [2][64 columns], O [128 columns]
constexpr uint32_t TCP_COL_S = 0, TCP_COL_O = 128;
constexpr uint32_t TCP_SBO = 1024;                        // 8 rows x 128 B between core-matrix groups
constexpr uint32_t TCP_IDESC_S = idesc_bf16_f32(TCP_ROWS, TILE, false, false);  // Q, K both K-major
constexpr uint32_t TCP_IDESC_PV = idesc_bf16_f32(TCP_ROWS, D, false, true);     // P from TMEM, V MN-major

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int G>
__global__ void __launch_bounds__(TCP_THREADS, 1)
    decode_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                            const DecodeArgs a, float *pfx_o, float2 *pfx_ml) {
    constexpr int MPI = TCP_ROWS / G;  // members per work item
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + TCP_OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TCP_OFF_TMEM);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + TCP_OFF_FLAGS);
    int *mem = reinterpret_cast<int *>(smem + TCP_OFF_MEM);
    uint32_t *wsum = reinterpret_cast<uint32_t *>(smem + TCP_OFF_WSUM);
    int *ctx_s = reinterpret_cast<int *>(smem + TCP_OFF_ARR);
    int *ps_s = ctx_s + (a.batch + 1), *pe_s = ps_s + (a.batch + 1), *lead = pe_s + (a.batch + 1);
    int *nmem = lead + (a.batch + 1), *cbase = nmem + (a.batch + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < TCP_NBAR; ++i) {
            const bool per_warp = i == T_PFULL || i == T_PFULL + 1 || i == T_QFULL || i == T_OEMPTY;
            mbar_init(&bar[i], per_warp ? 4u : 1u);  // the four softmax warps arrive one each
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == TCP_W_LOAD && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    if (warp == TCP_W_QK) {
        tmem_alloc(tmem_slot, TCP_TMEM_COLS);
        tmem_relinquish();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The decode kernel launched behind this one may start its set-up; it
    // reads the partials only after this grid has completed.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int nchunks =
        prefix_setup(a, MPI, reinterpret_cast<int *>(smem + TCP_OFF_K), ctx_s, ps_s, pe_s, lead, nmem, cbase, wsum);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nitems = nchunks * a.Hkv * kPrefixSplits;  // (split, kv head, chunk)
    uint32_t tc = 0, ui = 0;  // tiles through the ring, items with tiles (every role counts the same)
    bool ok = true, issued = false;
    uint32_t nk = 0, nv = 0;  // copies issued (loader)
    for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
        const int split = it / (nchunks * a.Hkv), g = (it / nchunks) % a.Hkv, ci = it % nchunks;
        const int L = chunk_leader(cbase, a.batch, ci);
        __syncthreads();  // the previous item's member list is no longer read
        if (warp == TCP_W_MEM) {
            const int n = chunk_members(L, ci - cbase[L], MPI, a.batch, lead, pe_s, mem);
            if (lane == 0) flags[1] = n;
        }
        __syncthreads();
        const int nm = flags[1];
        const int ntall = ps_s[L] / TILE;  // the shared prefix: whole tiles
        const int t0 = (int)((int64_t)ntall * split / kPrefixSplits);
        const int nt = (int)((int64_t)ntall * (split + 1) / kPrefixSplits) - t0;
        if (warp == TCP_W_LOAD) {
            if (lane == 0) {
                for (int j = 0; ok && j < nt; ++j) {
                    const uint32_t gg = tc + j;
                    const int st = gg % TCP_ST;
                    const int p0 = (t0 + j) * TILE;
                    const int blk = __ldg(a.block_tables + (int64_t)L * a.max_blocks + p0 / a.block_size);
                    const int row = (blk < 0 || blk >= a.num_blocks) ? -2 * TILE : blk * a.block_size + p0 % a.block_size;
                    if (!(ok = wait_or_abort(&bar[T_KEMPTY + st], ((gg / TCP_ST) & 1u) ^ 1u, flags, a, 160))) break;
                    mbar_arrive_expect_tx(&bar[T_KFULL + st], TCP_KV);
                    tma_load_4d_plain(smem + TCP_OFF_K + st * TCP_KV, &tmk, 0, row, 0, g, &bar[T_KFULL + st]);
                    ++nk;
                    if (!(ok = wait_or_abort(&bar[T_VEMPTY + st], ((gg / TCP_ST) & 1u) ^ 1u, flags, a, 161))) break;
                    mbar_arrive_expect_tx(&bar[T_VFULL + st], TCP_KV);
                    tma_load_4d_plain(smem + TCP_OFF_V + st * TCP_KV, &tmv, 0, row, 0, g, &bar[T_VFULL + st]);
                    ++nv;
                }
            }
        } else if (warp == TCP_W_QK) {
            if (lane == 0 && nt > 0) {
                ok = ok && wait_or_abort(&bar[T_QFULL], ui & 1u, flags, a, 162);
                tc_fence_after();
                const uint64_t qdesc = smem_desc_sw128(smem_addr(smem + TCP_OFF_Q), 16, TCP_SBO);
                for (int j = 0; ok && j < nt; ++j) {
                    const uint32_t gg = tc + j;
                    const int st = gg % TCP_ST, b = gg & 1;
                    if (!(ok = wait_or_abort(&bar[T_KFULL + st], (gg / TCP_ST) & 1u, flags, a, 163))) break;
                    // S(b) is free once the P.V that read it two tiles ago has completed.
                    if (!(ok = wait_or_abort(&bar[T_PDONE + b], ((gg >> 1) & 1u) ^ 1u, flags, a, 164))) break;
                    tc_fence_after();
                    const uint64_t kdesc = smem_desc_sw128(smem_addr(smem + TCP_OFF_K + st * TCP_KV), 16, TCP_SBO);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t qo = (uint64_t)(((kk >> 2) * TCP_QHALF + (kk & 3) * 32) >> 4);
                        const uint64_t ko = (uint64_t)(((kk >> 2) * (TCP_KV / 2) + (kk & 3) * 32) >> 4);
                        mma_bf16_ss(tmem + TCP_COL_S + b * TILE, qdesc + qo, kdesc + ko, TCP_IDESC_S, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&bar[T_SFULL + b]);
                    mma_commit(&bar[T_KEMPTY + st]);
                    issued = true;
                }
                if (ok) mma_commit(&bar[T_QEMPTY]);  // every Q.K of the item has read Q
            }
        } else if (warp == TCP_W_PV) {
            if (lane == 0 && nt > 0) {
                for (int j = 0; ok && j < nt; ++j) {
                    const uint32_t gg = tc + j;
                    const int st = gg % TCP_ST, b = gg & 1;
                    if (!(ok = wait_or_abort(&bar[T_VFULL + st], (gg / TCP_ST) & 1u, flags, a, 165))) break;
                    // O is free once the previous item's partials were read out of it.
                    if (j == 0 && !(ok = wait_or_abort(&bar[T_OEMPTY], (ui & 1u) ^ 1u, flags, a, 166))) break;
                    if (!(ok = wait_or_abort(&bar[T_PFULL + b], (gg >> 1) & 1u, flags, a, 167))) break;
                    tc_fence_after();
                    const uint64_t vdesc =
                        smem_desc_sw128(smem_addr(smem + TCP_OFF_V + st * TCP_KV), TCP_KV / 2, TCP_SBO);
#pragma unroll
                    for (int kk = 0; kk < TILE / 16; ++kk)  // 16 keys per step = 8 TMEM columns of P
                        mma_bf16_ts(tmem + TCP_COL_O, tmem + TCP_COL_S + b * TILE + kk * 8,
                                    vdesc + (uint64_t)((kk * 16 * 128) >> 4), TCP_IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bar[T_PDONE + b]);
                    mma_commit(&bar[T_VEMPTY + st]);
                    issued = true;
                }
            }
        } else if (warp >= TCP_W_SOFT) {
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;  // item row == TMEM lane
            const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
            const float sl = a.scale_log2;
            const int mrow = row / G, hrow = g * G + row % G;  // member slot and q head of the row
            const int brow = mrow < nm ? mem[mrow] : -1;
            auto wwait = [&](uint64_t *bb, uint32_t parity, int where) -> bool {
                return __all_sync(FULL, wait_or_abort(bb, parity, flags, a, where));
            };
            float m_run = -INFINITY, l_run = 0.f;
            if (nt > 0 && ok) {
                // Q rows of the item (zeros for rows past the members), once the
                // previous item's Q.K products have read the tile.
                if ((ok = wwait(&bar[T_QEMPTY], (ui & 1u) ^ 1u, 170))) {
                    const uint4 *src =
                        reinterpret_cast<const uint4 *>(a.q + (int64_t)max(brow, 0) * a.q_row_stride + (int64_t)hrow * D);
                    const uint32_t qs = smem_addr(smem + TCP_OFF_Q);
                    uint4 v[16];  // all loads in flight before the first store
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = brow >= 0 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        st_shared_u4(qs + (uint32_t)((c >> 3) * TCP_QHALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)),
                                     v[c]);
                    fence_proxy_async_smem();  // the MMA reads Q through the async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[T_QFULL]);
                }
            }
            for (int j = 0; ok && j < nt; ++j) {
                const uint32_t gg = tc + j;
                const int b = gg & 1;
                const uint32_t cs = t_lane + TCP_COL_S + b * TILE;
                if (!(ok = wwait(&bar[T_SFULL + b], (gg >> 1) & 1u, 171))) break;
                tc_fence_after();
                uint32_t r[TILE];
                tmem_ld32(cs, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(cs + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_ld_wait();
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k2 = 0; k2 < TILE / 2; ++k2)
                    m4[k2 & 3] = max3(m4[k2 & 3], __uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1]));
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                // Lazy rescaling: the reference max moves only when a score
                // exceeds it by more than 2^kLazyRescale.
                const bool grow = (mx - m_run) * sl > kLazyRescale;
                const float m_new = grow ? mx : m_run;
                const float alpha = grow ? fast_exp2((m_run - m_new) * sl) : 1.f;
                if (j > 0 && __any_sync(FULL, grow)) {
                    // O must hold P.V up to the previous tile before it is rescaled.
                    if (!(ok = wwait(&bar[T_PDONE + ((gg - 1) & 1)], ((gg - 1) >> 1) & 1u, 172))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + TCP_COL_O + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(t_lane + TCP_COL_O + c * 32, o);
                    }
                }
                l_run *= alpha;
                m_run = m_new;
                const float neg_m = -m_run * sl;
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[TILE / 2];
#pragma unroll
                for (int k2 = 0; k2 < TILE / 2; ++k2) {
                    const float p0 = fast_exp2(fmaf(__uint_as_float(r[2 * k2]), sl, neg_m));
                    const float p1 = fast_exp2(fmaf(__uint_as_float(r[2 * k2 + 1]), sl, neg_m));
                    rs[k2 & 3] += p0 + p1;
                    pk[k2] = pack_bf16(p0, p1);
                }
                tmem_st32(cs, pk);  // P over the first 32 columns of S(b)
                tmem_st_wait();
                l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[T_PFULL + b]);
            }
            // ---- the rows' partials: (m, l) in base 2 and unnormalised o
            if (nt > 0 && ok) {
                const uint32_t gl = tc + nt - 1;  // the item's last tile
                if ((ok = wwait(&bar[T_PDONE + (gl & 1)], (gl >> 1) & 1u, 173))) {
                    tc_fence_after();
                    uint32_t o[D];
                    tmem_ld32(t_lane + TCP_COL_O, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                    tmem_ld32(t_lane + TCP_COL_O + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                    tmem_ld32(t_lane + TCP_COL_O + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[64]));
                    tmem_ld32(t_lane + TCP_COL_O + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[96]));
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[T_OEMPTY]);  // O may be overwritten by the next item
                    // Rows through shared memory (the rings are idle: every tile of
                    // the item was consumed and the next item's copies start after
                    // the item barrier), so that each warp writes whole 512-byte rows.
                    // Staging row r at r * 528 B: 16-byte chunks of consecutive rows
                    // fall in different banks.
                    const uint32_t stg = smem_addr(smem + TCP_OFF_K) + (uint32_t)(quarter * 32) * 528u;
#pragma unroll
                    for (int c = 0; c < D / 4; ++c)
                        st_shared_u4(stg + (uint32_t)lane * 528u + 16u * c, make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
                    const int64_t rg_me =
                        brow >= 0 ? (int64_t)split * kMaxPrefixRows + (int64_t)pe_s[brow] * a.Hq + hrow : -1;
                    if (rg_me >= 0) pfx_ml[rg_me] = make_float2(m_run * sl, l_run);
                    __syncwarp();
                    for (int rr = 0; rr < 32; ++rr) {  // the warp's rows, one at a time
                        const int64_t rg = __shfl_sync(FULL, rg_me, rr);
                        if (rg < 0) continue;
                        uint4 w;
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                                     : "r"(stg + (uint32_t)rr * 528u + 16u * lane));
                        reinterpret_cast<uint4 *>(pfx_o + rg * D)[lane] = w;
                    }
                    fence_proxy_async_smem();  // the next item's copies write this memory
                }
            } else if (nt == 0 && brow >= 0) {
                // A split with no tile leaves (-inf, 0, 0): the merge skips it.
                const int64_t rg = (int64_t)split * kMaxPrefixRows + (int64_t)pe_s[brow] * a.Hq + hrow;
                float4 *dst = reinterpret_cast<float4 *>(pfx_o + rg * D);
                for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                pfx_ml[rg] = make_float2(-INFINITY, 0.f);
            }
        }
        tc += nt;
        if (nt > 0) ++ui;
    }
    // ---- wind-down: nothing in flight may outlive the CTA's shared memory or TMEM
    if (warp == TCP_W_LOAD && lane == 0 && !ok) {
        for (uint32_t x = (nk >= (uint32_t)TCP_ST ? nk - TCP_ST : 0); x < nk; ++x)
            (void)mbar_wait(&bar[T_KFULL + x % TCP_ST], (x / TCP_ST) & 1u);
        for (uint32_t x = (nv >= (uint32_t)TCP_ST ? nv - TCP_ST : 0); x < nv; ++x)
            (void)mbar_wait(&bar[T_VFULL + x % TCP_ST], (x / TCP_ST) & 1u);
    }
    if ((warp == TCP_W_QK || warp == TCP_W_PV) && lane == 0 && flags[0] && issued) {
        uint64_t *dr = &bar[warp == TCP_W_QK ? T_DRAIN : T_DRAIN2];
        mma_commit(dr);
        (void)mbar_wait(dr, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == TCP_W_QK) tmem_dealloc(tmem, TCP_TMEM_COLS);
}

// Per (device, instantiation): the shared-memory attribute has been set.
// Two threads making their first call together may both set it (the call is
// idempotent); the flag itself is an atomic, so there is no data race.
std::atomic<int> g_attr_done[64][8];

template <int G, bool STORE>
pa_status launch(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                 cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int gi = (G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3) + (STORE ? 4 : 0);
    if (dev >= 0 && dev < 64 && !g_attr_done[dev][gi].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(
            decode_kernel<G, STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)std::max(Cfg<G>::smem_bytes(kMaxBatch), Cfg<G>::smem_bytes(kMaxBatchCascade, true)));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_kernel)");
        g_attr_done[dev][gi].store(1, std::memory_order_release);
    }
    // Programmatic dependent launch: the grid may start while the previous
    // kernel on the stream finishes; it reads nothing before griddepcontrol.wait.
    return launch_pdl(decode_kernel<G, STORE>, dim3((unsigned)grid), dim3(Cfg<G>::NTHREADS),
                      Cfg<G>::smem_bytes(a.batch, a.cascade != 0), st, "decode_kernel", tk, tv, a);
}

std::atomic<int> g_pfx_attr_done[64][4];
std::atomic<int> g_tcp_attr_done[64][4];

// The prefix kernel for shared prefixes, launched (programmatic dependent
// launch) right before the decode kernel that folds its partials in.
template <int G>
pa_status launch_prefix(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int sms, cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
    if (dev >= 0 && dev < 64 && !g_pfx_attr_done[dev][gi].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_prefix_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)pfx_smem_bytes(kMaxBatchCascade));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_prefix_kernel)");
        g_pfx_attr_done[dev][gi].store(1, std::memory_order_release);
    }
    // Work items: (key split, kv head, chunk of MPI members of one group); at
    // most batch / 2 groups and batch members.
    auto grid_for = [&](int mpi) {
        const int64_t bound = (int64_t)a.Hkv * kPrefixSplits * ((a.batch + mpi - 1) / mpi + a.batch / 2);
        return (int)std::max<int64_t>(1, std::min<int64_t>(sms, bound));
    };
    if (a.box_rows == TILE) {  // whole 64-key tiles: the tensor-core kernel
        if (dev >= 0 && dev < 64 && !g_tcp_attr_done[dev][gi].load(std::memory_order_acquire)) {
            cudaError_t e = cudaFuncSetAttribute(decode_prefix_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)tcp_smem_bytes(kMaxBatchCascade));
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_prefix_tc_kernel)");
            g_tcp_attr_done[dev][gi].store(1, std::memory_order_release);
        }
        return launch_pdl(decode_prefix_tc_kernel<G>, dim3((unsigned)grid_for(TCP_ROWS / G)), dim3(TCP_THREADS),
                          tcp_smem_bytes(a.batch), st, "decode_prefix_tc_kernel", tk, tv, a,
                          const_cast<float *>(a.pfx_o), const_cast<float2 *>(a.pfx_ml));
    }
    return launch_pdl(decode_prefix_kernel<G>, dim3((unsigned)grid_for(PFX_ROWS / G)), dim3(PFX_THREADS),
                      pfx_smem_bytes(a.batch), st, "decode_prefix_kernel", tk, tv, a, const_cast<float *>(a.pfx_o),
                      const_cast<float2 *>(a.pfx_ml));
}

template <int G>
pa_status launch_g(const DecodeArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int grid, int sms,
                   cudaStream_t st) {
    if (a.cascade) {
        const pa_status s = launch_prefix<G>(a, tk, tv, sms, st);
        if (s != PA_OK) return s;
    }
    return a.new_k ? launch<G, true>(a, tk, tv, grid, st) : launch<G, false>(a, tk, tv, grid, st);
}

// Workspace: the two tail counters and the per-range arrival counters first
// (at offsets that do not depend on the shape, so a workspace can serve calls
// of any GQA group and stays zero-filled there), then (m, l) pairs and fp32
// partials, two slots of G heads per range.
struct WsLayout {
    size_t ctr_off, cnt_off, ml_off, o_off, total;
    size_t grp_off, pfx_ml_off, pfx_o_off, total_prefix;  // pa_decode_shared_prefix: groups and prefix partials
};

WsLayout ws_layout(int G) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t slots = 2 * (size_t)kMaxRanges * G;
    WsLayout L;
    L.ctr_off = 0;
    L.cnt_off = 256;
    L.ml_off = up(L.cnt_off + (size_t)kMaxRanges * sizeof(int));
    L.o_off = up(L.ml_off + slots * sizeof(float2));
    L.total = L.o_off + slots * D * sizeof(float);
    L.grp_off = up(L.total);
    L.pfx_ml_off = up(L.grp_off + 2 * (size_t)kMaxBatchCascade * sizeof(int));
    L.pfx_o_off = up(L.pfx_ml_off + (size_t)kPrefixSplits * kMaxPrefixRows * sizeof(float2));
    L.total_prefix = L.pfx_o_off + (size_t)kPrefixSplits * kMaxPrefixRows * D * sizeof(float);
    return L;
}

}  // namespace
}  // namespace pa

extern "C" {

size_t pa_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
    using namespace pa;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || head_dim != D) return 0;
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return 0;
    return ws_layout(G).total;
}

}  // extern "C"

namespace pa {
namespace {

pa_status decode_impl(void *out, const void *q, int64_t q_row_stride, void *k_cache, void *v_cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int32_t num_blocks, float softmax_scale, void *workspace, size_t workspace_bytes,
                      const void *new_k, int64_t new_k_row_stride, const void *new_v, int64_t new_v_row_stride,
                      pa_stream_t stream, bool cascade = false) {
    if (batch < 0) return fail(PA_ERR_INVALID_ARG, "batch < 0");
    if (batch == 0) return PA_OK;
    if (batch > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "batch %d > %d", batch, kMaxBatch);
    if (cascade && batch > kMaxBatchCascade)
        return fail(PA_ERR_UNSUPPORTED, "batch %d > %d with shared prefixes", batch, kMaxBatchCascade);
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
    // The per-head tile prefix sum is 32-bit: batch * ceil(max_blocks * B / 64) must fit.
    if ((int64_t)batch * (((int64_t)max_blocks_per_seq * block_size + TILE - 1) / TILE) >= 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "batch x block-table capacity too large (%d x %lld tokens)", batch,
                    (long long)max_blocks_per_seq * block_size);
    if (q_row_stride < (int64_t)num_q_heads * D || q_row_stride % 8)
        return fail(PA_ERR_INVALID_ARG, "q_row_stride must be >= num_q_heads*head_dim and a multiple of 8");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "out/q/cache pointers must be 16-byte aligned");
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
        return fail(PA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
    const WsLayout W = ws_layout(G);
    const size_t need = cascade ? W.total_prefix : W.total;
    if (!workspace || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    int box = 64;
    while (block_size % box) box >>= 1;  // gcd(block_size, 64) in {16, 32, 64}
    CUtensorMap tk, tv;
    pa_status st = encode_kv_tensor_map_halves(&tk, k_cache, (int64_t)num_blocks * block_size, num_kv_heads, box);
    if (st != PA_OK) return st;
    st = encode_kv_tensor_map_halves(&tv, v_cache, (int64_t)num_blocks * block_size, num_kv_heads, box);
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
    A.ctx_limit = max_blocks_per_seq * block_size;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    A.ws_ml = reinterpret_cast<float2 *>(ws + W.ml_off);
    A.ws_o = reinterpret_cast<float *>(ws + W.o_off);
    A.ws_cnt = reinterpret_cast<int *>(ws + W.cnt_off);
    A.ws_ctr = reinterpret_cast<int *>(ws + W.ctr_off);
    A.err = device_error_ptr();
    A.checked = checked_mode() ? 1 : 0;
    A.new_k = static_cast<const uint2 *>(new_k);
    A.new_v = static_cast<const uint2 *>(new_v);
    A.new_k_stride = new_k_row_stride / 4;
    A.new_v_stride = new_v_row_stride / 4;
    A.k_cache = static_cast<uint2 *>(k_cache);
    A.v_cache = static_cast<uint2 *>(v_cache);
    A.cascade = cascade ? 1 : 0;
    A.max_prefix_seqs = kMaxPrefixRows / num_q_heads;
    A.pfx_ml = cascade ? reinterpret_cast<const float2 *>(ws + W.pfx_ml_off) : nullptr;
    A.pfx_o = cascade ? reinterpret_cast<const float *>(ws + W.pfx_o_off) : nullptr;
    A.grp = cascade ? reinterpret_cast<int *>(ws + W.grp_off) : nullptr;

    const int sms = std::min(sm_count(), kMaxGrid);
    if (sms <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    // Small batches get fewer CTAs, so that a range still holds several tiles
    // (every range boundary inside a (sequence, kv head) pair costs a partial
    // and a merge).  The bound on the tiles comes from the table width, the
    // only size known on the host.
    const int64_t tiles_bound =
        (int64_t)batch * num_kv_heads * (((int64_t)max_blocks_per_seq * block_size + TILE - 1) / TILE);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (tiles_bound + kMinTilesPerCta - 1) / kMinTilesPerCta));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (G) {
        case 1: return launch_g<1>(A, tk, tv, grid, sms, s);
        case 2: return launch_g<2>(A, tk, tv, grid, sms, s);
        case 4: return launch_g<4>(A, tk, tv, grid, sms, s);
        default: return launch_g<8>(A, tk, tv, grid, sms, s);
    }
}

}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_decode(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                    float softmax_scale, void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    return pa::decode_impl(out, q, q_row_stride, const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                           block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, softmax_scale, workspace, workspace_bytes, nullptr, 0,
                           nullptr, 0, stream);
}

pa_status pa_decode_store(void *out, const void *q, int64_t q_row_stride, const void *new_k,
                          int64_t new_k_row_stride, const void *new_v, int64_t new_v_row_stride, void *k_cache,
                          void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float softmax_scale,
                          void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    using namespace pa;
    if (batch > 0) {
        if (!new_k || !new_v) return fail(PA_ERR_INVALID_ARG, "null new_k/new_v");
        if (!aligned16(new_k) || !aligned16(new_v)) return fail(PA_ERR_INVALID_ARG, "new_k/new_v must be 16-byte aligned");
        const int64_t row = (int64_t)num_kv_heads * D;
        if (new_k_row_stride < row || new_v_row_stride < row || new_k_row_stride % 8 || new_v_row_stride % 8)
            return fail(PA_ERR_INVALID_ARG, "new_k/new_v row strides must be >= num_kv_heads*head_dim and multiples of 8");
    }
    return decode_impl(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, softmax_scale, workspace,
                       workspace_bytes, new_k, new_k_row_stride, new_v, new_v_row_stride, stream);
}

size_t pa_decode_shared_prefix_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
    using namespace pa;
    if (pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim) == 0) return 0;
    return ws_layout(num_q_heads / num_kv_heads).total_prefix;
}

pa_status pa_decode_shared_prefix(void *out, const void *q, int64_t q_row_stride, const void *new_k,
                                  int64_t new_k_row_stride, const void *new_v, int64_t new_v_row_stride, void *k_cache,
                                  void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float softmax_scale, void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    using namespace pa;
    if (batch > 0 && (new_k != nullptr) != (new_v != nullptr))
        return fail(PA_ERR_INVALID_ARG, "new_k and new_v must both be given or both be null");
    if (batch > 0 && new_k) {
        if (!aligned16(new_k) || !aligned16(new_v)) return fail(PA_ERR_INVALID_ARG, "new_k/new_v must be 16-byte aligned");
        const int64_t row = (int64_t)num_kv_heads * D;
        if (new_k_row_stride < row || new_v_row_stride < row || new_k_row_stride % 8 || new_v_row_stride % 8)
            return fail(PA_ERR_INVALID_ARG, "new_k/new_v row strides must be >= num_kv_heads*head_dim and multiples of 8");
    }
    return decode_impl(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, softmax_scale, workspace,
                       workspace_bytes, new_k, new_k_row_stride, new_v, new_v_row_stride, stream, true);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode_static: decode attention for callers that cannot allocate device
// memory.  The split partials live in a fixed scratch array that is part of
// this library's device image instead of a caller-provided workspace.
// ---------------------------------------------------------------------------

// Split-partial scratch, enough for every shape (the workspace size depends
// only on the GQA group).  It is part of the module's device image, so every
// GPU that loads this library holds it until the process exits.  Its leading
// bytes are the work counters the kernel needs at zero when it starts; every
// call clears them first (see pa_decode_static), so no state carries over
// from an earlier call, not even one that stopped on a device error.
static constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char pa_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void *g_static_scratch_addr[64] = {};  // device address of the array, per device

// Device address of the array on the current device (looked up once per
// device, with that device current: the host-side name of a __device__
// variable is not a device address).
pa_status static_scratch(void **out) {
    using namespace pa;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, pa_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(pa_static_scratch)");
        g_static_scratch_addr[dev] = p;
    }
    *out = g_static_scratch_addr[dev];
    return PA_OK;
}
}  // namespace

extern "C" pa_status pa_decode_static(void *out, const void *q, int64_t q_row_stride, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float softmax_scale,
                                      pa_stream_t stream) {
    using namespace pa;
    static_assert(kStaticScratchBytes >= 2 * (size_t)kMaxRanges * 8 * (D * 4 + 8) + kMaxRanges * 4 + 1024,
                  "the static scratch holds the workspace of the largest GQA group");
    const size_t need = pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim);
    if (need == 0 || batch <= 0)  // batch == 0 or arguments pa_decode rejects: let it report
        return pa_decode(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         softmax_scale, nullptr, 0, stream);
    if (need > kStaticScratchBytes)
        return fail(PA_ERR_UNSUPPORTED, "decode scratch of %zu bytes exceeds the static %zu", need,
                    kStaticScratchBytes);
    void *scratch = nullptr;
    pa_status st = static_scratch(&scratch);
    if (st != PA_OK) return st;
    // The tail counter and the per-range arrival counters must be zero when
    // the kernel starts.  A completed call leaves them zero, but a call that
    // stopped on a device error (a wait that ran out) may not, and the caller
    // cannot reach this array to clear it: so clear them here, on the same
    // stream, before every launch (a few KiB; memset allocates nothing).
    const size_t counters = ws_layout(num_q_heads / num_kv_heads).ml_off;
    const cudaError_t e = cudaMemsetAsync(scratch, 0, counters, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static decode counters)");
    return pa_decode(out, q, q_row_stride, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, softmax_scale, scratch,
                     kStaticScratchBytes, stream);
}

extern "C" pa_status pa_decode_static_scratch(void **device_ptr, size_t *bytes) {
    using namespace pa;
    if (!device_ptr || !bytes) return fail(PA_ERR_INVALID_ARG, "null pointer");
    pa_status st = static_scratch(device_ptr);
    if (st != PA_OK) return st;
    *bytes = kStaticScratchBytes;
    return PA_OK;
}
