// The fused shrink -> expand -> add engine behind lora_apply and lora_moe_delta.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 2.3: every segment is a
// shrink X_seg A_i^T followed by an expand with B_i^T added to the base rows,
// and all segments run in one operator instance, spread over the cores;
// section 2.4: tile the token dimension first, then the rank/K dimension so a
// piece of A fits on chip, accumulating the pieces; section 4.2: the
// rank-sized intermediate S accumulates in fp32.
//
// GB300 form.  One persistent grid (one CTA per SM, cooperative launch) walks
// a work list that every CTA derives, identically, from the segment table.
// Each group (an adapter segment, or an (adapter, expert) group of the MoE
// variant) takes one of two paths:
//   * small tiles (at most LORA_OPT_TC_MIN_ROWS rows, decode-sized): up to
//     16 rows, warp-level m16n8k16 MMAs with the tokens as M (tiles of one or
//     two rows expand on CUDA cores).  At these sizes the per-batch
//     issue-to-commit latency of tcgen05 exceeds the whole product, while
//     warp-level MMAs finish in registers;
//   * 128-row tiles (more rows, prefill-sized): tcgen05 with the
//     accumulators in tensor memory.
// Three kinds of work item, in this order on every CTA:
//   1. shrink items (tile, K-chunk): fp32 partial X_tile A_chunk^T to L2
//      scratch, then a release bump of the tile's counter;
//   2. finish items (16 rows of a tile): once every chunk of the tile is in,
//      sum the partials in K order into S (bf16 in the MMA operand layout on
//      the tensor-core path, fp32 otherwise) and bump a second counter;
//   3. expand items (a run of output-column units of one slice of one tile):
//      y = y_base + scale * S B^T.  Small tiles with few expand items skip
//      step 2: their expand items sum the few partials they need themselves.
// Shrink items never wait on other CTAs, finish items wait only on shrink
// items and expand items only on the other two, and the whole grid is
// co-resident, so every wait ends.  Chunk and item sizes are picked per
// launch from the totals: small-tile K-chunks of about a CTA's share of the A
// bytes (as large as a staging slot holds where every CTA runs a long chain of
// them), and expand items of about a third (128-row tiles) or half (small
// tiles) of a CTA's share of the output.  Expand units stream through a
// three-stage ring that runs across item boundaries; the first units are put
// in flight while the shrink work is still running.  Operands move as bulk
// async copies (whole rows of x and y, contiguous runs of the packed table) or
// 2-D TMA tiles on mbarriers; tensor-core results leave as 2-D TMA boxes or
// bulk row stores.  The summation
// order never depends on timing or on which rows share a tile, so the same
// inputs always give the same bits.
//
// For decode-sized batches the segment build can run inside the launch
// (lora_build_and_apply): every CTA sorts the ids itself.  Launches may be
// scheduled while the kernel before them finishes (programmatic dependent
// launch); everything the previous work wrote is read after the wait on it.
//
// Most of a CTA's serial path runs once per launch, and there the size of the
// code, not its instruction count, sets the time: loops that run once stay
// rolled where that does not lengthen a latency chain, and no helper is
// duplicated on that path without a measured reason.
#include "common.cuh"
#include "tc.cuh"

namespace lora {

constexpr int kT = kEngineThreads;
constexpr int kGroupCap = 2048;                 // groups per launch held in shared memory
constexpr int kGroupCache = 128;                // group records and sizes cached in shared memory
constexpr int kRankCache = 512;                 // stored ranks cached in shared memory
constexpr int kPtrCache = 64;                   // groups whose table entries (A, B block, scale) are cached
// shared-memory pool: S at [0, 16K), three expand stages of 50 KB above it (stage 0 on top)
constexpr int kStageBytes = 50 * 1024;
constexpr int kEsDepth = 3;
constexpr int kSBytes = 16 * 1024;
constexpr int kPool = kSBytes + kEsDepth * kStageBytes;
constexpr int kTcShrinkBytes = kPool - kStageBytes;       // the shrink staging leaves expand stage 0 alone
// small tiles (at most 16 rows): warp-level MMAs (m16n8k16), the tile's tokens as M
constexpr int kSmRows = kBgmvRows;              // token rows of a small tile
// two staging slots (the next item's operands land while this one computes), then the cross-warp sums
// (a slot holds the A chunk [kc/8][R][8] at its start and the x rows [rows][kc + 8] right after it)
constexpr int kSmSlotBytes = 55 * 1024;
constexpr int kSmABytes = 40 * 1024;            // A chunk bytes, at most, while the items are about one per CTA
constexpr int kSmXBytes = kSmSlotBytes - kSmABytes;
constexpr int kSmRedOff = 2 * kSmSlotBytes;     // cross-warp sums of the shrink: [3][16][32] fp32 at most
constexpr int kFmaRows = 2;                     // small tiles of at most this many rows expand on CUDA cores
constexpr int kSmMaxUnit = 1024;                // output columns of one small expand unit, at most
constexpr int kSmSStride = kMaxRank + 8;        // bf16 per row of S in shared memory (padded rows)
constexpr int64_t kDirectLoads = 128 * 1024;    // partial loads of a tile's expand items below which they sum them
// tensor-core path
constexpr int kTcRows = 128;                    // MMA M: rows of one tile
constexpr int kTcKc = 512;                      // K elements of one shrink item (at least)
constexpr int kTcStageK = 64;                   // K elements of one shrink pipeline stage
constexpr int kTcCols = 128;                    // output columns of one expand unit (MMA N)
constexpr int kTcMaxDepth = 4;                  // shrink pipeline stages
constexpr int kFinRows = 16;                    // rows of one finish item
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemExpandCol = 256;        // shrink accumulator: [0, R); expand: [256, 384), [384, 512)
constexpr int kTcYOff = 16 * 1024;              // tensor-core stage: B [rp/8][128][8] at 0, y rows after
constexpr int kTcYStride = kTcCols * 2 + 16;    // padded rows: a warp (one row per lane) hits every bank group
constexpr int kItemsPerCta = 3;                 // 128-row tile expand items per CTA the plan aims for
static_assert(kTcYOff + kTcRows * kTcYStride <= kStageBytes, "tensor-core expand stage");
static_assert(kSmRedOff + 3 * 16 * 32 * 4 <= kTcShrinkBytes, "small-tile shrink staging");
static_assert(kSBytes >= (kMaxRank / 8) * kTcRows * 16, "S area");
static_assert(sizeof(EngineParams) % 4 == 0, "parameter mirror");

// trace slots (lora_set_trace)
enum {
    TS_ENTRY = 0, TS_WORKLIST = 1, TS_SH_START = 2, TS_SH_STAGE = 3 /* 8 slots */, TS_SH_MMA_DONE = 11,
    TS_SH_STORED = 12, TS_SH_PUBLISHED = 13, TS_EX_READY = 14, TS_EX_S = 15,
    TS_EX_UNIT = 16 /* 4 units x (landed, written) */, TS_PRO_LOADED = 24, TS_PRO_PLANNED = 25,
    TS_FIN_START = 26, TS_FIN_READY = 27, TS_FIN_DONE = 28, TS_PREFETCHED = 29, TS_SH_COMPUTED = 30,
    TS_EXIT = 31
};

__device__ __forceinline__ int es_off(int st) { return kPool - (st + 1) * kStageBytes; }

// One expand unit sitting in a stage; written by the thread that issued its copies.
struct UnitRec {
    int n0, nw, nrows, kgs, tw, yoff, ystride, tc;
    int run;   // 128-row tile of consecutive rows: y moves as 2-D TMA boxes ([2][128][128 B], 128-byte swizzle)
    float scale;
};

struct Plan {
    int ta;      // target A bytes of one small-tile shrink item
    int ue;      // 128-row tile expand units per item
    int ccol;    // output columns of one small-tile expand item the plan aims for
    int kctc;    // K elements of one tensor-core shrink item
};

struct GroupDims {
    int a, e, rows_off, count, rp, R;
    uint64_t ablk, bblk;   // packed A and B blocks of (a, e) (not filled by the plan's own size pass)
    float scale;
    bool tc, fin;   // 128-row tensor-core tiles (else small tiles); partials finished by finish items
    int tile_rows, rows1, tiles, kc, n_kc, uw, ue, ipt, fins;
    int64_t scratch;   // floats of hand-off scratch: partials, then S of each tile when finished
};

struct ExpandItem {
    int g, tile, s, u0, nu, r0, nrows, sa, tg;
    GroupDims d;
};


struct __align__(1024) EngineSmem {
    __align__(1024) unsigned char pool[kPool];
    uint64_t bar_sh[2];                  // small-tile shrink copies, per staging slot
    uint64_t bar_es[kEsDepth];           // expand stage copies
    uint64_t bar_s;                      // tensor-core expand: S copy
    uint64_t bar_stage[kTcMaxDepth];     // tensor-core shrink stage landed
    uint64_t bar_mma[kTcMaxDepth];       // tensor-core shrink stage consumed by the MMAs
    uint64_t bar_mmae[2];                // tensor-core expand MMAs done, per accumulator buffer
    EngineParams pc;                     // the launch parameters, mirrored (helpers read them from here)
    uint32_t tmem_base;
    int32_t G, flag, x_total;
    int32_t ta, ue, ccol, kctc;          // launch plan (see plan_launch)
    UnitRec unit[kEsDepth];
    int32_t row_dst[kEsDepth][kTcRows];
    float row_w[kEsDepth][kTcRows];
    int32_t row_src[kTcRows];            // (with the build fused in, where every tile is small: the row list)
    int32_t sh_pre[kGroupCap + 1];       // 128-row tile shrink items before group g
    int32_t shs_pre[kGroupCap + 1];      // small-tile shrink items before group g
    int32_t fin_pre[kGroupCap + 1];      // finish items before group g
    int32_t ex_pre[kGroupCap + 1];       // expand items before group g
    int32_t tile_pre[kGroupCap + 1];     // tiles before group g
    int32_t part_pre[kGroupCap + 1];     // scratch floats before group g
    int4 grp[kGroupCache];               // (adapter, expert, rows_off, count) of the first groups
    int4 gdim[kGroupCache];              // their packed sizes under the launch plan (pack_dims)
    int32_t rp_cache[kRankCache];        // stored rank of the first adapters
    uint64_t a_blk[kPtrCache];           // table entries of the first groups, loaded beside the plan
    uint64_t b_blk[kPtrCache];
    float g_scale[kPtrCache];
};

static_assert(sizeof(EngineSmem) <= 227 * 1024, "shared memory per CTA");
size_t engine_smem_bytes(int) { return sizeof(EngineSmem); }



// A group runs on 128-row tcgen05 tiles when it has more than tc_min_rows rows; groups whose A block has
// more than 128 rows switch at half that count, because their small-tile K-chunks (A staging / 2R)
// get short.
__device__ __forceinline__ bool group_on_tc(const EngineParams &p, int count, int R)
{
    return p.path == 2 || (p.path == 0 && count > (R > 128 ? p.tc_min_rows / 2 : p.tc_min_rows));
}

__device__ __forceinline__ int floor_pow2(int v) { return v <= 0 ? 0 : 1 << (31 - __clz(v)); }

// floor(a / b) for 0 <= a < 2^21, b >= 1.  The work-list arithmetic sits on every CTA's critical path,
// where an integer divide by a runtime value is a long instruction sequence; a single-precision
// reciprocal estimate of the quotient is off by less than one half here (relative error under
// 1.5 x 2^-23), so one correction step makes it exact.
__device__ __forceinline__ int qdiv_s(int a, int b)
{
    float rb;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rb) : "f"(__int2float_rn(b)));
    int q = __float2int_rz(__int2float_rn(a) * rb);
    const int r = a - q * b;
    q += r >= b ? 1 : (r < 0 ? -1 : 0);
    return q;
}
__device__ __noinline__ int qdiv_wide(int a, int b) { return a / b; }
// floor(a / b) for any a >= 0 (larger values out of line)
__device__ __forceinline__ int qdiv(int a, int b) { return a < (1 << 21) ? qdiv_s(a, b) : qdiv_wide(a, b); }
// x mod m in [0, m) for any x, m >= 1
__device__ __forceinline__ int pmod(int x, int m)
{
    if (x >= 0) return x - m * qdiv(x, m);
    return x + m * (qdiv(-x - 1, m) + 1);
}
__device__ __forceinline__ int ceil_log2(int v) { return v <= 1 ? 0 : 32 - __clz(v - 1); }

// Output columns of one small-tile expand unit: the widest power of two whose B rows and y rows fit a
// stage (at least 256 at the largest rank; measured faster than narrower units that pipeline more).
__device__ __forceinline__ int sm_unit_width(int rp, int rows1)
{
    return max(kTcCols, min(kSmMaxUnit, floor_pow2(qdiv_s(kStageBytes / 2, rp + rows1))));
}

// Sizes of group g under plan pl, from scratch.
__device__ __forceinline__ GroupDims group_dims_calc(const EngineParams &p, const EngineSmem &sm, int g, const Plan &pl)
{
    GroupDims d;
    const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
    d.a = gr.x;
    d.e = gr.y;
    d.rows_off = gr.z;
    d.count = gr.w;
    d.rp = d.a < kRankCache ? sm.rp_cache[d.a] : p.rpad[d.a];
    d.R = p.n_a * d.rp;
    d.tc = group_on_tc(p, d.count, d.R);
    d.tile_rows = d.tc ? kTcRows : kBgmvRows;
    d.tiles = d.tc ? (d.count + kTcRows - 1) >> 7 : (d.count + kBgmvRows - 1) >> 4;
    d.rows1 = min(d.count, d.tile_rows);
    const int kmax = (p.K + 63) & ~63;
    if (d.tc) {
        d.kc = min(pl.kctc, kmax);
        d.uw = kTcCols;
        d.ue = pl.ue;
    } else {
        // the A chunk and the x rows ([rows][kc + 8]) must fit one staging slot.  Where the chunk target is
        // past two chunks of kSmABytes (each CTA runs a chain of items, one or two in flight) A may fill
        // what the x rows leave of the slot, so the chain has fewer, larger steps; otherwise A stays
        // within kSmABytes, which spreads the about one item per CTA of small batches wider.
        // (ta is clipped below 2^21: any larger target is past the staging cap anyway)
        const int cap = max(64, (pl.ta > 2 * kSmABytes
                                     ? qdiv_s(kSmSlotBytes - 16 * d.rows1, 2 * (d.R + d.rows1))
                                     : min((qdiv_s(kSmXBytes, d.rows1) - 16) / 2, qdiv_s(kSmABytes / 2, d.R))) & ~63);
        const int want = max(64, (qdiv_s(min(pl.ta, (1 << 21) - 1), 2 * d.R) + 63) & ~63);
        d.kc = min(min(cap, kmax), want);
        d.uw = sm_unit_width(d.rp, d.rows1);
        // units per item: about ccol columns whatever the unit width, so that items of narrow-unit (high
        // rank) and wide-unit groups cost about the same
        d.ue = max(1, min(16, (pl.ccol + (d.uw >> 1)) >> ceil_log2(d.uw)));
    }
    d.n_kc = qdiv_s(p.K + d.kc - 1, d.kc);   // K <= 2^20
    const int lw = ceil_log2(d.uw);   // unit widths are powers of two
    int ipt = 0;
    #pragma unroll 1
    for (int s = 0; s < p.n_slices; ++s) {
        const int us = (p.slice_n[s] + d.uw - 1) >> lw;
        ipt += qdiv_s(us + d.ue - 1, d.ue);
    }
    d.ipt = ipt;
    d.fin = d.tc || (int64_t)d.rows1 * d.rp * d.n_kc * ipt > kDirectLoads;
    d.fins = !d.fin ? 0 : (d.tc ? (d.count + kFinRows - 1) / kFinRows : d.tiles);
    d.scratch = (int64_t)d.n_kc * d.count * d.R +
                (!d.fin ? 0 : d.tc ? (int64_t)d.tiles * (kTcRows / 2) * d.R : (int64_t)d.count * d.R);
    return d;
}

// The same for groups past the shared-memory cache (rare: out of line).
__device__ __noinline__ GroupDims group_dims_full(const EngineParams &p, const EngineSmem &sm, int g, const Plan &pl)
{
    GroupDims d = group_dims_calc(p, sm, g, pl);
    d.ablk = p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)];
    d.bblk = p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)];
    d.scale = p.scale[d.a];
    return d;
}

// Packed sizes of a cached group, written by the plan: (kc, flags, ipt, n_kc), flags = log2(uw) |
// ue << 5 | fin << 13 | tc << 14 (ue < 256).
__device__ __forceinline__ int4 pack_dims(const GroupDims &d)
{
    return make_int4(d.kc, ceil_log2(d.uw) | (d.ue << 5) | ((int)d.fin << 13) | ((int)d.tc << 14), d.ipt,
                     d.n_kc);
}

// Sizes of group g under the launch plan: unpacked from shared memory for the first groups.
__device__ __forceinline__ GroupDims group_dims(const EngineParams &p, const EngineSmem &sm, int g, const Plan &pl)
{
    if (g >= kGroupCache) return group_dims_full(p, sm, g, pl);
    GroupDims d;
    const int4 gr = sm.grp[g];
    const int4 gd = sm.gdim[g];
    d.a = gr.x;
    d.e = gr.y;
    d.rows_off = gr.z;
    d.count = gr.w;
    d.rp = d.a < kRankCache ? sm.rp_cache[d.a] : p.rpad[d.a];
    d.R = p.n_a * d.rp;
    d.kc = gd.x;
    d.uw = 1 << (gd.y & 31);
    d.ue = (gd.y >> 5) & 255;
    d.fin = (gd.y >> 13) & 1;
    d.tc = (gd.y >> 14) & 1;
    d.ipt = gd.z;
    d.n_kc = gd.w;
    if (g < kPtrCache) {
        d.ablk = sm.a_blk[g];
        d.bblk = sm.b_blk[g];
        d.scale = sm.g_scale[g];
    } else {
        d.ablk = p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)];
        d.bblk = p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)];
        d.scale = p.scale[d.a];
    }
    d.tile_rows = d.tc ? kTcRows : kBgmvRows;
    d.tiles = (d.count + d.tile_rows - 1) >> (d.tc ? 7 : 4);
    d.rows1 = min(d.count, d.tile_rows);
    d.fins = !d.fin ? 0 : (d.tc ? (d.count + kFinRows - 1) >> 4 : d.tiles);
    d.scratch = 0;   // only the plan needs it
    return d;
}

__device__ __forceinline__ int find_group(const int32_t *pre, int G, int item)
{
    int lo = 0, hi = G;   // pre[lo] <= item < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= item) lo = mid; else hi = mid;
    }
    return lo;
}

// Every thread waits on the mbarrier (so each observes the copied bytes); the
// CTA proceeds only if all of them saw the phase complete in time.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, const EngineParams &p)
{
    const bool ok = mbar_wait_bounded(bar, parity, p.timeout_ns, p.err);
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// Release: makes every write this CTA made before the last __syncthreads
// visible at GPU scope, then bumps the counter.
__device__ __forceinline__ void release_add(int32_t *ctr, int v)
{
    asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// Thread 0 waits (bounded) until *ctr >= target (acquire); returns false on timeout.
__device__ __noinline__ bool wait_counter(const int32_t *ctr, int target, const EngineParams &p)
{
    if (ld_acquire_gpu(ctr) >= target) return true;
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(ctr) < target) {
        if (globaltimer() - t0 > p.timeout_ns) {
            atomicOr(p.err, kErrTimeout);
            return false;
        }
        nanosleep_ns(32);
    }
    return true;
}

// Phase stamps for lora_set_trace (slot k of this block).
__device__ __forceinline__ void stamp(const EngineParams &p, int k)
{
    if (p.trace != nullptr && threadIdx.x == 0 && (int)blockIdx.x < p.trace_ctas)
        p.trace[(size_t)blockIdx.x * kTraceSlots + k] = globaltimer();
}

// mbarrier phase parities kept in one register per thread
struct Phases {
    uint32_t bits;
    __device__ __forceinline__ uint32_t get(int b) const { return (bits >> b) & 1u; }
    __device__ __forceinline__ void flip(int b) { bits ^= 1u << b; }
};
enum { PH_SHRINK = 0, PH_ES = 1 /* 3 bits */, PH_S = 4, PH_STAGE = 5 /* 4 bits */, PH_MMA = 9 /* 4 bits */,
       PH_MMAE = 13 /* 2 bits */, PH_SHRINK1 = 15 };
__device__ __forceinline__ int ph_shrink(int slot) { return slot ? PH_SHRINK1 : PH_SHRINK; }

// ===========================================================================
// shrink items, small tiles (at most 16 rows)
// ===========================================================================
struct BgShrink {
    int r0, nrows, k0, kw;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x1(uint32_t addr, uint32_t &r0)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];" : "=r"(r0) : "r"(addr));
}
// D[16][8] += A[16][16] B[16][8] (bf16 in, fp32 accumulate), warp-wide
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D[16][8] += A[16][8] B[8][8]
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ BgShrink sm_shrink_desc(const EngineParams &p, const GroupDims &d, int tile, int chunk)
{
    BgShrink b;
    b.r0 = tile * kSmRows;
    b.nrows = min(kSmRows, d.count - b.r0);
    b.k0 = chunk * d.kc;
    b.kw = min(d.kc, p.K - b.k0);
    return b;
}

// Put the item's A chunk ([kw/8][R][8], one run of the packed table) and its
// x rows (one bulk copy per row into padded rows of kc + 8 elements) in flight
// into staging slot `slot`, on bar_sh[slot].
__device__ __forceinline__ void sm_shrink_issue(const EngineParams &p, EngineSmem &sm, const GroupDims &d,
                                                const BgShrink &b, int slot)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned char *base = sm.pool + slot * kSmSlotBytes;
    uint64_t *bar = &sm.bar_sh[slot];
    const uint32_t x_bytes = (uint32_t)b.kw * 2;
    if (tid == 0) {
        const __nv_bfloat16 *ablk = reinterpret_cast<const __nv_bfloat16 *>(d.ablk);
        const uint32_t a_bytes = (uint32_t)(b.kw / 8) * d.R * 16;
        mbar_arrive_expect_tx(bar, a_bytes + b.nrows * x_bytes);
        bulk_g2s(base, ablk + (int64_t)(b.k0 / 8) * d.R * 8, a_bytes, bar);
    }
    if (warp == 1 && lane < b.nrows) {
        const int v = p.rows[d.rows_off + b.r0 + lane], src = p.src_div == 1 ? v : qdiv_s(v, p.src_div);
        bulk_g2s(base + (size_t)d.kc * d.R * 2 + (size_t)lane * (d.kc * 2 + 16), p.x + (int64_t)src * p.ldx + b.k0,
                 x_bytes, bar);
    }
}

// Form the fp32 partial X_rows A_chunk^T (operands in place) with
// m16n8k16 MMAs (rows past the tile read row 0; their results are dropped).
// Warp w takes 8-column tiles of the partial; when there are fewer than
// eight tiles, the warps of a tile split K and meet in shared memory in a
// fixed order.  Each warp keeps four accumulators (K steps in fours) and adds
// them at the end, so the summation order is fixed by the sizes alone.
__device__ __forceinline__ bool sm_shrink_wait(const EngineParams &p, EngineSmem &sm, Phases &ph, int slot, bool first)
{
    if (!cta_wait(&sm.bar_sh[slot], ph.get(ph_shrink(slot)), p)) return false;
    ph.flip(ph_shrink(slot));
    if (first) stamp(p, TS_SH_STAGE);
    return true;
}

__device__ __forceinline__ void sm_shrink_run(const EngineParams &p, EngineSmem &sm, const GroupDims &d,
                                              const BgShrink &b, int g, int chunk, int slot, bool first)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = d.R;
    const int ntiles = R / 8;
    const int nw8 = min(ntiles, 8);                     // warps per K slice
    const int ksplit = ntiles >= 8 ? 1 : qdiv_s(8, ntiles);
    const int kgs = b.kw / 8, steps = (kgs + 1) / 2;
    const int xstride = d.kc * 2 + 16;
    const uint32_t a_base = smem_u32(sm.pool + slot * kSmSlotBytes);
    const int xrow = (lane & 15) < b.nrows ? (lane & 15) : 0;
    const uint32_t x_base = a_base + d.kc * R * 2 + xrow * xstride;
    float *red = reinterpret_cast<float *>(sm.pool + kSmRedOff);   // [ksplit - 1][16][R]
    float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * b.r0 * R + (int64_t)chunk * b.nrows * R;
    const int gr = lane >> 2, qc = (lane & 3) * 2;
    const int kpart = qdiv_s(warp, nw8);
    const int s_lo = qdiv_s(steps * kpart, ksplit), s_hi = qdiv_s(steps * (kpart + 1), ksplit);
    for (int nt0 = 0; nt0 < ntiles; nt0 += 8) {   // uniform: every warp runs the same number of rounds
        const int nt = nt0 + warp - kpart * nw8;
        const bool act = nt < ntiles && kpart < ksplit;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        float d2[4] = {0.f, 0.f, 0.f, 0.f}, d3[4] = {0.f, 0.f, 0.f, 0.f};
        if (act) {
            const uint32_t a_row = a_base + (nt * 8 + (lane & 7)) * 16;
            auto full_step = [&](int st, float (&d)[4]) {
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x4(x_base + (2 * st + (lane >> 4)) * 16, a0, a1, a2, a3);
                ldsm_x2(a_row + (2 * st + ((lane >> 3) & 1)) * R * 16, b0, b1);
                mma16816(d, a0, a1, a2, a3, b0, b1);
            };
            // four independent accumulators over K steps st, st + 1, st + 2, st + 3
            const int full_hi = min(s_hi, kgs / 2);   // steps with both of their K-groups present
            int st = s_lo;
            for (; st + 3 < full_hi; st += 4) {
                full_step(st, d0);
                full_step(st + 1, d1);
                full_step(st + 2, d2);
                full_step(st + 3, d3);
            }
            for (; st < full_hi; ++st) full_step(st, d0);
            if (s_hi > full_hi && full_hi >= s_lo) {   // a last odd K-group: one k8 step
                uint32_t a0, a1, b0;
                ldsm_x2(x_base + (2 * full_hi) * 16, a0, a1);
                ldsm_x1(a_row + (2 * full_hi) * R * 16, b0);
                mma1688(d0, a0, a1, b0);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) d0[q] += (d1[q] + d2[q]) + d3[q];
        const int col = nt * 8 + qc;
        if (ksplit > 1) {   // K slices 1.. hand their sums to slice 0
            if (act && kpart > 0) {
                float *rr = red + (size_t)(kpart - 1) * kSmRows * R;
                rr[gr * R + col] = d0[0];
                rr[gr * R + col + 1] = d0[1];
                rr[(gr + 8) * R + col] = d0[2];
                rr[(gr + 8) * R + col + 1] = d0[3];
            }
            __syncthreads();
            if (act && kpart == 0) {
                for (int k = 0; k < ksplit - 1; ++k) {
                    const float *rr = red + (size_t)k * kSmRows * R;
                    d0[0] += rr[gr * R + col];
                    d0[1] += rr[gr * R + col + 1];
                    d0[2] += rr[(gr + 8) * R + col];
                    d0[3] += rr[(gr + 8) * R + col + 1];
                }
            }
            __syncthreads();
        }
        if (act && kpart == 0) {
            if (gr < b.nrows) *reinterpret_cast<float2 *>(dst + gr * R + col) = make_float2(d0[0], d0[1]);
            if (gr + 8 < b.nrows) *reinterpret_cast<float2 *>(dst + (gr + 8) * R + col) = make_float2(d0[2], d0[3]);
        }
    }
    if (first) stamp(p, TS_SH_COMPUTED);
    __syncthreads();
}

// ===========================================================================
// shrink items, tensor-core path
// ===========================================================================
__device__ __forceinline__ int tc_stage_bytes(int R) { return kTcRows * kTcStageK * 2 + R * kTcStageK * 2; }

struct TcShrink {
    int r0, nrows, k0, kw, nst, depth;
    bool run;
};

// Put one shrink pipeline stage in flight: 128 token rows x 64 K in the
// 128-byte swizzled K-major layout, and the matching A chunk (one bulk copy).
// When the tile's rows are one run of consecutive rows of x with the whole
// 128-row box inside x, a single TMA tile load brings them; otherwise every
// thread gathers 16-byte pieces with cp.async into the same swizzled places
// (zero for rows past the tile or columns past K).
__device__ __noinline__ void tc_issue_stage(const EngineParams &p, const CUtensorMap *xmap, EngineSmem &sm,
                                            uint64_t ablk_addr, int R, int nrows, int k0, int kw, int depth, int run,
                                            int s)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = s - depth * qdiv_s(s, depth);
    unsigned char *Xs = sm.pool + slot * tc_stage_bytes(R);
    unsigned char *As = Xs + kTcRows * kTcStageK * 2;
    const int kb = k0 + s * kTcStageK;
    const int vkg = min(8, (kw - s * kTcStageK) / 8);       // K-groups of 8 present in this stage
    const int need = ((vkg + 1) / 2) * 2;                   // K-groups the MMAs read (whole K=16 steps)
    if (vkg < need) {   // odd K-group count at the end of K: the last A K-group reads as zero
        uint4 *z = reinterpret_cast<uint4 *>(As + vkg * R * 16);
        for (int i = tid; i < R; i += kT) z[i] = make_uint4(0u, 0u, 0u, 0u);
        tc::fence_proxy_async_smem();
    }
    if (!run) {
        // thread (warp, lane): rows 16 warp + (lane & 15), 16-byte chunks 2q + (lane >> 4)
        const int row = warp * 16 + (lane & 15);
        const __nv_bfloat16 *xrow = p.x + (int64_t)sm.row_src[row] * p.ldx + kb;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = 2 * q + (lane >> 4);
            if (c < need) {
                const bool valid = row < nrows && c < vkg;
                tc::cp_async16(Xs + row * 128 + ((c ^ (row & 7)) * 16),
                               valid ? (const void *)(xrow + c * 8) : (const void *)p.x, valid);
            }
        }
        tc::cp_async_commit();
    }
    if (tid == 0) {
        const __nv_bfloat16 *ablk = reinterpret_cast<const __nv_bfloat16 *>(ablk_addr);
        const uint32_t bytes = (uint32_t)vkg * R * 16;
        mbar_arrive_expect_tx(&sm.bar_stage[slot], bytes + (run ? kTcRows * kTcStageK * 2 : 0));
        bulk_g2s(As, ablk + (int64_t)(kb / 8) * R * 8, bytes, &sm.bar_stage[slot]);
        if (run) tc::tma_tile2d(Xs, xmap, kb, sm.row_src[0], &sm.bar_stage[slot]);
    }
}

__device__ __forceinline__ void cp_wait_pending(int pending)
{
    if (pending <= 0) tc::cp_async_wait<0>();
    else if (pending == 1) tc::cp_async_wait<1>();
    else if (pending == 2) tc::cp_async_wait<2>();
    else tc::cp_async_wait<3>();
}

// Record the tile's source rows, decide between TMA runs and gathers, and put
// the first pipeline stages in flight.
__device__ __forceinline__ TcShrink tc_shrink_issue(const EngineParams &p, const CUtensorMap *xmap, EngineSmem &sm,
                                                    const GroupDims &d, int tile, int chunk)
{
    TcShrink t;
    const int tid = threadIdx.x;
    t.r0 = tile * kTcRows;
    t.nrows = min(kTcRows, d.count - t.r0);
    t.k0 = chunk * d.kc;
    t.kw = min(d.kc, p.K - t.k0);
    t.nst = (t.kw + kTcStageK - 1) / kTcStageK;
    t.depth = min(min(kTcMaxDepth, qdiv_s(kTcShrinkBytes, tc_stage_bytes(d.R))), t.nst);
    int my_row = 0;
    if (tid < kTcRows) {
        const int v = tid < t.nrows ? p.rows[d.rows_off + t.r0 + tid] : 0;
        my_row = p.src_div == 1 ? v : qdiv_s(v, p.src_div);
        sm.row_src[tid] = my_row;
    }
    __syncthreads();
    // one TMA tile per stage when the rows are one run of consecutive rows and the 128-row box stays inside x
    const int x_total = sm.x_total;
    const bool consecutive = tid >= t.nrows || my_row == sm.row_src[0] + tid;
    t.run = __syncthreads_and(consecutive ? 1 : 0) != 0 && p.x_rows > 0 && sm.row_src[0] + kTcRows <= x_total;
    for (int s = 0; s < t.depth; ++s) tc_issue_stage(p, xmap, sm, d.ablk, d.R, t.nrows, t.k0, t.kw, t.depth, t.run, s);
    return t;
}

// The MMA loop of a tensor-core shrink item (partial = X_rows[:, K-chunk]
// A[:, K-chunk]^T into tensor memory), then the partial out to the tile's
// scratch slot.  A stage is refilled one iteration after its MMAs were
// issued.  Returns false if a wait ran out.
__device__ __forceinline__ bool tc_shrink_run(const EngineParams &p, const CUtensorMap *xmap, EngineSmem &sm,
                                              const GroupDims &d, const TcShrink &t, int g,
                              int chunk, Phases &ph, bool first)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t idesc = tc::idesc_bf16(kTcRows, d.R);
    uint32_t pending = 0;   // slots whose MMA commit has not been waited for
    bool ok = true;
    for (int s = 0; s < t.nst && ok; ++s) {
        const int slot = s - t.depth * qdiv_s(s, t.depth);
        if (s >= 1 && s - 1 + t.depth < t.nst) {   // refill the previous stage's slot
            const int ps = (s - 1) - t.depth * qdiv_s(s - 1, t.depth);
            ok = cta_wait(&sm.bar_mma[ps], ph.get(PH_MMA + ps), p);
            ph.flip(PH_MMA + ps);
            pending &= ~(1u << ps);
            if (!ok) break;
            tc_issue_stage(p, xmap, sm, d.ablk, d.R, t.nrows, t.k0, t.kw, t.depth, t.run, s - 1 + t.depth);
        }
        if (!t.run) {
            cp_wait_pending(min(t.nst, s + t.depth) - (s + 1));
            tc::fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            const bool landed = mbar_wait_bounded(&sm.bar_stage[slot], ph.get(PH_STAGE + slot), p.timeout_ns, p.err);
            sm.flag = landed ? 1 : 0;
            if (landed) {
                tc::fence_after_sync();
                const unsigned char *Xs = sm.pool + slot * tc_stage_bytes(d.R);
                const unsigned char *As = Xs + kTcRows * kTcStageK * 2;
                const int vkg = min(8, (t.kw - s * kTcStageK) / 8);
                const int steps = (vkg + 1) / 2;
                for (int j = 0; j < steps; ++j) {
                    const uint64_t ad = tc::smem_desc_sw128(smem_u32(Xs) + j * 32);
                    const uint64_t bd = tc::smem_desc(smem_u32(As) + j * 2 * d.R * 16, d.R * 16, 128);
                    tc::mma_bf16(sm.tmem_base, ad, bd, idesc, (s > 0 || j > 0) ? 1u : 0u);
                }
                tc::mma_commit(&sm.bar_mma[slot]);
                if (first && s < 8) stamp(p, TS_SH_STAGE + s);
            }
        }
        ph.flip(PH_STAGE + slot);
        __syncthreads();
        ok = sm.flag != 0;
        if (ok) pending |= 1u << slot;
    }
    // commits complete in order: retire every outstanding one
    for (int slot = 0; slot < kTcMaxDepth; ++slot) {
        if (pending & (1u << slot)) {
            const bool done = cta_wait(&sm.bar_mma[slot], ph.get(PH_MMA + slot), p);
            ph.flip(PH_MMA + slot);
            ok = ok && done;
        }
    }
    tc::cp_async_wait<0>();
    if (!ok) return false;
    tc::fence_after_sync();
    if (first) stamp(p, TS_SH_MMA_DONE);

    // tensor memory -> the partial slot: warp w reads rows 32 (w % 4) + lane, 16-column blocks w / 4, w / 4 + 2, ...
    const int row = (warp & 3) * 32 + lane;
    float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * t.r0 * d.R + (int64_t)chunk * t.nrows * d.R +
                 (int64_t)row * d.R;
    for (int c0 = (warp >> 2) * 16; c0 < d.R; c0 += 32) {
        float v[16];
        tc::tmem_ld16(sm.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + c0, v);
        if (row < t.nrows) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4 *>(dst + c0 + 4 * q) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (first) stamp(p, TS_SH_STORED);
    return true;
}

// ===========================================================================
// finish items
// ===========================================================================
// Scratch of a group: [tiles][n_kc][rows of the tile][R] fp32 partials, then
// the finished S: per tile bf16 [R/8][128][8] (tensor cores), or fp32
// [rows][R] of the whole group (small tiles).
__device__ __forceinline__ float *fin_area(const EngineParams &p, const EngineSmem &sm, const GroupDims &d, int g,
                                           int tile)
{
    return p.partials + sm.part_pre[g] + (int64_t)d.n_kc * d.count * d.R +
           (int64_t)tile * (d.tc ? kTcRows / 2 : kBgmvRows) * d.R;
}

// Rows [16 sl, 16 sl + 16) of a tile: S = sum over K-chunks (ascending) of the
// partials, rounded once to bf16 on the tensor-core path.
__device__ __forceinline__ bool finish_item(const EngineParams &p, EngineSmem &sm, const Plan &pl, int G, int f, bool first)
{
    if (first) stamp(p, TS_FIN_START);
    const int tid = threadIdx.x;
    const int g = find_group(sm.fin_pre, G, f);
    const GroupDims d = group_dims(p, sm, g, pl);
    const int local = f - sm.fin_pre[g];
    const int tile = d.tc ? local / (kTcRows / kFinRows) : local;
    const int sl = d.tc ? local % (kTcRows / kFinRows) : 0;
    const int r0 = tile * d.tile_rows;
    const int nrows = min(d.tile_rows, d.count - r0);
    const int tg = sm.tile_pre[g] + tile;
    if (tid == 0) sm.flag = wait_counter(&p.sync[tg * 4 + 0], d.n_kc, p) ? 1 : 0;
    __syncthreads();
    if (sm.flag == 0) return false;
    if (first) stamp(p, TS_FIN_READY);
    const int R = d.R, c4s = R / 4;
    const float *part = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * R;
    const int64_t stride = (int64_t)nrows * R;
    float *fa = fin_area(p, sm, d, g, tile);
    #pragma unroll 1
    for (int u = tid; u < kFinRows * c4s; u += kT) {
        const int uq = qdiv_s(u, c4s);
        const int row = sl * kFinRows + uq, c = (u - uq * c4s) * 4;
        if (row >= nrows) continue;
        const float *src = part + (int64_t)row * R + c;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q0 = 0; q0 < d.n_kc; q0 += 8) {
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q0 + q < d.n_kc) v[q] = __ldcg(reinterpret_cast<const float4 *>(src + (q0 + q) * stride));
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q0 + q < d.n_kc) {
                    acc.x += v[q].x; acc.y += v[q].y; acc.z += v[q].z; acc.w += v[q].w;
                }
            }
        }
        if (d.tc) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t *>(&lo);
            w.y = *reinterpret_cast<uint32_t *>(&hi);
            __nv_bfloat16 *S = reinterpret_cast<__nv_bfloat16 *>(fa);
            *reinterpret_cast<uint2 *>(S + ((int64_t)(c / 8) * kTcRows + row) * 8 + (c % 8)) = w;
        } else {
            *reinterpret_cast<float4 *>(fa + (int64_t)row * R + c) = acc;
        }
    }
    __syncthreads();
    if (tid == 0) release_add(&p.sync[tg * 4 + 2], 1);
    if (first) stamp(p, TS_FIN_DONE);
    return true;
}

// ===========================================================================
// expand items
// ===========================================================================

__device__ __forceinline__ ExpandItem decode_expand(const EngineParams &p, const EngineSmem &sm, const Plan &pl, int G,
                                                    int item)
{
    ExpandItem it;
    it.g = find_group(sm.ex_pre, G, item);
    it.d = group_dims(p, sm, it.g, pl);
    const int local = item - sm.ex_pre[it.g];
    it.tile = qdiv(local, it.d.ipt);
    int q = local - it.tile * it.d.ipt;
    const int lw = ceil_log2(it.d.uw);
    int s = 0;
    #pragma unroll 1
    for (; s < p.n_slices - 1; ++s) {
        const int is = qdiv_s(((p.slice_n[s] + it.d.uw - 1) >> lw) + it.d.ue - 1, it.d.ue);
        if (q < is) break;
        q -= is;
    }
    const int us = (p.slice_n[s] + it.d.uw - 1) >> lw;
    it.s = s;
    it.u0 = q * it.d.ue;
    it.nu = min(it.d.ue, us - it.u0);
    it.r0 = it.tile * it.d.tile_rows;
    it.nrows = min(it.d.tile_rows, it.d.count - it.r0);
    it.sa = (p.n_a == 1) ? 0 : s;
    it.tg = sm.tile_pre[it.g] + it.tile;
    return it;
}

// The issue side of the expand ring: the next unit of this CTA's expand
// items to put in flight.
// Put one expand unit in flight into stage seq % 3: its B rows and its output
// rows (bulk copies on bar_es), with a record of the unit.  The unit is column
// unit uu of slice s of a tile of nrows output rows; for the first unit of an
// item, thread t brings the tile's row t and its weight (read ahead by the
// caller), later units take them from the previous unit's stage (same thread,
// same row).  bblk_addr and scale are the group's B block and adapter scale.
__device__ __noinline__ void issue_unit(const EngineParams &p, const CUtensorMap *ymap, EngineSmem &sm, int seq, int s,
                                        int uu, int nrows, bool first, int first_row, float first_w,
                                        uint64_t bblk_addr, float scale, int rp, int uw, bool tc)
{
    const int tid = threadIdx.x;
    const int st = seq % kEsDepth;
    unsigned char *base = sm.pool + es_off(st);
    const int n0 = p.slice_off[s] + uu * uw;
    const int nw = min(uw, p.slice_n[s] - uu * uw);
    const int ystride = tc ? kTcYStride : uw * 2;
    const int yoff = tc ? kTcYOff : uw * rp * 2;
    if (tid < nrows) {
        int row;
        float w;
        if (first) {
            row = first_row;
            w = first_w;
        } else {
            const int pst = (seq + kEsDepth - 1) % kEsDepth;   // the previous unit, same item
            row = sm.row_dst[pst][tid];
            w = sm.row_w[pst][tid];
        }
        sm.row_dst[st][tid] = row;
        sm.row_w[st][tid] = w;
    }
    // a full 128-column unit of a 128-row tile whose rows are one run inside the rows of y moves as 2-D boxes
    bool run = false;
    if (tc) {
        __syncthreads();
        const int row0 = sm.row_dst[st][0];
        const bool mine = tid >= nrows || sm.row_dst[st][tid] == row0 + tid;
        run = __syncthreads_and(mine ? 1 : 0) != 0 && p.y_rows > 0 && nw == kTcCols &&
              row0 + kTcRows <= sm.x_total / p.m_mult * p.y_mult;
    }
    if (!run && tid < nrows)
        bulk_g2s(base + yoff + tid * ystride, p.y + (int64_t)sm.row_dst[st][tid] * p.ldy + n0, (uint32_t)nw * 2,
                 &sm.bar_es[st]);
    if (tid == 0) {
        const __nv_bfloat16 *bblk = reinterpret_cast<const __nv_bfloat16 *>(bblk_addr);
        const uint32_t y_bytes = run ? 2u * kTcRows * 128 : (uint32_t)nrows * nw * 2;
        const int kgs = rp / 8;
        UnitRec r;
        r.n0 = n0;
        r.nw = nw;
        r.nrows = nrows;
        r.kgs = kgs;
        r.yoff = yoff;
        r.ystride = ystride / 2;
        r.tc = tc;
        r.run = run;
        r.scale = scale;
        // the unit's 128-row B tiles are consecutive in the packed block: one bulk copy
        const int tile0 = p.slice_tile_off[s] + uu * (uw / kNTile);
        const int ntl = (nw + kNTile - 1) / kNTile;
        const uint32_t b_bytes = (uint32_t)ntl * kNTile * rp * 2;
        r.tw = kNTile;
        mbar_arrive_expect_tx(&sm.bar_es[st], b_bytes + y_bytes);
        bulk_g2s(base, bblk + (int64_t)tile0 * kNTile * rp, b_bytes, &sm.bar_es[st]);
        if (run)
            for (int h = 0; h < 2; ++h)
                tc::tma_tile2d(base + kTcYOff + h * kTcRows * 128, ymap, n0 + 64 * h, sm.row_dst[st][0],
                               &sm.bar_es[st]);
        sm.unit[st] = r;
    }
}

// The last consumer of a tile resets its counters for the next launch.  Thread 0 counts itself in as
// soon as its wait is over, and looks at the count only here, an item later (or at exit), so that the
// atomic's round trip stays off the path.
struct ConsumerTick {
    int tg = -1, old = 0, ipt = 0;
};
__device__ __forceinline__ void settle_tick(const EngineParams &p, ConsumerTick &c)
{
    if (threadIdx.x == 0 && c.tg >= 0 && c.old == c.ipt - 1) {
        p.sync[c.tg * 4 + 0] = 0;
        p.sync[c.tg * 4 + 1] = 0;
        p.sync[c.tg * 4 + 2] = 0;
    }
    c.tg = -1;
}

// Wait until the item's tile has its shrink results, then bring S into
// shared memory: bf16 [rp/8][128][8] by a bulk copy (tensor cores), fp32
// [16][rp] (padded rows) from the finished S or summed from the partials (small tiles).
__device__ __forceinline__ bool item_ready(const EngineParams &p, EngineSmem &sm, const ExpandItem &it, Phases &ph,
                                           bool first, ConsumerTick &tick)
{
    const int tid = threadIdx.x;
    const GroupDims &d = it.d;
    settle_tick(p, tick);
    if (tid == 0) {
        const bool ok = d.fin ? wait_counter(&p.sync[it.tg * 4 + 2], d.tc ? (it.nrows + kFinRows - 1) / kFinRows : 1, p)
                              : wait_counter(&p.sync[it.tg * 4 + 0], d.n_kc, p);
        if (ok) {
            tick.tg = it.tg;
            tick.ipt = d.ipt;
            tick.old = atomicAdd(&p.sync[it.tg * 4 + 1], 1);
        }
        if (ok && d.tc) {
            // S was written by other CTAs through ordinary stores: order them before the async copy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t s_bytes = (uint32_t)(d.rp / 8) * kTcRows * 16;
            const __nv_bfloat16 *S = reinterpret_cast<const __nv_bfloat16 *>(fin_area(p, sm, d, it.g, it.tile)) +
                                     (int64_t)it.sa * (d.rp / 8) * kTcRows * 8;
            mbar_arrive_expect_tx(&sm.bar_s, s_bytes);
            bulk_g2s(sm.pool, S, s_bytes, &sm.bar_s);
        }
        sm.flag = ok ? 1 : 0;
    }
    if (first) stamp(p, TS_EX_READY);
    __syncthreads();
    bool ready = sm.flag != 0;
    if (ready && !d.tc) {
        // small tile: S in bf16, row-major [16][rp] with padded rows (the MMA A operand)
        __nv_bfloat16 *S = reinterpret_cast<__nv_bfloat16 *>(sm.pool);
        const int rp = d.rp;
        const int64_t stride = (int64_t)it.nrows * d.R;
        const float *part = p.partials + sm.part_pre[it.g] + (int64_t)d.n_kc * it.r0 * d.R + it.sa * rp;
        const float *fin = d.fin ? fin_area(p, sm, d, it.g, it.tile) + it.sa * rp : nullptr;
        for (int idx = tid; idx < it.nrows * rp; idx += kT) {
            const int i = qdiv_s(idx, rp), jj = idx - i * rp;
            float acc = 0.f;
            if (d.fin) {
                acc = __ldcg(fin + (int64_t)i * d.R + jj);
            } else {   // sum over K-chunks q (ascending) of the published partials
                const float *src = part + (int64_t)i * d.R + jj;
                for (int q0 = 0; q0 < d.n_kc; q0 += 16) {
                    float v[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) v[u] = (q0 + u < d.n_kc) ? __ldcg(src + (q0 + u) * stride) : 0.f;
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (q0 + u < d.n_kc) acc += v[u];
                }
            }
            S[i * kSmSStride + jj] = __float2bfloat16_rn(acc);
        }
    }
    if (ready && d.tc) {
        ready = cta_wait(&sm.bar_s, ph.get(PH_S), p);
        ph.flip(PH_S);
    }
    __syncthreads();
    if (first) stamp(p, TS_EX_S);
    return ready;
}

// Small-tile units in stages st, st + 1, ..., st + n - 1 (mod 3), consecutive units of one item (same
// rows, same S): D[16][nw] = S B_unit^T with m16n8k16 MMAs (tokens as M, 8 output columns per MMA
// tile, warp w takes column tiles w, w + 8, ..., four at a time), then y = bf16(y_base + scale * w_row
// * D) for the tile's rows, two columns per store.  Ends with a barrier: the stages are free again.
__device__ __noinline__ void sm_unit(const EngineParams &p, EngineSmem &sm, int st, int n)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const UnitRec r0 = sm.unit[st];
    const uint32_t s_row = smem_u32(sm.pool) + (lane & 15) * kSmSStride * 2;
    const int gr = lane >> 2, qc = (lane & 3) * 2;
    const float s0 = gr < r0.nrows ? r0.scale * sm.row_w[st][gr] : 0.f;
    const float s1 = gr + 8 < r0.nrows ? r0.scale * sm.row_w[st][gr + 8] : 0.f;
    __nv_bfloat16 *const y0row = p.y + (int64_t)(gr < r0.nrows ? sm.row_dst[st][gr] : 0) * p.ldy;
    __nv_bfloat16 *const y1row = p.y + (int64_t)(gr + 8 < r0.nrows ? sm.row_dst[st][gr + 8] : 0) * p.ldy;
    if (r0.nrows <= kFmaRows) {
        // a few rows: CUDA-core dot products, two adjacent output columns per thread (the MMAs' 16-row
        // tiles would be mostly empty, and their dependent rounds cost more than the arithmetic)
        const __nv_bfloat16 *S = reinterpret_cast<const __nv_bfloat16 *>(sm.pool);
        const int tid = threadIdx.x, nr = r0.nrows;
        float sc[kFmaRows];
        __nv_bfloat16 *yr[kFmaRows];
#pragma unroll
        for (int i = 0; i < kFmaRows; ++i) {
            sc[i] = i < nr ? r0.scale * sm.row_w[st][i] : 0.f;
            yr[i] = p.y + (int64_t)sm.row_dst[st][i < nr ? i : 0] * p.ldy;
        }
        // column pairs of all n units, spread over every thread
        int pairs = 0;
        for (int j = 0; j < n; ++j) pairs += sm.unit[st + j < kEsDepth ? st + j : st + j - kEsDepth].nw >> 1;
        for (int q = tid; q < pairs; q += kT) {
            int j = 0, c = 2 * q;
            int sj = st;
            UnitRec r = sm.unit[sj];
            while (c >= r.nw) {   // (at most three units)
                c -= r.nw;
                ++j;
                sj = st + j < kEsDepth ? st + j : st + j - kEsDepth;
                r = sm.unit[sj];
            }
            const unsigned char *base = sm.pool + es_off(sj);
            const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(base + r.yoff);
            // B rows c, c + 1 of K-group kg: [(tl * kgs + kg) * tw + col] in 16-byte units
            const uint4 *bp = reinterpret_cast<const uint4 *>(base) + ((c >> 7) * r.kgs) * r.tw + (c & 127);
            float acc[kFmaRows][2];
#pragma unroll
            for (int i = 0; i < kFmaRows; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 1
            for (int kg = 0; kg < r.kgs; ++kg, bp += r.tw) {
                float b0[8], b1[8];
                bf16x8_to_f32(bp[0], b0);
                bf16x8_to_f32(bp[1], b1);
#pragma unroll
                for (int i = 0; i < kFmaRows; ++i) {
                    if (i < nr) {
                        float sv[8];
                        bf16x8_to_f32(*reinterpret_cast<const uint4 *>(S + i * kSmSStride + kg * 8), sv);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            acc[i][0] = fmaf(sv[e], b0[e], acc[i][0]);
                            acc[i][1] = fmaf(sv[e], b1[e], acc[i][1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kFmaRows; ++i) {
                if (i < nr) {
                    const __nv_bfloat162 yb = *reinterpret_cast<const __nv_bfloat162 *>(ys + i * r.ystride + c);
                    *reinterpret_cast<__nv_bfloat162 *>(yr[i] + r.n0 + c) = __floats2bfloat162_rn(
                        fmaf(sc[i], acc[i][0], __bfloat162float(yb.x)), fmaf(sc[i], acc[i][1], __bfloat162float(yb.y)));
                }
            }
        }
        __syncthreads();
        return;
    }
    const int steps = r0.kgs / 2;
    // (the K loop stays rolled and reloads its S fragment: this code runs about once per launch, where
    // its size, not its instruction count, sets the time)
    for (int j = 0; j < n; ++j) {
    const int sj = st + j < kEsDepth ? st + j : st + j - kEsDepth;
    const UnitRec r = sm.unit[sj];
    const unsigned char *base = sm.pool + es_off(sj);
    const uint32_t b_base = smem_u32(base);
    const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(base + r.yoff);
    __nv_bfloat16 *y0 = y0row + r.n0, *y1 = y1row + r.n0;
    const int ntiles = r.nw / 8;
    // four column tiles per round (w, w + 8, w + 16, w + 24), their MMAs interleaved
    for (int nt0 = warp; nt0 < ntiles; nt0 += 32) {
        float d[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll 1
        for (int k = 0; k < steps; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(s_row + (2 * k + (lane >> 4)) * 16, a0, a1, a2, a3);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = (nt0 + 8 * i) * 8;
                if (n < r.nw) {
                    // B rows n .. n + 7 of K-group kg: [(tl * kgs + kg) * tw + col] in 16-byte units
                    const int tl = n / kNTile, col = n % kNTile;
                    uint32_t b0, b1;
                    ldsm_x2(b_base + ((tl * r.kgs + 2 * k + ((lane >> 3) & 1)) * r.tw + col + (lane & 7)) * 16,
                            b0, b1);
                    mma16816(d[i], a0, a1, a2, a3, b0, b1);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (nt0 + 8 * i) * 8 + qc;
            if (c >= r.nw) continue;
            if (gr < r.nrows) {
                const __nv_bfloat162 yb = *reinterpret_cast<const __nv_bfloat162 *>(ys + gr * r.ystride + c);
                *reinterpret_cast<__nv_bfloat162 *>(y0 + c) = __floats2bfloat162_rn(
                    fmaf(s0, d[i][0], __bfloat162float(yb.x)), fmaf(s0, d[i][1], __bfloat162float(yb.y)));
            }
            if (gr + 8 < r.nrows) {
                const __nv_bfloat162 yb = *reinterpret_cast<const __nv_bfloat162 *>(ys + (gr + 8) * r.ystride + c);
                *reinterpret_cast<__nv_bfloat162 *>(y1 + c) = __floats2bfloat162_rn(
                    fmaf(s1, d[i][2], __bfloat162float(yb.x)), fmaf(s1, d[i][3], __bfloat162float(yb.y)));
            }
        }
    }
    }
    __syncthreads();
}

// Tensor-core unit in stage st: D(buf) = S B^T (one thread issues, commit on bar_mmae[buf]).
__device__ __forceinline__ void tc_unit_mma(EngineSmem &sm, int st, int buf)
{
    const UnitRec r = sm.unit[st];
    const unsigned char *base = sm.pool + es_off(st);
    const uint32_t acc = sm.tmem_base + kTmemExpandCol + buf * kTcCols;
    tc::fence_after_sync();
    for (int j = 0; j < r.kgs / 2; ++j) {
        const uint64_t ad = tc::smem_desc(smem_u32(sm.pool) + j * 2 * kTcRows * 16, kTcRows * 16, 128);
        const uint64_t bd = tc::smem_desc(smem_u32(base) + j * 2 * kTcCols * 16, kTcCols * 16, 128);
        tc::mma_bf16(acc, ad, bd, tc::idesc_bf16(kTcRows, kTcCols), j > 0 ? 1u : 0u);
    }
    tc::mma_commit(&sm.bar_mmae[buf]);
}

// Tensor-core epilogue of the unit in stage st, accumulator buffer buf: warp w
// owns row 32 (w % 4) + lane and 64 columns from 64 (w / 4); the result
// bf16(y_base + scale * w_row * D) overwrites the staged y row, which then
// leaves as one bulk store per row.  On return the stage is free again.
__device__ __noinline__ void tc_unit_epilogue(const EngineParams &p, const CUtensorMap *ymap_st, EngineSmem &sm,
                                              int st, int buf)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const UnitRec r = sm.unit[st];
    unsigned char *base = sm.pool + es_off(st);
    const int row = (warp & 3) * 32 + lane;
    const int cbase = (warp >> 2) * 64;
    const bool live = row < r.nrows;
    const float sc = r.scale * (live ? sm.row_w[st][row] : 0.f);
    // run tiles: rows below nrows rounded down to 32 go back to shared memory for the box stores, the
    // rest straight to y
    const int boxed = r.run ? (r.nrows & ~31) : 0;
    const bool to_smem = !r.run || row < boxed;
    __nv_bfloat16 *yg = p.y + (int64_t)(live ? sm.row_dst[st][row] : 0) * p.ldy + r.n0;
    const uint32_t acc = sm.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kTmemExpandCol + buf * kTcCols;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c0 = cbase + h * 32;
        float v[32];
        tc::tmem_ld32(acc + c0, v);
        if (live) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + 8 * q;
                if (c < r.nw) {
                    // padded rows, or 16-byte chunk (c % 64) / 8 of the row swizzled within its 1 KB atom
                    unsigned char *yp = r.run ? base + r.yoff + (c >> 6) * kTcRows * 128 + row * 128 +
                                                    ((((c & 63) >> 3) ^ (row & 7)) << 4)
                                              : base + r.yoff + row * kTcYStride + c * 2;
                    float yf[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(yp), yf);
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = __float2bfloat16_rn(fmaf(sc, v[8 * q + e], yf[e]));
                    if (to_smem) *reinterpret_cast<uint4 *>(yp) = *reinterpret_cast<const uint4 *>(o);
                    else *reinterpret_cast<uint4 *>(yg + c) = *reinterpret_cast<const uint4 *>(o);
                }
            }
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (r.run) {
        if (tid == 0 && boxed > 0) {
            const int row0 = sm.row_dst[st][0];
            for (int rb = 0; rb < boxed; rb += 32)
                for (int h = 0; h < 2; ++h)
                    tc::tma_store2d(ymap_st, r.n0 + 64 * h, row0 + rb, base + r.yoff + h * kTcRows * 128 + rb * 128);
            bulk_commit();
            bulk_wait_read();
        }
    } else if (tid < r.nrows) {
        bulk_s2g(p.y + (int64_t)sm.row_dst[st][tid] * p.ldy + r.n0, base + r.yoff + tid * kTcYStride,
                 (uint32_t)r.nw * 2);
        bulk_commit();
        bulk_wait_read();
    }
    __syncthreads();
}

// ===========================================================================
// the kernel
// ===========================================================================
// Warp 1, while warp 0 makes the plan: this CTA's share (by bytes) of every
// group's A block is asked into L2, so the shrink copies issued after the
// plan find it there.
__device__ __forceinline__ void prefetch_a_l2(const EngineParams &p, const EngineSmem &sm, int G)
{
    const int lane = threadIdx.x & 31;
    const int grid = gridDim.x, b = blockIdx.x;
    auto block = [&](int g, long long &bytes) -> uint64_t {
        bytes = 0;
        if (g >= G) return 0;
        const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
        if (gr.x < 0 || gr.x >= p.L || gr.y < 0 || gr.y >= p.num_experts) return 0;
        const int rp = gr.x < kRankCache ? sm.rp_cache[gr.x] : p.rpad[gr.x];
        bytes = (long long)p.n_a * rp * p.K * 2;
        return p.a_ptr[gr.x * p.E_A + (p.E_A == 1 ? 0 : gr.y)];
    };
    long long total = 0;
#pragma unroll 1
    for (int base = 0; base < G; base += 32) {
        long long bytes;
        block(base + lane, bytes);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        total += bytes;
    }
    const long long lo = total * b / grid, hi = total * (b + 1) / grid;
    long long carry = 0;
#pragma unroll 1
    for (int base = 0; base < G; base += 32) {
        long long bytes;
        const uint64_t addr = block(base + lane, bytes);
        long long incl = bytes;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const long long start = carry + incl - bytes;
        const long long a = max(lo, start) & ~15ll, e = min(hi, start + bytes);
        if (bytes > 0 && e > a) {
            const uint32_t size = (uint32_t)min(((e - a) + 15) & ~15ll, start + bytes - a);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr + (a - start)), "r"(size) : "memory");
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// Warp 0: size the chunks and units for this launch and lay out the work
// list (per-group prefix counts, packed sizes of the cached groups).
// Returns false for a workspace that lora_build_segments never filled.
__device__ __forceinline__ bool plan_launch(const EngineParams &p, EngineSmem &sm, int G, bool &any_tc)
{
    const int lane = threadIdx.x & 31;
    const int grid = gridDim.x;
    int N = 0, tc_units = 0;   // output columns; 128-column units of one tile over all slices
#pragma unroll 1
    for (int s = 0; s < p.n_slices; ++s) {
        N += p.slice_n[s];
        tc_units += (p.slice_n[s] + kTcCols - 1) >> 7;
    }
    // pass 1: validate; small-tile A and B bytes (in units of K and N bf16 elements), 128-row tile units
    bool bad = false;
    int bga = 0;            // (below 2^21: at most 65536 / 16 + 2048 tiles of at most 256 rows)
    int stiles = 0;         // small tiles
    int tcu = 0, tci = 0;
    any_tc = false;
#pragma unroll 1
    for (int g = lane; g < G; g += 32) {
        const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
        if (gr.x < 0 || gr.x >= p.L || gr.y < 0 || gr.y >= p.num_experts || gr.z < 0 || gr.w < 1 ||
            (int64_t)gr.z + gr.w > p.rows_capacity) {
            bad = true;
            continue;
        }
        const int rp = gr.x < kRankCache ? sm.rp_cache[gr.x] : p.rpad[gr.x];
        const bool tc = group_on_tc(p, gr.w, p.n_a * rp);
        if (tc) {
            const int tiles = (gr.w + kTcRows - 1) >> 7;
            any_tc = true;
            tcu += tiles * tc_units;
            tci += tiles;
        } else {
            const int tiles = (gr.w + kBgmvRows - 1) >> 4;
            bga += tiles * p.n_a * rp;
            stiles += tiles;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bga += __shfl_xor_sync(0xffffffffu, bga, o);
        stiles += __shfl_xor_sync(0xffffffffu, stiles, o);
        tcu += __shfl_xor_sync(0xffffffffu, tcu, o);
        tci += __shfl_xor_sync(0xffffffffu, tci, o);
    }
    bad = __any_sync(0xffffffffu, bad);
    any_tc = __any_sync(0xffffffffu, any_tc);
    if (bad) return false;
    // small-tile chunks of about a CTA's share of the A bytes (a quarter more, so that rounding up to
    // whole chunks rarely needs a second wave)
    Plan pl;
    // 128-row tile K-chunks of kTcKc; when that would make between one and two waves of shrink items
    // (some CTAs with two, most with one), chunks just long enough for one wave instead
    const int kmax = (p.K + 63) & ~63;
    int kctc = kTcKc;
    if (tci > 0 && tci * ((p.K + kTcKc - 1) / kTcKc) < 2 * grid) {
        const int nk = max(1, qdiv_s(grid, tci));
        kctc = min(kmax, max(kTcKc, (qdiv_s(p.K + nk - 1, nk) + 63) & ~63));
    }
    tci *= qdiv_s(p.K + kctc - 1, kctc);   // 128-row tile shrink items
    const int spare = max(grid / 4, grid - tci);
    // (targets, not sizes: the fast divides only need to agree between CTAs, and they run the same code)
    pl.ta = (int)fminf(268435456.f, fmaxf(8192.f, __fdividef(2.5f * (float)p.K * (float)bga, (float)spare)));
    pl.ue = min(128, max(1, qdiv(tcu + kItemsPerCta * grid - 1, kItemsPerCta * grid)));
    pl.kctc = kctc;
    // small-tile expand items of about half a CTA's share of all (tile, output column) pairs
    pl.ccol = (int)fminf(1073741824.f, __fdividef((float)stiles * (float)N, (float)(2 * grid)) + 1.f);
    // pass 2: per-group item counts and their exclusive prefix sums, 32 groups per step; larger chunks
    // until the hand-off scratch fits the workspace
#pragma unroll 1
    for (int iter = 0; iter < 8; ++iter) {
        int c_sh = 0, c_shs = 0, c_fin = 0, c_ex = 0, c_tile = 0;
        unsigned c_part = 0;   // scratch floats, saturating at 2^31 - 1 (a workspace error)
#pragma unroll 1
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int v_sh = 0, v_shs = 0, v_fin = 0, v_ex = 0, v_tile = 0;
            unsigned v_part = 0;
            if (g < G) {
                const GroupDims d = group_dims_calc(p, sm, g, pl);
                (d.tc ? v_sh : v_shs) = d.tiles * d.n_kc;
                v_fin = d.fins;
                v_ex = d.tiles * d.ipt;
                v_tile = d.tiles;
                v_part = (unsigned)min(d.scratch, (int64_t)INT32_MAX);
                if (g < kGroupCache) sm.gdim[g] = pack_dims(d);
            }
            int i_sh = v_sh, i_shs = v_shs, i_fin = v_fin, i_ex = v_ex, i_tile = v_tile;
            unsigned i_part = v_part;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, i_sh, o), b = __shfl_up_sync(0xffffffffu, i_fin, o);
                const int c = __shfl_up_sync(0xffffffffu, i_ex, o), e = __shfl_up_sync(0xffffffffu, i_tile, o);
                const unsigned f = __shfl_up_sync(0xffffffffu, i_part, o);
                const int h = __shfl_up_sync(0xffffffffu, i_shs, o);
                if (lane >= o) {
                    i_sh += a; i_fin += b; i_ex += c; i_tile += e; i_shs += h;
                    i_part = min(i_part + f, 0x7FFFFFFFu);
                }
            }
            if (g < G) {
                sm.sh_pre[g] = c_sh + i_sh - v_sh;
                sm.shs_pre[g] = c_shs + i_shs - v_shs;
                sm.fin_pre[g] = c_fin + i_fin - v_fin;
                sm.ex_pre[g] = c_ex + i_ex - v_ex;
                sm.tile_pre[g] = c_tile + i_tile - v_tile;
                sm.part_pre[g] = (int)min(c_part + (i_part - v_part), 0x7FFFFFFFu);
            }
            c_sh += __shfl_sync(0xffffffffu, i_sh, 31);
            c_shs += __shfl_sync(0xffffffffu, i_shs, 31);
            c_fin += __shfl_sync(0xffffffffu, i_fin, 31);
            c_ex += __shfl_sync(0xffffffffu, i_ex, 31);
            c_tile += __shfl_sync(0xffffffffu, i_tile, 31);
            c_part = min(c_part + __shfl_sync(0xffffffffu, i_part, 31), 0x7FFFFFFFu);
        }
        if (lane == 0) {
            sm.sh_pre[G] = c_sh;
            sm.shs_pre[G] = c_shs;
            sm.fin_pre[G] = c_fin;
            sm.ex_pre[G] = c_ex;
            sm.tile_pre[G] = c_tile;
            sm.part_pre[G] = (int)c_part;
            sm.ta = pl.ta;
            sm.ue = pl.ue;
            sm.kctc = pl.kctc;
            sm.ccol = pl.ccol;
        }
        if ((int64_t)c_part <= p.partial_floats || (pl.ta >= (1 << 27) && pl.kctc >= p.K)) break;
        pl.ta = min(1 << 28, pl.ta * 4);
        pl.kctc = min(1 << 20, pl.kctc * 4);
    }
    __syncwarp();
    return true;
}

__global__ void __launch_bounds__(kEngineThreads, 1) engine_kernel(const __grid_constant__ EngineParams pk)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    EngineSmem &sm = *reinterpret_cast<EngineSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = blockIdx.x, grid = gridDim.x;
    if (pk.trace != nullptr && tid > 0 && tid < kTraceSlots && b < pk.trace_ctas)
        pk.trace[(size_t)b * kTraceSlots + tid] = 0;
    stamp(pk, TS_ENTRY);
    {   // mirror the parameters in shared memory: out-of-line helpers read them there
        const uint32_t *src = reinterpret_cast<const uint32_t *>(&pk);
        uint32_t *dst = reinterpret_cast<uint32_t *>(&sm.pc);
        for (int i = tid; i < (int)(sizeof(EngineParams) / 4); i += kT) dst[i] = src[i];
    }
    const EngineParams &p = sm.pc;
    pdl_trigger();

    // ---- prologue: one round trip for the count, the first group records and the stored ranks ----
    if (tid == 0) {
        sm.flag = 0;
        mbar_init(&sm.bar_sh[0], 1);
        mbar_init(&sm.bar_sh[1], 1);
        for (int i = 0; i < kEsDepth; ++i) mbar_init(&sm.bar_es[i], 1);
        mbar_init(&sm.bar_s, 1);
        for (int i = 0; i < kTcMaxDepth; ++i) {
            mbar_init(&sm.bar_stage[i], 1);
            mbar_init(&sm.bar_mma[i], 1);
        }
        mbar_init(&sm.bar_mmae[0], 1);
        mbar_init(&sm.bar_mmae[1], 1);
        fence_mbar_init();
    }
    pdl_wait();   // everything below may read what earlier work on the stream wrote
    if (pk.ids != nullptr) {
        // the segment build fused in (dense, at most 32 tokens): warp 0 of every CTA sorts the ids itself,
        // and CTA 0 also leaves the table in the workspace for later launches
        if (warp == 0) {
            const int lane = tid, M = pk.ids_M, L = pk.L;
            const WarpRank r = warp_rank_ids(pk.ids, nullptr, M, L);
            const bool start = r.first && r.key < L;
            const int num_segments = __popc(__ballot_sync(0xffffffffu, start));
            const int num_valid = __popc(__ballot_sync(0xffffffffu, lane < M && r.key < L));
            sm.row_src[r.rank] = lane;   // (the slots are a permutation of the 32 lanes)
            const int4 seg = make_int4(r.key, 0, r.rank, r.count);
            if (start) sm.grp[r.seg] = seg;
            if (lane == 0) {
                sm.G = num_segments;
                sm.x_total = M;
            }
            if (b == 0) {
                if (lane < M) pk.ws_perm[r.rank] = lane;
                if (start) pk.ws_segments[r.seg] = seg;
                if (__any_sync(0xffffffffu, r.bad) && lane == 0) atomicOr(pk.err, kErrBadId);
                if (lane == 0) {
                    pk.ws_header[H_M] = M;
                    pk.ws_header[H_NUM_SEGMENTS] = num_segments;
                    pk.ws_header[H_NUM_VALID] = num_valid;
                    pk.ws_header[H_NUM_MOE_GROUPS] = 0;
                    pk.ws_header[H_BLOCK_M] = 0;
                }
            }
            // the row list is read through the parameter mirror: point it at this CTA's copy
            if (lane == 0) sm.pc.rows = sm.row_src;
        }
    } else {
        if (tid == 0) {
            sm.G = *pk.num_groups;
            sm.x_total = *pk.m_ptr * pk.m_mult;
        }
        const int gpre = min(pk.group_capacity, kGroupCache);
        for (int g = tid; g < gpre; g += kT) sm.grp[g] = pk.groups[g];
    }
    for (int a = tid; a < min(pk.L, kRankCache); a += kT) sm.rp_cache[a] = pk.rpad[a];
    __syncthreads();
    stamp(p, TS_PRO_LOADED);
    const int G = sm.G;
    if (G <= 0) return;
    if (G > p.group_capacity || G > kGroupCap) {
        if (b == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    if (warp == 0) {
        bool any_tc = false;
        const bool good = plan_launch(p, sm, G, any_tc);
        if (tid == 0) sm.flag = good ? (any_tc ? 2 : 0) : 1;
    } else if (warp == 1) {
        prefetch_a_l2(p, sm, G);
    } else if (warp == 2) {
        // the first groups' table entries, so that no copy issue waits on a table read
        for (int g = tid - 64; g < min(G, kPtrCache); g += 32) {
            const int4 gr = sm.grp[g];
            const bool ok = gr.x >= 0 && gr.x < p.L && gr.y >= 0 && gr.y < p.num_experts;
            sm.a_blk[g] = ok ? p.a_ptr[gr.x * p.E_A + (p.E_A == 1 ? 0 : gr.y)] : 0;
            sm.b_blk[g] = ok ? p.b_ptr[gr.x * p.E_B + (p.E_B == 1 ? 0 : gr.y)] : 0;
            sm.g_scale[g] = ok ? p.scale[gr.x] : 0.f;
        }
    }
    __syncthreads();
    stamp(p, TS_PRO_PLANNED);
    if (sm.flag == 1) {
        if (b == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    const bool use_tc = sm.flag == 2;
    const int n_sh_tc = sm.sh_pre[G], n_sh_sm = sm.shs_pre[G];
    const int n_shrink = n_sh_tc + n_sh_sm, n_fin = sm.fin_pre[G], n_expand = sm.ex_pre[G];
    if (sm.tile_pre[G] > p.max_tiles || (int64_t)sm.part_pre[G] > p.partial_floats ||
        sm.part_pre[G] == INT32_MAX) {
        if (b == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    if (use_tc && (smem_u32(sm.pool) & 1023u) != 0) {   // swizzled TMA tiles need a 1024-byte aligned pool
        if (b == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    // one warp allocates the tensor memory this CTA's MMAs accumulate into (launches with 128-row tiles only)
    if (use_tc) {
        if (warp == 0) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    const Plan pl = {sm.ta, sm.ue, sm.ccol, sm.kctc};
    stamp(p, TS_WORKLIST);

    Phases ph = {0u};
    uint32_t inflight = 0;   // expand stages whose copies have not been waited for
    int issued = 0;          // expand units put in flight
    bool alive = true;

    // this CTA's items, each kind dealt on from where the previous one stopped (so CTAs with less of one
    // kind take the next first): 128-row tile shrink items b, b + grid, ...; small-tile shrink items;
    // finish items; expand items
    const int my_tc = b < n_sh_tc ? qdiv(n_sh_tc - b + grid - 1, grid) : 0;
    const int s0 = pmod(b - n_sh_tc, grid);
    const int my_shrink = my_tc + (s0 < n_sh_sm ? qdiv(n_sh_sm - s0 + grid - 1, grid) : 0);
    // the CTA's j-th shrink item: group and index within the group
    auto shrink_item = [&](int j, int &g, int &local) {
        if (j < my_tc) {
            const int t = b + j * grid;
            g = find_group(sm.sh_pre, G, t);
            local = t - sm.sh_pre[g];
        } else {
            const int u = s0 + (j - my_tc) * grid;
            g = find_group(sm.shs_pre, G, u);
            local = u - sm.shs_pre[g];
        }
    };
    const int f0 = pmod(b - n_shrink, grid);
    const int e0 = pmod(b - n_shrink - n_fin, grid);
    // the expand issuer starts at item e0; expand units may be in flight while the shrink items run:
    // stage 0 beside a tensor-core shrink, stages 0 and 1 beside a small-tile one.  Set up after the
    // first shrink item's copies are on their way.
    int npre = kEsDepth;
    bool iss_ready = false;
    // issue side of the expand ring, kept by every thread alike: unit iss_k of item iss_item
    int iss_item = n_expand, iss_k = 0;
    ExpandItem iss_it;
    int iss_row = 0;        // this thread's output row of the item's tile, and its weight (read ahead)
    float iss_w = 1.f;
    auto iss_enter = [&](int item) {
        iss_item = item;
        if (item >= n_expand) return;
        iss_it = decode_expand(p, sm, pl, G, item);
        if (tid < iss_it.nrows) {
            iss_row = p.rows[iss_it.d.rows_off + iss_it.r0 + tid];
            iss_w = p.row_weight ? p.row_weight[iss_row] : 1.f;
        }
    };
    auto setup_issuer = [&]() {
        iss_enter(e0);
        if (my_shrink > 0) npre = 1;   // the shrink staging (and its cross-warp sums) reach into stage 1
        iss_ready = true;
    };
    // put units in flight until `upto` have been issued (units must have left stage (upto - 1) % 3)
    auto prefetch = [&](int upto) {
        while (issued < upto && iss_item < n_expand) {
            inflight |= 1u << (issued % kEsDepth);
            const GroupDims &d = iss_it.d;
            issue_unit(p, &pk.y_map_ld, sm, issued++, iss_it.s, iss_it.u0 + iss_k, iss_it.nrows, iss_k == 0, iss_row,
                       iss_w, d.bblk, d.scale, d.rp, d.uw, d.tc);
            if (++iss_k == iss_it.nu) {
                iss_k = 0;
                iss_enter(iss_item + grid);
            }
        }
    };

    // ------------------------------------------------------------------ shrink items
    uint32_t sh_inflight = 0;   // small-tile staging slots whose copies have not been waited for
    for (int j = 0; j < my_shrink && alive; ++j) {
        int g, local;
        shrink_item(j, g, local);
        const GroupDims d = group_dims(p, sm, g, pl);
        const int tile = qdiv(local, d.n_kc), chunk = local - tile * d.n_kc;
        const int tg = sm.tile_pre[g] + tile;
        const bool first = j == 0;
        if (first) stamp(p, TS_SH_START);
        bool ok;
        if (d.tc) {
            const TcShrink t = tc_shrink_issue(p, &pk.x_map, sm, d, tile, chunk);
            if (first) {
                setup_issuer();
                prefetch(npre);
            }
            ok = tc_shrink_run(p, &pk.x_map, sm, d, t, g, chunk, ph, first);
        } else {
            // small tiles alternate between two staging slots: the next item's operands are put in flight
            // before this one's are waited for
            const int slot = (j - my_tc) & 1;
            const BgShrink bs = sm_shrink_desc(p, d, tile, chunk);
            if (j == my_tc) {
                sm_shrink_issue(p, sm, d, bs, slot);
                sh_inflight |= 1u << slot;
            }
            if (first) setup_issuer();
            if (j + 1 < my_shrink) {
                int g2, local2;
                shrink_item(j + 1, g2, local2);
                const GroupDims d2 = group_dims(p, sm, g2, pl);
                const int tile2 = qdiv(local2, d2.n_kc);
                sm_shrink_issue(p, sm, d2, sm_shrink_desc(p, d2, tile2, local2 - tile2 * d2.n_kc), slot ^ 1);
                sh_inflight |= 1u << (slot ^ 1);
            }
            // the first expand units go in flight while the shrink operands land: issuing them is
            // longer than their bytes are large, so it stays off the hand-off's path
            if (first) prefetch(npre);
            ok = sm_shrink_wait(p, sm, ph, slot, first);
            sh_inflight &= ~(1u << slot);
            if (ok) sm_shrink_run(p, sm, d, bs, g, chunk, slot, first);
        }
        if (!ok) {
            alive = false;
            break;
        }
        if (tid == 0 && !p.withhold) release_add(&p.sync[tg * 4 + 0], 1);
        if (first) stamp(p, TS_SH_PUBLISHED);
    }
    // the shrink staging is free: the rest of the ring may fill while the finish items run
    if (!iss_ready) setup_issuer();
    if (alive) prefetch(kEsDepth);
    stamp(p, TS_PREFETCHED);

    // ------------------------------------------------------------------ finish items
    for (int f = f0; f < n_fin && alive; f += grid)
        if (!finish_item(p, sm, pl, G, f, f == f0)) alive = false;

    // ------------------------------------------------------------------ expand items
    int seq = 0;     // units computed
    ConsumerTick tick;   // thread 0: the last tile this CTA counted itself in on
    int pend = -1;   // unit whose MMAs are issued and whose epilogue is pending
    auto drain = [&]() -> bool {   // epilogue of the pending unit, then refill its stage
        const int q = pend, st = q % kEsDepth, buf = q & 1;
        if (!cta_wait(&sm.bar_mmae[buf], ph.get(PH_MMAE + buf), p)) return false;
        ph.flip(PH_MMAE + buf);
        tc::fence_after_sync();
        tc_unit_epilogue(p, &pk.y_map_st, sm, st, buf);
        if (q < 4) stamp(p, TS_EX_UNIT + 2 * q + 1);
        pend = -1;
        prefetch(q + 1 + kEsDepth);
        return true;
    };
    for (int item = e0; item < n_expand && alive; item += grid) {
        const ExpandItem it = decode_expand(p, sm, pl, G, item);
        if (pend >= 0 && !drain()) {
            alive = false;
            break;
        }
        if (!item_ready(p, sm, it, ph, item == e0, tick)) {
            alive = false;
            break;
        }
        for (int k = 0; k < it.nu; ++k, ++seq) {
            const int st = seq % kEsDepth;
            if (!cta_wait(&sm.bar_es[st], ph.get(PH_ES + st), p)) {
                alive = false;
                break;
            }
            ph.flip(PH_ES + st);
            inflight &= ~(1u << st);
            if (seq < 4) stamp(p, TS_EX_UNIT + 2 * seq);
            if (!it.d.tc) {
                if (pend >= 0 && !drain()) {   // units leave the ring in order
                    alive = false;
                    break;
                }
                // the item's next units whose copies have already landed join this pass
                int n = 1;
                while (n < it.nu - k && n < issued - seq) {
                    const int sn = (seq + n) % kEsDepth;
                    if (!__syncthreads_and(mbar_try_wait(&sm.bar_es[sn], ph.get(PH_ES + sn)) ? 1 : 0)) break;
                    ph.flip(PH_ES + sn);
                    inflight &= ~(1u << sn);
                    ++n;
                }
                sm_unit(p, sm, st, n);   // ends with a barrier: the n stages are free again
                seq += n - 1;
                k += n - 1;
                if (seq < 4) stamp(p, TS_EX_UNIT + 2 * seq + 1);
                prefetch(seq + 1 + kEsDepth);
                continue;
            }
            // this unit's MMAs go in while the previous unit's epilogue runs
            if (tid == 0) tc_unit_mma(sm, st, seq & 1);
            if (pend >= 0 && !drain()) {
                alive = false;
                break;
            }
            pend = seq;
        }
    }
    if (alive && pend >= 0 && !drain()) alive = false;
    settle_tick(p, tick);

    // a CTA that gave up still lets its copies land and its MMAs finish before it leaves
    for (int sl = 0; sl < 2; ++sl)
        if (sh_inflight & (1u << sl))
            mbar_wait_bounded(&sm.bar_sh[sl], ph.get(ph_shrink(sl)), p.timeout_ns, p.err);
    for (int st = 0; st < kEsDepth; ++st)
        if (inflight & (1u << st)) mbar_wait_bounded(&sm.bar_es[st], ph.get(PH_ES + st), p.timeout_ns, p.err);
    if (pend >= 0) mbar_wait_bounded(&sm.bar_mmae[pend & 1], ph.get(PH_MMAE + (pend & 1)), p.timeout_ns, p.err);
    bulk_wait_all();
    stamp(p, TS_EXIT);
    if (use_tc) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(sm.tmem_base, kTmemCols);
    }
}

const void *engine_kernel_ptr() { return reinterpret_cast<const void *>(engine_kernel); }

void launch_engine(const EngineParams &p, int grid, size_t smem, cudaStream_t s, bool pdl, cudaError_t *err)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kEngineThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    *err = cudaLaunchKernelEx(&cfg, engine_kernel, p);
}

}  // namespace lora
