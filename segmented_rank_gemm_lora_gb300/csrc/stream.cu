// The streaming path behind lora_apply and lora_moe_delta: two kernels
// chained on the stream with programmatic dependent launch.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 2.3: every segment is a
// shrink X_seg A_i^T followed by an expand with B_i^T added to the base rows,
// all segments in one operator instance spread over the cores; section 2.4:
// the work of every core is fixed before the compute starts, the token
// dimension is tiled first and then K, so a piece of A fits on chip and the
// pieces are accumulated; section 4.2: the rank-sized intermediate S
// accumulates in fp32.
//
// GB300 form.  Every byte the delta needs crosses HBM once (B once per row
// tile), so the kernels are built to keep the memory system busy rather than
// the tensor cores.  Contiguous runs (packed A and B, S) move as bulk copies;
// gathered rows of x and y move as 16-byte cp.async pieces from groups of four
// warps, because one warp alone issues them far below the memory's rate and
// the bulk-copy engine spends a fixed time per copy.
//   plan    every block of the shrink, from the group table alone (no block
//           waits for another): cuts every group (an adapter segment, or an
//           (adapter, expert) group of the MoE variant) into row tiles of at
//           most 64 rows, every tile's shrink into K-chunks (the same cut for
//           all tiles of a group) and its expand into units of W output
//           columns of one slice; a group's tiles differ by at most one row,
//           so every tile's positions have a closed form.  Each block takes a
//           contiguous run of chunks of about equal bytes, keeps the records
//           of their tiles, and writes its share of the launch's records.
//   shrink  one block per SM, launched cooperatively.  Warps 8-11 fill a
//           six-stage ring: each stage is the chunk's next K columns of A
//           (one bulk copy) and of the tile's x rows (cp.async pieces), both
//           in the tensor core's K-major operand layout, with the stage's
//           (tile, chunk); one thread issues tcgen05 MMAs (the A block's rows
//           as the 128-row M operand, the tile's rows as N) into one of two
//           tensor-memory accumulators per chunk; warps 4-7 move each chunk's
//           fp32 partial to L2 scratch and count it on its tile.  A block
//           leaves as soon as its chunks are done.
//   expand  one block per SM, warp-specialised; its blocks start on the SMs
//           that shrink blocks leave, once every shrink block has written its
//           share of the launch's tile records.  Warp 0 (the leader) walks
//           the block's units (its share, then units of the launch's tail
//           claimed one at a time) and hands each to the other roles through
//           a shared-memory queue while it streams the unit's packed B columns
//           into a three-stage ring; warps 4-7 gather the unit's y rows into a
//           six-slot ring (neither needs the shrink).  The twelve epilogue
//           warps of every block sum an equal run of the launch's S chunks
//           (a tile's partials in chunk order, bf16 into the operand layout),
//           each tile's once all its K-chunks are counted, and count the sums
//           on the tile; warp 1 loads S per (tile, slice block) once all of
//           the tile's sums are counted; warp 2 issues tcgen05 MMAs
//           D = B_unit S^T (the unit's output columns as the 128-row M
//           operand, the tile's rows as N) into one of four tensor-memory
//           accumulators; three epilogue warpgroups take units in rotation:
//           each reads its accumulator, adds scale * D into the staged rows
//           and stores them.  The hand-offs inside a block are mbarriers; the
//           waits across blocks are bounded spins on counters that the last
//           expand block to end resets for the next launch.
//
// Summation orders depend only on a group's sizes (its K-chunk cut, the MMA
// shapes), never on timing, on which block ran a piece, or on which rows
// share a tile, so the same inputs give the same bits and permuting tokens
// permutes the output bits.
#include "common.cuh"
#include "tc.cuh"

namespace lora {

constexpr int kPlanItems = 3;                   // shrink chunks per block the plan aims for
constexpr int kPartialPerRow = 8192;            // fp32 partials per row of a tile, at most (bounds the K-chunk from below)
constexpr int kTileRows = 64;                   // rows of a tile, at most
constexpr int kShWarps = 8;                     // warps before the producers: MMA issuer, tensor-memory owner, epilogue
constexpr int kShProd = 128;                    // producer threads (the four warps after them)
constexpr int kShThreads = 32 * kShWarps + kShProd;
constexpr uint32_t kShAccCols = 128;            // tensor-memory columns of one shrink accumulator (two of them)
constexpr int kShStages = 6;
constexpr int kMyTiles = 16;                    // tiles of its own chunks a shrink block keeps on chip
constexpr int kShStageBytes = 32 * 1024;        // A columns and x rows of one stage, at most
constexpr int kExGroups = 3;                    // epilogue warpgroups (units dealt round-robin)
constexpr int kExYProd = 128;                   // y producer threads: warps 4-7
constexpr int kExThreads = 128 + kExYProd + 128 * kExGroups;   // B producer, S loader, MMA issuer, a spare warp,
                                                               // y producers, epilogue groups
constexpr int kExEpi = 128;                     // threads of one epilogue warpgroup
constexpr int kExBStages = 3;
constexpr int kExBBytes = 32 * 1024;            // B columns of one unit, at most
constexpr int kExYStages = 6;
constexpr int kExYBytes = 16 * 1024;            // y rows of one unit, at most
constexpr int kExSBytes = 8 * 1024;             // S of one slice block: at most 64 ranks x 64 rows, bf16
constexpr int kExQ = 16;                        // entries of the expand's unit queue
constexpr int kExPoolDiv = 6;                   // the expand claims the last 1 / kExPoolDiv of its cost at run time
constexpr int kExUposCap = 2048;                // tiles whose first units the expand keeps on chip for its claims
constexpr int kExAcc = 4;                       // tensor-memory accumulators of kExAccCols columns
constexpr int kExAccCols = 128;
constexpr uint32_t kExTmemCols = kExAcc * kExAccCols;
constexpr int kCostUnit = 512;                  // bytes per unit of the plan's cost positions

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ TileRec load_tile(const TileRec *t)
{
    const int4 *q = reinterpret_cast<const int4 *>(t);
    const int4 v0 = __ldcg(q), v1 = __ldcg(q + 1), v2 = __ldcg(q + 2), v3 = __ldcg(q + 3);
    TileRec r;
    r.a = v0.x; r.e = v0.y; r.row0 = v0.z; r.m = v0.w;
    r.rp = v1.x; r.R = v1.y; r.n_pad = v1.z; r.kc = v1.w;
    r.n_kc = v2.x; r.ks = v2.y; r.W = v2.z; r.n_units = v2.w;
    r.p_off = v3.x; r.s_off = v3.y; r.c0 = v3.z; r.u0 = v3.w;
    return r;
}

// Bounded wait for *flag >= want (gpu-scope acquire); false (and the timeout bit) when it ran out.
__device__ __forceinline__ bool wait_at_least(const StreamParams &p, const int32_t *flag, int want)
{
    if (ld_acquire_gpu(flag) >= want) return true;
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(flag) < want) {
        if (globaltimer() - t0 > p.timeout_ns) {
            atomicOr(p.err, kErrTimeout);
            return false;
        }
        nanosleep_ns(64);
    }
    return true;
}

// (t, j) comes before the end marker e in the (tile, item) order
__device__ __forceinline__ bool before(int t, int j, int2 e) { return t < e.x || (t == e.x && j < e.y); }

// Named barrier over `count` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool bar_and(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Phase stamps (lora_set_trace): kernel k (0 shrink, 1 expand), slot s of this block.
__device__ __forceinline__ void tstamp(const StreamParams &p, int k, int s)
{
    if (p.trace != nullptr && (int)blockIdx.x < p.trace_ctas)
        p.trace[((size_t)k * p.trace_ctas + blockIdx.x) * kTraceSlots + s] = globaltimer();
}

// ===========================================================================
// plan (block 0 of the shrink grid)
// ===========================================================================
template <class T>
__device__ __forceinline__ T warp_sum(T v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
template <class T>
__device__ __forceinline__ T warp_inclusive(T v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// The plan of one group: its row tiles (m = base + 1 for the first rem tiles, else base), the shrink
// chunk cut and stage K, the expand unit width.
struct GroupPlan {
    int a, e, row_off, count, rp, R, ntl, base, rem, kc, n_kc, ks, W, n_units;
};

__device__ __forceinline__ int group_tiles(const StreamParams &p, int count)
{
    const int tmax = min(p.tile_max, kTileRows);
    return (count + tmax - 1) / tmax;
}

// `target` is the shrink bytes the plan aims to give one chunk.  Only 32-bit integer and fp32 arithmetic:
// a 64-bit integer divide is a long emulated sequence on this GPU.
__device__ __forceinline__ GroupPlan group_plan(const StreamParams &p, int4 gr, int rp, float target)
{
    GroupPlan g;
    g.a = gr.x;
    g.e = gr.y;
    g.row_off = gr.z;
    g.count = gr.w;
    g.rp = rp;
    g.R = p.n_a * rp;
    g.ntl = group_tiles(p, g.count);
    g.base = g.count / g.ntl;
    g.rem = g.count - g.base * g.ntl;
    const int m_max = g.base + (g.rem > 0 ? 1 : 0);
    const int K = p.K;
    // shrink: a stage (ks columns of A and of the tile's x rows, both as [ks / 8][rows][8] with the x rows
    // rounded up to 16) fills at most one ring stage; the chunk (the same cut for every tile of the group) is
    // about `target` bytes, and gives no more than kPartialPerRow partial floats per row
    const int ks = min(512, kShStageBytes / 2 / (g.R + ((m_max + 15) & ~15))) / 16 * 16;
    const int k_all = (K + ks - 1) / ks * ks;
    const int kc_min = min(((K * g.R + kPartialPerRow - 1) / kPartialPerRow + ks - 1) / ks * ks, k_all);   // K R < 2^29
    const float want = fminf(target / (2.f * (g.R + m_max)), (float)k_all);
    int kc = (int)ceilf(want / ks) * ks;
    kc = min(max(kc, max(ks, kc_min)), k_all);
    g.ks = ks;
    g.kc = kc;
    g.n_kc = (K + kc - 1) / kc;
    // expand: unit width W (its B columns and its y rows each fill at most one stage; its accumulator fits
    // kExAccCols tensor-memory columns)
    const int npad_max = (m_max + 15) & ~15;
    int W = 1024;
    while (W > 128 && (W * g.rp * 2 > kExBBytes || W * m_max * 2 > kExYBytes || (W / 128) * npad_max > kExAccCols))
        W >>= 1;
    g.W = W;
    int n_units = 0;
#pragma unroll
    for (int s = 0; s < kMaxSlices; ++s)
        if (s < p.n_slices) n_units += (p.slice_n[s] + W - 1) / W;
    g.n_units = n_units;
    return g;
}

// Cost of one shrink chunk and of one expand unit of a tile of m rows, in units of kCostUnit bytes (at
// least 1).
__device__ __forceinline__ int chunk_cost(int kc, int R, int m) { return max(1, kc * (R + m) * 2 / kCostUnit); }
__device__ __forceinline__ int unit_cost(int W, int rp, int m) { return max(1, W * (rp + 2 * m) * 2 / kCostUnit); }

// G blocks over a total cost T: block c starts at position c q + min(c, r), q = T / G, r = T % G
// (contiguous shares that differ by at most one; start(G) = T).
struct Split {
    int G, q, r;
    __device__ __forceinline__ Split(int T, int G_) : G(G_), q(T / G_), r(T - (T / G_) * G_) {}
    __device__ __forceinline__ int start(int c) const { return c * q + min(c, r); }
};

// Launch-wide position of a group's first item in every order the plan keeps: shrink cost, expand cost,
// S chunks (16 bytes each; S bytes are 16 times this), tiles, chunks, units, partial floats.  Entry G holds
// the totals.
struct GroupPos {
    int32_t sh, ex, rd, t, c, u, P;
};
enum PlanOrder { ORD_SH = 0, ORD_EX = 1, ORD_RD = 2 };

// The first `rem` tiles of a group have base + 1 rows and the others base rows, so an amount per tile takes
// one of two values (A, B) and a tile's position in any order has a closed form.
struct TwoWay {
    int A, B, rem;
    __device__ __forceinline__ int before(int i) const { return min(i, rem) * A + max(0, i - rem) * B; }
    // the tile holding offset off (0 <= off < the group's total)
    __device__ __forceinline__ int find(int off) const { return off < rem * A ? off / A : rem + (off - rem * A) / B; }
};
__device__ __forceinline__ int npad16(int m) { return (m + 15) & ~15; }
__device__ __forceinline__ TwoWay two_way(const GroupPlan &g, int order)
{
    const int m1 = g.base + 1, m0 = g.base;
    switch (order) {
    case ORD_SH: return {g.n_kc * chunk_cost(g.kc, g.R, m1), g.n_kc * chunk_cost(g.kc, g.R, m0), g.rem};
    case ORD_EX: return {g.n_units * unit_cost(g.W, g.rp, m1), g.n_units * unit_cost(g.W, g.rp, m0), g.rem};
    default: return {g.R * npad16(m1) / 8, g.R * npad16(m0) / 8, g.rem};
    }
}

// Shared memory of a block while it plans (it overlays the stage ring, which is not in use yet).
constexpr int kPlanGroups = 4096;   // groups whose positions fit; a larger plan fails with LORA_ERR_WORKSPACE
constexpr int kPlanKept = 512;      // groups whose plans are kept (later groups are planned again when needed)
struct GroupKept {
    int32_t ntl, base, rem, kc, n_kc, ks, W, n_units;
};
struct PlanSmem {
    GroupPos pos[kPlanGroups + 1];
    int4 gr[kPlanGroups];        // the group records
    int32_t rp[kPlanGroups];     // their adapters' stored ranks
    GroupKept kept[kPlanKept];
    int32_t G, bad;
    float target;
};

__device__ __forceinline__ int gpos_field(const GroupPos &q, int order)
{
    return order == ORD_SH ? q.sh : order == ORD_EX ? q.ex : q.rd;
}

// The group holding position `lo` of an order, or tile `t` (order -1): the last g with pos[g] <= lo.
__device__ __forceinline__ int find_group(const PlanSmem &ps, int order, int lo)
{
    int l = 0, h = ps.G;
    while (h - l > 1) {
        const int mid = (l + h) >> 1;
        if ((order < 0 ? ps.pos[mid].t : gpos_field(ps.pos[mid], order)) <= lo) l = mid;
        else h = mid;
    }
    return l;
}

__device__ __forceinline__ GroupPlan load_group_plan(const StreamParams &p, const PlanSmem &ps, int g)
{
    if (g >= kPlanKept) return group_plan(p, ps.gr[g], ps.rp[g], ps.target);
    const int4 gr = ps.gr[g];
    const GroupKept &k = ps.kept[g];
    GroupPlan r;
    r.a = gr.x;
    r.e = gr.y;
    r.row_off = gr.z;
    r.count = gr.w;
    r.rp = ps.rp[g];
    r.R = p.n_a * r.rp;
    r.ntl = k.ntl;
    r.base = k.base;
    r.rem = k.rem;
    r.kc = k.kc;
    r.n_kc = k.n_kc;
    r.ks = k.ks;
    r.W = k.W;
    r.n_units = k.n_units;
    return r;
}

// Warp 0 of every block: the group table, its plan and every group's positions.  Reads only what the
// build wrote, so no block waits for another to plan.
__device__ void plan_groups(const StreamParams &p, PlanSmem &ps)
{
    const int lane = threadIdx.x & 31;
    // the group count, the first 32 group records and the first 32 stored ranks in one round trip
    const int G = max(0, min(__ldcg(p.num_groups), p.group_capacity));
    const int4 gr0 = lane < p.group_capacity ? __ldcg(p.groups + lane) : make_int4(0, 0, 0, 0);
    const int rp0 = lane < p.L ? __ldg(p.rpad + lane) : 0;
    auto rank_of = [&](int a) {   // stored rank of adapter a (a shuffle for the first 32)
        const int v = __shfl_sync(0xffffffffu, rp0, a & 31);
        return a < 32 ? v : __ldg(p.rpad + a);
    };
    // tiles, and the shrink bytes of the whole launch
    long long est = 0;
    int ntot = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        const int4 gr = g0 == 0 ? gr0 : (g < G ? __ldcg(p.groups + g) : make_int4(0, 0, 0, 0));
        const int rp = rank_of(gr.x);
        if (g < G) {
            const int ntl = group_tiles(p, gr.w);
            ntot += ntl;
            est += (long long)p.K * 2 * ((long long)p.n_a * rp * ntl + gr.w);
            if (g < kPlanGroups) {
                ps.gr[g] = gr;
                ps.rp[g] = rp;
            }
        }
    }
    est = warp_sum(est);
    ntot = warp_sum(ntot);
    if (lane == 0) tstamp(p, 0, 10);
    const float target = fmaxf(1.f, (float)est / ((float)p.grid_s * kPlanItems));
    bool bad = G > kPlanGroups || ntot > p.max_tiles;
    // every group's positions: exclusive prefix sums over the groups, 32 at a time
    long long run[7] = {0, 0, 0, 0, 0, 0, 0};
    for (int g0 = 0; !bad && g0 < G; g0 += 32) {
        const int g = g0 + lane;
        long long v[7] = {0, 0, 0, 0, 0, 0, 0};
        if (g < G) {
            const GroupPlan gp = group_plan(p, ps.gr[g], ps.rp[g], target);
            if (g < kPlanKept) ps.kept[g] = {gp.ntl, gp.base, gp.rem, gp.kc, gp.n_kc, gp.ks, gp.W, gp.n_units};
            v[0] = two_way(gp, ORD_SH).before(gp.ntl);
            v[1] = two_way(gp, ORD_EX).before(gp.ntl);
            v[2] = two_way(gp, ORD_RD).before(gp.ntl);
            v[3] = gp.ntl;
            v[4] = (long long)gp.ntl * gp.n_kc;
            v[5] = (long long)gp.ntl * gp.n_units;
            v[6] = (long long)gp.n_kc * gp.R * gp.count;
        }
        long long incl[7];
#pragma unroll
        for (int k = 0; k < 7; ++k) incl[k] = warp_inclusive(v[k]);
        if (g < G) {
            GroupPos &q = ps.pos[g];
            q.sh = (int)(run[0] + incl[0] - v[0]);
            q.ex = (int)(run[1] + incl[1] - v[1]);
            q.rd = (int)(run[2] + incl[2] - v[2]);
            q.t = (int)(run[3] + incl[3] - v[3]);
            q.c = (int)(run[4] + incl[4] - v[4]);
            q.u = (int)(run[5] + incl[5] - v[5]);
            q.P = (int)(run[6] + incl[6] - v[6]);
        }
#pragma unroll
        for (int k = 0; k < 7; ++k) run[k] += __shfl_sync(0xffffffffu, incl[k], 31);
    }
    bad = bad || run[6] > p.partial_cap || run[2] * 16 > p.s_cap || run[2] * 16 >= (1ll << 31);
#pragma unroll
    for (int k = 0; k < 7; ++k) bad = bad || run[k] >= (1ll << 31);
    if (lane == 0) {
        GroupPos &q = ps.pos[bad ? 0 : G];
        q.sh = bad ? 0 : (int)run[0];
        q.ex = bad ? 0 : (int)run[1];
        q.rd = bad ? 0 : (int)run[2];
        q.t = bad ? 0 : (int)run[3];
        q.c = bad ? 0 : (int)run[4];
        q.u = bad ? 0 : (int)run[5];
        q.P = bad ? 0 : (int)run[6];
        ps.G = bad ? 0 : G;
        ps.bad = bad;
        ps.target = target;
        tstamp(p, 0, 11);
    }
}

// The record of tile t (t < the launch's tiles).
__device__ TileRec plan_tile(const StreamParams &p, const PlanSmem &ps, int t)
{
    const int g = find_group(ps, -1, t);
    const GroupPos &q = ps.pos[g];
    const GroupPlan gp = load_group_plan(p, ps, g);
    const int i = t - q.t, m = gp.base + (i < gp.rem ? 1 : 0);
    TileRec r;
    r.a = gp.a;
    r.e = gp.e;
    r.row0 = gp.row_off + i * gp.base + min(i, gp.rem);
    r.m = m;
    r.rp = gp.rp;
    r.R = gp.R;
    r.n_pad = npad16(m);
    r.kc = gp.kc;
    r.n_kc = gp.n_kc;
    r.ks = gp.ks;
    r.W = gp.W;
    r.n_units = gp.n_units;
    r.p_off = q.P + TwoWay{gp.n_kc * gp.R * (gp.base + 1), gp.n_kc * gp.R * gp.base, gp.rem}.before(i);
    r.s_off = 16 * (q.rd + two_way(gp, ORD_RD).before(i));
    r.c0 = q.c + i * gp.n_kc;
    r.u0 = q.u + i * gp.n_units;
    return r;
}

// The first (tile, item) at or past position lo of an order (the launch's end when lo is past the last).
__device__ int2 plan_start(const StreamParams &p, const PlanSmem &ps, int order, int lo)
{
    const GroupPos &end = ps.pos[ps.G];
    if (lo >= gpos_field(end, order)) return make_int2(end.t, 0);
    const int g = find_group(ps, order, lo);
    const GroupPos &q = ps.pos[g];
    const GroupPlan gp = load_group_plan(p, ps, g);
    const TwoWay tw = two_way(gp, order);
    const int off = lo - gpos_field(q, order);
    const int i = tw.find(off), m = gp.base + (i < gp.rem ? 1 : 0);
    int per, n;
    if (order == ORD_SH) {
        per = chunk_cost(gp.kc, gp.R, m);
        n = gp.n_kc;
    } else if (order == ORD_EX) {
        per = unit_cost(gp.W, gp.rp, m);
        n = gp.n_units;
    } else {
        per = 1;
        n = gp.R * npad16(m) / 8;
    }
    const int j = (off - tw.before(i) + per - 1) / per;
    const int t = q.t + i;
    return j >= n ? make_int2(t + 1, 0) : make_int2(t, j);
}

// ===========================================================================
// shrink
// ===========================================================================
// A group of gs threads (gt: this thread's index in it) copies P 16-byte pieces of each of m rows into
// shared memory, as cp.async: row r's pieces are read from src(r) and land at dst + r * stride.  With
// P <= gs a thread keeps one piece column and steps over rows (gs / P rows per step); otherwise the group
// walks the pieces of one row at a time.  The iterations are independent, so the source-row lookups of
// several rows are in flight together.  One warp issuing alone leaves the gather far below the memory's
// rate, hence groups of several warps.  Piece c of row r lands at dst + r * rstride + c * cstride.
template <class Src>
__device__ __forceinline__ void group_gather(unsigned char *dst, int rstride, int cstride, int m, int P, int gt, int gs,
                                             Src src)
{
    if (P <= gs) {
        const int rpi = gs / P, rsub = gt / P, c = gt - rsub * P;
        if (rsub < rpi) {
#pragma unroll 4
            for (int r = rsub; r < m; r += rpi) tc::cp_async16(dst + r * rstride + c * cstride, src(r) + c * 8, true);
        }
    } else {
        for (int r = 0; r < m; ++r) {
            const __nv_bfloat16 *g = src(r);
#pragma unroll 2
            for (int c = gt; c < P; c += gs) tc::cp_async16(dst + r * rstride + c * cstride, g + c * 8, true);
        }
    }
}

// The x rows of a shrink stage, [ks/8][n_pad][8]: each warp of the group takes blocks of 8 rows x 4 pieces
// (lanes 8 q .. 8 q + 7: piece 4 b + q of rows 8 a .. 8 a + 7), so every 8 lanes fill 128 contiguous bytes of
// shared memory and every row's 4 pieces are 64 contiguous bytes of x.
template <class Src>
__device__ __forceinline__ void x_gather(unsigned char *dst, int n_pad, int m, int P, int gt, Src src)
{
    constexpr int warps = kShProd / 32;
    const int lane = gt & 31, w = gt >> 5, l8 = lane & 7, q = lane >> 3;
    const int nrb = (m + 7) >> 3, npq = (P + 3) >> 2;
    int rb = w, pq = 0;
    while (rb >= nrb && pq < npq) {
        rb -= nrb;
        ++pq;
    }
    for (; pq < npq;) {
        const int r = rb * 8 + l8, c = pq * 4 + q;
        if (r < m && c < P) tc::cp_async16(dst + (c * n_pad + r) * 16, src(r) + c * 8, true);
        rb += warps;
        while (rb >= nrb && pq < npq) {
            rb -= nrb;
            ++pq;
        }
    }
}

struct __align__(128) ShrinkSmem {
    union {
        // stage: A columns [ks/8][R][8], then the same K columns of the tile's x rows [ks/8][n_pad][8]
        unsigned char stage[kShStages][kShStageBytes];
        PlanSmem plan;   // while the block plans, before the streams start
    };
    // an A operand of fewer than 128 (or 256) rows is read as 128 (256) rows: the rows past R, which only
    // reach accumulator lanes nobody reads, come from the bytes after the stage's copied A columns (later
    // A columns or the x rows, inside the stage); the pad keeps even the last stage's reads inside the block
    unsigned char pad[2048];
    uint64_t full[kShStages], empty[kShStages];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int32_t xsrc[2][kTileRows];   // source rows of the producers' tiles, by tile parity
    TileRec mytile[kMyTiles];     // records of the tiles of this block's chunks (when they are few enough)
    int2 smeta[kShStages];        // the (tile, chunk) of every stage; tile -1 ends the sequence
    int2 range[2];                // this block's first and end (tile, chunk)
    int32_t flag;
};

// Walks this block's chunks (tile, chunk) in order; the tile record is reloaded when the tile changes.
struct ChunkWalk {
    int t, j, cur;
    int2 end;
    const TileRec *mine;   // the block's own records, tile b0.x first (null: read the launch's records)
    int t_base;
    TileRec tr;
    __device__ __forceinline__ ChunkWalk(int2 b0, int2 b1, const TileRec *mine_)
        : t(b0.x), j(b0.y), cur(-1), end(b1), mine(mine_), t_base(b0.x) {}
    __device__ __forceinline__ bool valid(const StreamParams &p)
    {
        if (!before(t, j, end)) return false;
        if (t != cur) {
            tr = mine ? mine[t - t_base] : load_tile(p.tiles + t);
            cur = t;
        }
        return true;
    }
    __device__ __forceinline__ void next()
    {
        if (++j == tr.n_kc) {
            ++t;
            j = 0;
        }
    }
};

// Warps 8-11 (kShProd threads): the block's chunks, stage by stage, into the ring, then an end mark.  Thread
// 0 of the group copies a stage's A columns (one bulk copy) and writes its (tile, chunk); the group gathers
// the same K columns of the tile's x rows as 16-byte cp.async pieces into the operand layout
// [ks/8][n_pad][8].  A stage whose K columns end with a group of 8 gets zeros for the other 8 columns of
// its last K=16 step (A and x).  The stage's full barrier completes once the bulk copy's bytes and every
// producer thread's pieces have landed.  One barrier per stage keeps
// the four warps in step (and lets them leave together when a wait runs out); the tile's source rows are
// double-buffered by tile parity, so a warp may write the next tile's rows while another still gathers the
// last stage of the previous tile.
__device__ __forceinline__ void shrink_produce(const StreamParams &p, ShrinkSmem &sm, int2 b0, int2 b1,
                                               const TileRec *mine)
{
    const int gt = threadIdx.x - 32 * kShWarps, lane = threadIdx.x & 31;
    uint32_t s = 0;
    int cur = -1, par = 1;
    // the next free stage for every producer thread (false: a wait ran out, and the group stops)
    auto next_slot = [&]() -> bool {
        bool got = true;
        if (s >= kShStages) {
            if (lane == 0)
                got = mbar_wait_suspend(&sm.empty[s % kShStages], ((s / kShStages) - 1) & 1, p.timeout_ns, p.err);
            got = __shfl_sync(0xffffffffu, got, 0);
        }
        return got;
    };
    // every stage of chunk j of tile t
    auto stage_chunk = [&](int t, int j, const TileRec &tr) -> bool {
        bool fresh = false;
        if (t != cur) {
            cur = t;
            par ^= 1;
            fresh = true;
        }
        const unsigned char *ablk =
            reinterpret_cast<const unsigned char *>(__ldg(p.a_ptr + tr.a * p.E_A + (p.E_A == 1 ? 0 : tr.e)));
        const int k0 = j * tr.kc, kend = min(k0 + tr.kc, p.K);
        const int xoff = tr.R * tr.ks * 2;
        for (int kb = k0; kb < kend; kb += tr.ks, ++s) {
            const int slot = s % kShStages;
            const bool got = next_slot();
            const int kk = min(tr.ks, kend - kb);
            if (gt == 0 && got) {   // the A copy needs nothing the group writes: it leaves first
                const uint32_t bytes = (uint32_t)tr.R * kk * 2;
                sm.smeta[slot] = make_int2(t, j);
                mbar_arrive_expect_tx(&sm.full[slot], bytes);
                bulk_g2s(sm.stage[slot], ablk + (size_t)(kb / 8) * tr.R * 16, bytes, &sm.full[slot]);
                if (s < 8) tstamp(p, 0, 12 + s);
            }
            if (fresh) {
                for (int r = gt; r < tr.m; r += kShProd) sm.xsrc[par][r] = __ldcg(p.rows + tr.row0 + r) / p.src_div;
                fresh = false;
            }
            if (!bar_and(2, kShProd, got)) return false;
            const __nv_bfloat16 *xk = p.x + kb;
            const int64_t ldx = p.ldx;
            const int32_t *xs = sm.xsrc[par];
            unsigned char *xd = sm.stage[slot] + xoff;
            x_gather(xd, tr.n_pad, tr.m, kk >> 3, gt, [&](int r) { return xk + (int64_t)xs[r] * ldx; });
            if (kk & 8) {   // zero-filling copies (no bytes read)
                for (int i = gt; i < tr.R; i += kShProd) tc::cp_async16(sm.stage[slot] + ((kk >> 3) * tr.R + i) * 16, xk, false);
                for (int i = gt; i < tr.n_pad; i += kShProd) tc::cp_async16(xd + ((kk >> 3) * tr.n_pad + i) * 16, xk, false);
            }
            tc::cp_async_arrive_noinc(&sm.full[slot]);
        }
        return true;
    };
    bool ok = true;
    for (ChunkWalk w(b0, b1, mine); ok && w.valid(p); w.next()) ok = stage_chunk(w.t, w.j, w.tr);
    // the end mark: a stage with tile -1
    if (ok && bar_and(2, kShProd, next_slot())) {
        if (gt == 0) sm.smeta[s % kShStages] = make_int2(-1, 0);
        bar_sync(2, kShProd);
        if (gt == 0) mbar_arrive(&sm.full[s % kShStages]);
        mbar_arrive(&sm.full[s % kShStages]);
        ++s;
    }
    if (gt == 0)
        for (uint32_t q = s > kShStages ? s - kShStages : 0; q < s; ++q)
            mbar_wait_suspend(&sm.full[q % kShStages], (q / kShStages) & 1, p.timeout_ns, p.err);
    tc::cp_async_wait_all();
}

// Half h & 1 of S chunk h >> 1 of a tile (S chunk i: 16 bytes of its S layout, slice block sb, rank group kg,
// row; a half: 4 of those rank columns): the tile's partials of those columns summed in chunk order, rounded
// once to bf16.  S is stored per slice block sb as [rp / 8][n_pad][8], the operand layout the expand reads;
// rows past m are zero.
__device__ __forceinline__ void reduce_s_half(const StreamParams &p, const TileRec &tr, int h)
{
    constexpr int kBatch = 16;   // chunks whose loads are in flight together
    const int i = h >> 1, half = h & 1;
    const int per_sb = (tr.rp >> 3) * tr.n_pad;
    const int sb = i / per_sb, rem = i - sb * per_sb;
    const int kg = rem / tr.n_pad, row = rem - kg * tr.n_pad;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (row < tr.m) {
        const float *q = p.partials + tr.p_off + row * tr.R + sb * tr.rp + kg * 8 + half * 4;
        const int64_t cstride = (int64_t)tr.m * tr.R;
        for (int c0 = 0; c0 < tr.n_kc; c0 += kBatch, q += kBatch * cstride) {
            float4 u[kBatch];
#pragma unroll
            for (int c = 0; c < kBatch; ++c)
                u[c] = c0 + c < tr.n_kc ? __ldcg(reinterpret_cast<const float4 *>(q + c * cstride))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBatch; ++c) {
                if (c0 + c < tr.n_kc) {
                    a[0] += u[c].x; a[1] += u[c].y; a[2] += u[c].z; a[3] += u[c].w;
                }
            }
        }
    }
    __align__(8) __nv_bfloat16 o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __float2bfloat16_rn(a[e]);
    *reinterpret_cast<uint2 *>(p.s_area + tr.s_off + (int64_t)i * 16 + half * 8) = *reinterpret_cast<const uint2 *>(o);
}

// Warp 0, one thread: the stages the producers announce, until the end mark.  Each chunk accumulates into
// one of two tensor-memory accumulators (in turn): D[r][n] = sum over the chunk's K columns of A[r][k] x[n][k],
// the A block's rows as the 128-row M operand (two blocks of 128 rows when R > 128) and the tile's rows,
// rounded up to 16, as N.  A stage is released by the commit after its MMAs; a chunk's accumulator goes to
// the epilogue with the commit after its last stage.  Within a chunk the MMAs run in K order, so a
// partial's sums depend on the chunk cut alone.
__device__ __forceinline__ void shrink_mma(const StreamParams &p, ShrinkSmem &sm, int2 b0, const TileRec *mine,
                                           int n_my)
{
    uint32_t s = 0;
    int ci = -1, cur_t = -1, cur_j = -1, kb = 0, kend = 0;
    TileRec tr{};
    for (;; ++s) {
        const int slot = s % kShStages;
        if (!mbar_wait_suspend(&sm.full[slot], (s / kShStages) & 1, p.timeout_ns, p.err)) break;
        const int2 e = sm.smeta[slot];
        if (e.x != cur_t || e.y != cur_j) {   // a chunk ends here (or the sequence does)
            if (ci >= 0) tc::mma_commit(&sm.acc_full[ci & 1]);
            if (e.x < 0) break;
            ++ci;
            if (ci >= 2 && !mbar_wait_suspend(&sm.acc_empty[ci & 1], ((ci >> 1) - 1) & 1, p.timeout_ns, p.err)) break;
            if (e.x != cur_t) tr = mine && e.x - b0.x < n_my ? mine[e.x - b0.x] : load_tile(p.tiles + e.x);
            cur_t = e.x;
            cur_j = e.y;
            kb = e.y * tr.kc;
            kend = min(kb + tr.kc, p.K);
        }
        tc::fence_proxy_async_smem();   // the producers' cp.async pieces, seen through the barrier, to the tensor core
        tc::fence_after_sync();
        const int nk = (min(tr.ks, kend - kb) + 15) >> 4;
        const uint32_t a_s = smem_u32(sm.stage[slot]), x_s = a_s + tr.R * tr.ks * 2;
        const uint32_t idesc = tc::idesc_bf16(128, tr.n_pad);
        const uint32_t d = sm.tmem_base + (ci & 1) * kShAccCols;
        // descriptors advance by their start-address field (16-byte units; stays below 2^14 in shared memory)
        uint64_t ad = tc::smem_desc(a_s, tr.R * 16, 128), xd = tc::smem_desc(x_s, tr.n_pad * 16, 128);
        const uint64_t astep = (uint64_t)(tr.R * 2), xstep = (uint64_t)(tr.n_pad * 2);
        uint32_t acc = kb == cur_j * tr.kc ? 0u : 1u;   // the chunk's first K step starts the accumulator
        if (tr.R <= 128) {
            for (int k = 0; k < nk; ++k, ad += astep, xd += xstep, acc = 1u) tc::mma_bf16(d, ad, xd, idesc, acc);
        } else {   // two 128-row blocks of A, 128 rows (2048 bytes, 128 units) apart
            for (int k = 0; k < nk; ++k, ad += astep, xd += xstep, acc = 1u) {
                tc::mma_bf16(d, ad, xd, idesc, acc);
                tc::mma_bf16(d + tr.n_pad, ad + 128, xd, idesc, acc);
            }
        }
        kb += min(tr.ks, kend - kb);
        tc::mma_commit(&sm.empty[slot]);   // the stage is free once these MMAs are done
        if (s < 8) tstamp(p, 0, 20 + s);
    }
    // every MMA issued is done before the tensor memory is freed
    if (s > 0) {
        tc::mma_commit(&sm.drain);
        mbar_wait_suspend(&sm.drain, 0, p.timeout_ns, p.err);
    }
}

// Warps 4-7: every chunk's accumulator, in the block's chunk order, to the tile's partial slot [m][R] (fp32):
// thread (quarter q, lane) reads tensor-memory lane 32 q + lane of each 128-row block (A row r) for the
// tile's rows; then the chunk counts on its tile (the expand sums a tile's S once all its chunks are counted).
__device__ __forceinline__ void shrink_epilogue(const StreamParams &p, ShrinkSmem &sm, int2 b0, int2 b1,
                                                const TileRec *mine)
{
    const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3, et = threadIdx.x - 128;
    int ci = 0;
    for (ChunkWalk w(b0, b1, mine); w.valid(p); w.next(), ++ci) {
        const int b = ci & 1;
        if (!bar_and(3, 128, mbar_wait_suspend(&sm.acc_full[b], (ci >> 1) & 1, p.timeout_ns, p.err))) break;
        tc::fence_after_sync();
        const TileRec &tr = w.tr;
        float *dst = p.partials + tr.p_off + (int64_t)w.j * tr.m * tr.R;
        for (int mb = 0; mb * 128 < tr.R; ++mb) {
            const int r = mb * 128 + q * 32 + lane;
            const uint32_t ta = sm.tmem_base + ((uint32_t)(q * 32) << 16) + b * kShAccCols + mb * tr.n_pad;
            for (int n0 = 0; n0 < tr.n_pad; n0 += 16) {
                float v[16];
                tc::tmem_ld16(ta + n0, v);
                if (r < tr.R) {
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        if (n0 + n < tr.m) dst[(n0 + n) * tr.R + r] = v[n];
                }
            }
        }
        tc::fence_before_sync();
        bar_sync(3, 128);   // the partial is out of the accumulator and stored
        if (et == 0) {
            mbar_arrive(&sm.acc_empty[b]);
            if (ci < 4) tstamp(p, 0, 3 + ci);
            __threadfence();   // every thread's stores (ordered by the barrier) before the count
            atomicAdd(p.tile_cnt + w.t, 1);
        }
    }
}

__global__ void __launch_bounds__(kShThreads, 1) shrink_kernel(const __grid_constant__ StreamParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ShrinkSmem &sm = *reinterpret_cast<ShrinkSmem *>(smem_raw);
    const int tid = threadIdx.x;
    if (tid == 0) {
        tstamp(p, 0, 0);
        for (int s = 0; s < kShStages; ++s) {
            mbar_init(&sm.full[s], 1 + kShProd);   // the A copy's expect-tx arrival and one per producer thread
            mbar_init(&sm.empty[s], 1);            // the MMA issuer's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);         // the MMA issuer's commit
            mbar_init(&sm.acc_empty[b], 1);        // the epilogue
        }
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();      // the segment table of the build, and everything before it
    if (tid == 0) tstamp(p, 0, 1);
    if (blockIdx.x == 0 && tid == 0) *p.ex_claim = 0;   // the expand of the launch before has ended
    if (tid < 32) plan_groups(p, sm.plan);
    else if (tid < 64) tc::tmem_alloc(&sm.tmem_base, 2 * kShAccCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // the expand may launch now; it waits for this grid's records before it reads anything.  This block holds
    // its tensor memory already, so an expand block (which takes all of an SM's tensor memory) never gets it
    // first on a shared SM and then waits on this block's chunks
    pdl_trigger();
    const PlanSmem &ps = sm.plan;
    const GroupPos &tot = ps.pos[ps.G];
    const int G = p.grid_s, c = blockIdx.x, nt = tot.t;
    // this block's chunks (threads 0 and 32), then the records of their tiles (warp 0); the other warps write
    // this block's share of the launch's plan, read by the expand: the records of tiles c, c + G, ..., the
    // first (tile, S chunk) of expand block c's S sums and the first unit of expand block c
    const Split ss(tot.sh, G);
    if (tid == 0) sm.range[0] = plan_start(p, ps, ORD_SH, ss.start(c));
    if (tid == 32) sm.range[1] = plan_start(p, ps, ORD_SH, ss.start(c + 1));
    if (tid >= 64)
        for (int t = c + G * (tid - 64); t < nt; t += G * (blockDim.x - 64)) p.tiles[t] = plan_tile(p, ps, t);
    if (tid == 64) {   // the first (tile, S chunk) of expand block c's share of the S sums
        const Split sr(tot.rd, p.grid_e);
        p.rd_start[c] = plan_start(p, ps, ORD_RD, sr.start(c));
        if (c == G - 1)
            for (int k = G; k <= p.grid_e; ++k) p.rd_start[k] = plan_start(p, ps, ORD_RD, sr.start(k));
    }
    if (tid == 96) {
        // the expand splits all but the last 1 / kExPoolDiv of its cost ahead of time and claims the units
        // of that tail one by one (its claims look tiles up in a copy of u0 that holds kExUposCap tiles)
        const Split se(nt <= kExUposCap ? tot.ex - tot.ex / kExPoolDiv : tot.ex, p.grid_e);
        p.ex_start[c] = plan_start(p, ps, ORD_EX, se.start(c));
        if (c == G - 1) {
            const int2 b = plan_start(p, ps, ORD_EX, se.start(p.grid_e));
            p.ex_start[p.grid_e] = b;
            p.plan_hdr[PL_POOL_U] = (b.x < nt ? plan_tile(p, ps, b.x).u0 : tot.u) + b.y;
        }
    }
    if (c == 0 && tid == 128) {
        p.plan_hdr[PL_TILES] = nt;
        p.plan_hdr[PL_UNITS] = tot.u;
        if (ps.bad) atomicOr(p.err, kErrWorkspace);
    }
    __syncthreads();
    const int2 b0 = sm.range[0], b1 = sm.range[1];
    const int n_my = b1.x - b0.x + (b1.y > 0 ? 1 : 0);
    const TileRec *mine = n_my <= kMyTiles ? sm.mytile : nullptr;
    if (mine && tid < n_my) sm.mytile[tid] = plan_tile(p, ps, b0.x + tid);
    __syncthreads();   // the block's records are in; the stages may overwrite the plan now
    if (tid == 0) {
        // this block's share of the launch's plan is out: its first arrival on the grid counter (thread 0 would
        // wait for its first stage anyway)
        tstamp(p, 0, 2);
        __threadfence();
        atomicAdd(p.cnt, 1);
        // a block with more tiles than it keeps reads the launch's records, once every block has written its share
        sm.flag = 1;
        if (!mine) {
            const uint64_t t0 = globaltimer();
            while (ld_acquire_gpu(p.cnt) < G) {
                if (globaltimer() - t0 > p.timeout_ns) {
                    atomicOr(p.err, kErrTimeout);
                    sm.flag = 0;
                    break;
                }
                nanosleep_ns(32);
            }
            __threadfence();
        }
    }
    bool go = true;
    if (!mine) {   // block-uniform
        __syncthreads();
        go = sm.flag != 0;
    }
    const int warp = tid >> 5;
    if (go) {
        if (warp == 0) {
            if (tid == 0) shrink_mma(p, sm, b0, mine, n_my);
        } else if (warp >= 4 && warp < kShWarps) {
            shrink_epilogue(p, sm, b0, b1, mine);
        } else if (warp >= kShWarps) {
            shrink_produce(p, sm, b0, b1, mine);
        }
        __syncwarp();
        if (tid == 128) tstamp(p, 0, 8);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(sm.tmem_base, 2 * kShAccCols);
    }
    if (tid == 0) tstamp(p, 0, 31);
}

// ===========================================================================
// expand
// ===========================================================================
// A unit's B columns in a B stage (for the MMA issuer) and its y rows in a y slot (for the epilogue), each
// described by the warp that filled it.
struct ExBMeta {
    int32_t t, sb, n_pad, rp, w_eff;
};
struct __align__(16) ExYMeta {
    float f[kTileRows];       // scale * row weight (read as float4)
    int32_t row[kTileRows];   // y row of every tile row
    int32_t W, m, w_eff, n_pad, col;
};

struct __align__(1024) ExpandSmem {
    unsigned char bstage[kExBStages][kExBBytes];     // B tiles [W/128][rp/8][128][8]
    unsigned char ystage[kExYStages][kExYBytes];     // y rows [m][W]
    unsigned char sbuf[2][kExSBytes];                // S of one (tile, slice block): [rp/8][n_pad][8]
    ExBMeta bmeta[kExBStages];
    ExYMeta ymeta[kExYStages];
    uint64_t full_b[kExBStages], empty_b[kExBStages];
    uint64_t full_y[kExYStages], empty_y[kExYStages];
    uint64_t s_full[2], s_empty[2];
    uint64_t acc_full[kExAcc], acc_empty[kExAcc];
    uint64_t drain;                                  // the MMA issuer's last MMAs are done
    int2 uq[kExQ];                                   // unit queue: (tile, unit), tile -1 ends the sequence
    uint64_t uq_full[kExQ], uq_empty[kExQ];
    uint64_t u0_ready;
    int32_t u0[kExUposCap + 1];                      // first unit of every tile, then the launch's unit count
    int32_t nt;
    int32_t flag, rd_ok;
    uint32_t tmem_base;
};

// Slice and column block of unit u of a tile whose units are W columns wide.
__device__ __forceinline__ void unit_slice(const StreamParams &p, int W, int u, int &s, int &cb)
{
    s = 0;
    for (; s < p.n_slices - 1; ++s) {
        const int c = (p.slice_n[s] + W - 1) / W;
        if (u < c) break;
        u -= c;
    }
    cb = u;
}

// Walks this block's units in order; the tile record is reloaded when the tile changes.
struct UnitWalk {
    int t, u;
    int2 end;
    int cur;
    TileRec tr;
    __device__ __forceinline__ UnitWalk(int2 b0, int2 b1) : t(b0.x), u(b0.y), end(b1), cur(-1) {}
    __device__ __forceinline__ bool valid(const StreamParams &p)
    {
        if (!before(t, u, end)) return false;
        if (t != cur) {
            tr = load_tile(p.tiles + t);
            cur = t;
        }
        return true;
    }
    __device__ __forceinline__ void next()
    {
        if (++u == tr.n_units) {
            ++t;
            u = 0;
        }
    }
};

// The unit sequence of a block: its share of the units split ahead of time, then units of the launch's
// tail claimed one at a time, so that blocks that ran ahead take more of the tail.  Warp 0 (the leader)
// walks it and hands every unit on: to the y producers and the S loader through the unit queue, to the MMA
// issuer with the unit's B columns; the y producers hand it to the epilogue with the unit's y rows.  The
// end of the sequence travels the same ways, as tile -1.

// Tile l with u0[l] <= g < u0[l + 1].
__device__ __forceinline__ int find_tile(const int32_t *u0, int nt, int g)
{
    int l = 0, h = nt;
    while (h - l > 1) {
        const int mid = (l + h) >> 1;
        if (u0[mid] <= g) l = mid;
        else h = mid;
    }
    return l;
}

// Warp 0, one thread: the unit sequence into the unit queue, and the packed B columns of every unit (one
// bulk copy each) into the B ring with the unit's description for the MMA issuer.
__device__ __forceinline__ void expand_lead(const StreamParams &p, ExpandSmem &sm, int2 b0, int2 b1)
{
    uint32_t i = 0;
    const unsigned char *bblk = nullptr;
    int blk_t = -1;
    auto emit = [&](int t, int u, const TileRec &tr) -> bool {
        const int q = i % kExQ;
        if (i >= kExQ && !mbar_wait_suspend(&sm.uq_empty[q], ((i / kExQ) - 1) & 1, p.timeout_ns, p.err))
            return false;
        sm.uq[q] = make_int2(t, u);
        mbar_arrive(&sm.uq_full[q]);
        const int slot = i % kExBStages;
        if (i >= kExBStages &&
            !mbar_wait_suspend(&sm.empty_b[slot], ((i / kExBStages) - 1) & 1, p.timeout_ns, p.err))
            return false;
        ++i;
        ExBMeta &mt = sm.bmeta[slot];
        mt.t = t;
        if (t < 0) {
            mbar_arrive(&sm.full_b[slot]);
            return true;
        }
        if (blk_t != t) {
            bblk = reinterpret_cast<const unsigned char *>(__ldg(p.b_ptr + tr.a * p.E_B + (p.E_B == 1 ? 0 : tr.e)));
            blk_t = t;
        }
        int s, cb;
        unit_slice(p, tr.W, u, s, cb);
        const int w_eff = min(tr.W, p.slice_n[s] - cb * tr.W);
        mt.sb = p.n_a == 1 ? 0 : s;
        mt.n_pad = tr.n_pad;
        mt.rp = tr.rp;
        mt.w_eff = w_eff;
        const uint32_t bbytes = (uint32_t)((w_eff + 127) >> 7) * tr.rp * 256;
        if (i - 1 >= 8 && i - 1 < 12) tstamp(p, 1, 13 + (i - 1 - 8));
        mbar_arrive_expect_tx(&sm.full_b[slot], bbytes);
        bulk_g2s(sm.bstage[slot], bblk + (size_t)(p.slice_tile_off[s] + cb * (tr.W >> 7)) * tr.rp * 256, bbytes,
                 &sm.full_b[slot]);
        return true;
    };
    bool ok = true;
    TileRec tr{};
    for (UnitWalk w(b0, b1); ok && w.valid(p); w.next()) ok = emit(w.t, w.u, w.tr);
    const int U = __ldcg(p.plan_hdr + PL_UNITS), g0 = __ldcg(p.plan_hdr + PL_POOL_U);
    if (ok && g0 < U) {
        ok = mbar_wait_suspend(&sm.u0_ready, 0, p.timeout_ns, p.err);
        const int nt = sm.nt;
        int g = ok ? g0 + atomicAdd(p.ex_claim, 1) : U, cur = -1;
        while (ok && g < U) {
            const int gn = g0 + atomicAdd(p.ex_claim, 1);   // the next claim's round trip overlaps this unit
            const int t = find_tile(sm.u0, nt, g);
            if (t != cur) {
                tr = load_tile(p.tiles + t);
                cur = t;
            }
            ok = emit(t, g - sm.u0[t], tr);
            g = gn;
        }
    }
    emit(-1, 0, tr);
    for (uint32_t q = i > kExBStages ? i - kExBStages : 0; q < i; ++q)
        mbar_wait_suspend(&sm.full_b[q % kExBStages], (q / kExBStages) & 1, p.timeout_ns, p.err);
}

// Warps 4-7 (kExYProd threads): for every unit of the queue, its y rows (16-byte cp.async pieces over the
// group) and its description into the next y slot; at the end of the sequence one end mark (m = -1) per
// epilogue group.  One barrier per unit keeps the four warps in step (and lets them leave together when a
// wait runs out).
__device__ __forceinline__ void expand_produce_y(const StreamParams &p, ExpandSmem &sm)
{
    const int gt = threadIdx.x - 128, lane = threadIdx.x & 31;
    uint32_t i = 0;
    int cur = -1;
    TileRec tr{};
    int yr = 0;      // y row gt of the current tile (gt < m) and its factor
    float yf = 0.f;
    bool live = true;
    for (;; ++i) {
        const int q = i % kExQ;
        bool got = true;
        if (lane == 0) got = mbar_wait_suspend(&sm.uq_full[q], (i / kExQ) & 1, p.timeout_ns, p.err);
        got = __shfl_sync(0xffffffffu, got, 0);
        const int2 e = sm.uq[q];
        const bool end = !got || e.x < 0;
        const int slot = i % kExYStages;
        int col = 0, w_eff = 0;
        if (!end) {
            if (i >= kExYStages) {
                if (lane == 0) got = mbar_wait_suspend(&sm.empty_y[slot], ((i / kExYStages) - 1) & 1, p.timeout_ns, p.err);
                got = __shfl_sync(0xffffffffu, got, 0);
            }
            if (e.x != cur) {
                tr = load_tile(p.tiles + e.x);
                const float sc = __ldg(p.scale + tr.a);
                yr = gt < tr.m ? __ldcg(p.rows + tr.row0 + gt) : 0;
                yf = p.row_weight ? sc * __ldg(p.row_weight + yr) : sc;
                cur = e.x;
            }
            int s, cb;
            unit_slice(p, tr.W, e.y, s, cb);
            w_eff = min(tr.W, p.slice_n[s] - cb * tr.W);
            col = p.slice_off[s] + cb * tr.W;
            if (got) {
                ExYMeta &mt = sm.ymeta[slot];
                if (gt < tr.m) {
                    mt.row[gt] = yr;
                    mt.f[gt] = yf;
                }
                if (gt == 0) {
                    mt.W = tr.W;
                    mt.m = tr.m;
                    mt.w_eff = w_eff;
                    mt.n_pad = tr.n_pad;
                    mt.col = col;
                }
            }
        }
        // every thread has read the entry; the slot is free for the whole group and its rows are written
        if (!bar_and(5, kExYProd, got)) {
            live = false;
            break;
        }
        if (gt == 0) mbar_arrive(&sm.uq_empty[q]);
        if (end) break;
        const __nv_bfloat16 *yc = p.y + col;
        const int64_t ldy = p.ldy;
        const ExYMeta &mt = sm.ymeta[slot];
        if (i >= 8 && i < 12 && gt == 0) tstamp(p, 1, 17 + (i - 8));
        group_gather(sm.ystage[slot], tr.W * 2, 16, tr.m, w_eff >> 3, gt, kExYProd,
                     [&](int r) { return yc + (int64_t)mt.row[r] * ldy; });
        tc::cp_async_arrive_noinc(&sm.full_y[slot]);   // once every piece of this thread has landed
    }
    for (int k = 0; live && k < kExGroups; ++k, ++i) {   // an end mark for each epilogue group
        const int slot = i % kExYStages;
        bool got = true;
        if (i >= kExYStages) {
            if (lane == 0) got = mbar_wait_suspend(&sm.empty_y[slot], ((i / kExYStages) - 1) & 1, p.timeout_ns, p.err);
            got = __shfl_sync(0xffffffffu, got, 0);
        }
        if (got && gt == 0) sm.ymeta[slot].m = -1;
        if (!bar_and(5, kExYProd, got)) break;
        mbar_arrive(&sm.full_y[slot]);
    }
    tc::cp_async_wait_all();
}

// Warp 1, one thread: S of every (tile, slice block) the unit queue meets, into two buffers in rotation, each
// tile's once every S chunk of the tile is summed.
__device__ __forceinline__ void expand_load_s(const StreamParams &p, ExpandSmem &sm)
{
    uint32_t k = 0;
    int prev_t = -1, prev_sb = -1, cur = -1, ready = -1;
    TileRec tr{};
    for (uint32_t i = 0;; ++i) {
        const int q = i % kExQ;
        if (!mbar_wait_suspend(&sm.uq_full[q], (i / kExQ) & 1, p.timeout_ns, p.err)) break;
        const int2 e = sm.uq[q];
        mbar_arrive(&sm.uq_empty[q]);
        if (e.x < 0) break;
        if (e.x != cur) {
            tr = load_tile(p.tiles + e.x);
            cur = e.x;
        }
        int s, cb;
        unit_slice(p, tr.W, e.y, s, cb);
        const int sb = p.n_a == 1 ? 0 : s;
        if (e.x == prev_t && sb == prev_sb) continue;
        if (e.x != ready && !p.withhold) {
            if (!wait_at_least(p, p.s_done + e.x, tr.R * tr.n_pad / 8)) break;
            __threadfence();
            tc::fence_proxy_async_global();   // S was written by threads; the bulk copies read it
            ready = e.x;
        }
        const int slot = k & 1;
        if (k >= 2 && !mbar_wait_suspend(&sm.s_empty[slot], ((k >> 1) - 1) & 1, p.timeout_ns, p.err)) break;
        if (k == 0) tstamp(p, 1, 3);
        const uint32_t bytes = (uint32_t)tr.rp * tr.n_pad * 2;
        mbar_arrive_expect_tx(&sm.s_full[slot], bytes);
        if (!p.withhold) bulk_g2s(sm.sbuf[slot], p.s_area + tr.s_off + (size_t)sb * bytes, bytes, &sm.s_full[slot]);
        ++k;
        prev_t = e.x;
        prev_sb = sb;
    }
    if (!p.withhold)
        for (uint32_t q = k > 2 ? k - 2 : 0; q < k; ++q)
            mbar_wait_suspend(&sm.s_full[q & 1], (q >> 1) & 1, p.timeout_ns, p.err);
}

// Warp 2, one thread: D(acc) = B_unit S^T for every unit (M = 128 output columns per B tile, N = the tile's
// rows rounded up to 16, K = the stored rank).
__device__ __forceinline__ void expand_mma(const StreamParams &p, ExpandSmem &sm)
{
    uint32_t i = 0, k = 0;
    int prev_t = -1, prev_sb = -1;
    for (;; ++i) {
        const int slot = i % kExBStages;
        if (!mbar_wait_suspend(&sm.full_b[slot], (i / kExBStages) & 1, p.timeout_ns, p.err)) break;
        const ExBMeta &mt = sm.bmeta[slot];
        const int t = mt.t, sb = mt.sb, n_pad = mt.n_pad, rp = mt.rp, w_eff = mt.w_eff;
        if (t < 0) break;   // the end of the sequence
        if (i == 0) tstamp(p, 1, 2);
        if (i >= 8 && i < 12) tstamp(p, 1, 5 + (i - 8));
        if (t != prev_t || sb != prev_sb) {
            if (k > 0) tc::mma_commit(&sm.s_empty[(k - 1) & 1]);   // the previous S is free once these MMAs end
            if (!mbar_wait_suspend(&sm.s_full[k & 1], (k >> 1) & 1, p.timeout_ns, p.err)) break;
            if (k == 0) tstamp(p, 1, 4);
            ++k;
            prev_t = t;
            prev_sb = sb;
        }
        const int b = i % kExAcc;
        if (i >= kExAcc && !mbar_wait_suspend(&sm.acc_empty[b], ((i / kExAcc) - 1) & 1, p.timeout_ns, p.err)) break;
        if (i >= 8 && i < 12) tstamp(p, 1, 25 + (i - 8));
        tc::fence_after_sync();
        const uint32_t idesc = tc::idesc_bf16(128, n_pad);
        const uint32_t s_addr = smem_u32(sm.sbuf[(k - 1) & 1]);
        const uint32_t b_addr = smem_u32(sm.bstage[slot]);
        const int nq = (w_eff + 127) >> 7, nk = rp >> 4;
        for (int q = 0; q < nq; ++q) {
            for (int kk = 0; kk < nk; ++kk) {
                const uint64_t ad = tc::smem_desc(b_addr + q * rp * 256 + kk * 2 * 2048, 2048, 128);
                const uint64_t bd = tc::smem_desc(s_addr + kk * 2 * n_pad * 16, n_pad * 16, 128);
                tc::mma_bf16(sm.tmem_base + b * kExAccCols + q * n_pad, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
        }
        tc::mma_commit(&sm.acc_full[b]);
        tc::mma_commit(&sm.empty_b[slot]);   // the B columns are free once these MMAs end
    }
    // tensor memory is freed when the block ends: every MMA issued must be done by then
    if (i > 0) {
        tc::mma_commit(&sm.drain);
        mbar_wait_suspend(&sm.drain, 0, p.timeout_ns, p.err);
    }
}

// Warpgroup wg (warps 4 + 4 wg .. 7 + 4 wg) takes units wg, wg + kExGroups, ...  Thread (quarter qw, lane)
// owns output column 32 qw + lane of every 128-column group of a unit: it reads that column's accumulator
// for all rows and adds it into the staged y rows; the rows then leave as 16-byte stores.
__device__ __forceinline__ void expand_epilogue(const StreamParams &p, ExpandSmem &sm, int wg)
{
    const int lane = threadIdx.x & 31, qw = (threadIdx.x >> 5) & 3, et = threadIdx.x & 127;
    const int bar = 1 + wg;
    for (int k = 0;; ++k) {
        const uint32_t i = kExGroups * k + wg;   // the unit's index in the block's sequence
        const int slot = i % kExYStages, b = i % kExAcc;
        if (!bar_and(bar, kExEpi, mbar_wait_suspend(&sm.full_y[slot], (i / kExYStages) & 1, p.timeout_ns, p.err)))
            break;
        const ExYMeta &mt = sm.ymeta[slot];
        const int m = mt.m, W = mt.W, w_eff = mt.w_eff, n_pad = mt.n_pad;
        if (m < 0) break;   // the end of the sequence
        if (!bar_and(bar, kExEpi, mbar_wait_suspend(&sm.acc_full[b], (i / kExAcc) & 1, p.timeout_ns, p.err))) break;
        tc::fence_after_sync();
        __nv_bfloat16 *ys = reinterpret_cast<__nv_bfloat16 *>(sm.ystage[slot]);
        const uint32_t tbase = sm.tmem_base + ((uint32_t)(qw * 32) << 16) + b * kExAccCols;
        const int nq = (w_eff + 127) >> 7;
        for (int j0 = 0; j0 < n_pad; j0 += 32) {
            const int nrow = min(32, m - j0);
            for (int q = 0; q < nq; ++q) {
                const int c = q * 128 + qw * 32 + lane;
                float v[32];
                // the second half re-reads the first when only 16 rows remain (stays inside the accumulator)
                const uint32_t ta = tbase + q * n_pad + j0;
                tc::tmem_ld16x2(ta, j0 + 16 < n_pad ? ta + 16 : ta, v);
                if (c < w_eff) {
                    __nv_bfloat16 *yc = ys + j0 * W + c;
#pragma unroll
                    for (int h = 0; h < 32; h += 8) {
                        if (h < nrow) {
                            // the rows' factors (the same for every thread)
                            const float4 fa = *reinterpret_cast<const float4 *>(&mt.f[(j0 + h) & (kTileRows - 8)]);
                            const float4 fb = *reinterpret_cast<const float4 *>(&mt.f[((j0 + h) & (kTileRows - 8)) + 4]);
                            const float f[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
                            float yv[8];
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) yv[jj] = h + jj < nrow ? __bfloat162float(yc[(h + jj) * W]) : 0.f;
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj)
                                if (h + jj < nrow) yc[(h + jj) * W] = __float2bfloat16_rn(fmaf(f[jj], v[h + jj], yv[jj]));
                        }
                    }
                }
            }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
        bar_sync(bar, kExEpi);   // every column of the unit updated
        const int col = mt.col, cpr = w_eff >> 3;
        const unsigned char *yb = sm.ystage[slot];
        auto store = [&](int row, int c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(yb + row * W * 2 + c * 16);
            *reinterpret_cast<uint4 *>(p.y + (int64_t)mt.row[row] * p.ldy + col + c * 8) = v;
        };
        if ((cpr & (cpr - 1)) == 0) {
            const int sh = __ffs(cpr) - 1;
            for (int q = et; q < (m << sh); q += kExEpi) store(q >> sh, q & (cpr - 1));
        } else {
            for (int q = et; q < m * cpr; q += kExEpi) {
                const int row = q / cpr;
                store(row, q - row * cpr);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty_y[slot]);   // this warp is done with the slot
    }
}

__global__ void __launch_bounds__(kExThreads, 1) expand_kernel(const __grid_constant__ StreamParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ExpandSmem &sm = *reinterpret_cast<ExpandSmem *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tstamp(p, 1, 0);
        for (int s = 0; s < kExBStages; ++s) {
            mbar_init(&sm.full_b[s], 1);
            mbar_init(&sm.empty_b[s], 1);       // the MMA issuer's commit
        }
        for (int s = 0; s < kExYStages; ++s) {
            mbar_init(&sm.full_y[s], kExYProd);   // every y producer thread, once its pieces landed
            mbar_init(&sm.empty_y[s], 4);       // the 4 warps of an epilogue group
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_empty[s], 1);
        }
        for (int s = 0; s < kExAcc; ++s) {
            mbar_init(&sm.acc_full[s], 1);
            mbar_init(&sm.acc_empty[s], 4);
        }
        for (int s = 0; s < kExQ; ++s) {
            mbar_init(&sm.uq_full[s], 1);    // the leader
            mbar_init(&sm.uq_empty[s], 2);   // the S loader and the y producers
        }
        mbar_init(&sm.u0_ready, 1);
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    if (warp == 2) tc::tmem_alloc(&sm.tmem_base, kExTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // The expand starts while the shrink still runs (its blocks take the SMs that shrink blocks leave): it
    // reads the launch's records once every shrink block has written its share (the shrink's first arrival
    // count; the shrink grid is co-resident and never waits on this one), and the S loader waits for each
    // tile's S on its own.  The B and y copies need nothing the shrink writes.
    if (threadIdx.x == 0) {
        sm.flag = wait_at_least(p, p.cnt, p.grid_s);
        __threadfence();
    }
    __syncthreads();
    const bool go = sm.flag != 0;
    const int2 b0 = go ? __ldcg(p.ex_start + blockIdx.x) : make_int2(0, 0);
    const int2 b1 = go ? __ldcg(p.ex_start + blockIdx.x + 1) : make_int2(0, 0);
    if (threadIdx.x == 0) tstamp(p, 1, 1);
    if (!go) {
    } else if (warp == 0) {
        if (lane == 0) expand_lead(p, sm, b0, b1);
    } else if (warp == 1) {
        if (lane == 0) expand_load_s(p, sm);
    } else if (warp == 2) {
        if (lane == 0) expand_mma(p, sm);
    } else if (warp == 3) {
        // the tiles' first units, for the leader's claims (none when the tiles are too many to keep)
        const int nt = __ldcg(p.plan_hdr + PL_TILES);
        if (nt <= kExUposCap) {
            for (int t = lane; t < nt; t += 32) sm.u0[t] = __ldcg(&p.tiles[t].u0);
            if (lane == 0) sm.u0[nt] = __ldcg(p.plan_hdr + PL_UNITS);
        }
        __syncwarp();
        if (lane == 0) {
            sm.nt = nt;
            mbar_arrive(&sm.u0_ready);
        }
    } else if (warp < 8) {
        expand_produce_y(p, sm);
    } else {
        // warps 8-19, idle until the first accumulator: this block's equal run of the launch's S chunks (each
        // the sum of a tile's partials in chunk order, in two halves), each tile's once all its K-chunks are
        // counted, then the sums counted on the tile (what the S loaders wait for)
        constexpr int nthr = 128 * kExGroups;
        const int et = threadIdx.x - 256;
        const int2 r0 = __ldcg(p.rd_start + blockIdx.x), r1 = __ldcg(p.rd_start + blockIdx.x + 1);
        for (int t = r0.x; t < r1.x || (t == r1.x && r1.y > 0); ++t) {
            const TileRec tr = load_tile(p.tiles + t);
            const int lo = t == r0.x ? r0.y : 0;
            const int hi = t == r1.x ? r1.y : tr.R * tr.n_pad / 8;
            if (et == 0) {
                sm.rd_ok = wait_at_least(p, p.tile_cnt + t, tr.n_kc);
                __threadfence();
                if (t == r0.x) tstamp(p, 1, 29);
            }
            bar_sync(4, nthr);
            if (!sm.rd_ok) break;   // block-uniform
            for (int h = 2 * lo + et; h < 2 * hi; h += nthr) reduce_s_half(p, tr, h);
            bar_sync(4, nthr);
            if (et == 0) {
                __threadfence();
                atomicAdd(p.s_done + t, hi - lo);
                tstamp(p, 1, 30);
            }
        }
        expand_epilogue(p, sm, (warp - 8) >> 2);
    }
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(sm.tmem_base, kExTmemCols);
    }
    // the last block out resets the launch's counters for the next launch (the shrink grid has ended: every
    // block waits for it here)
    if (threadIdx.x == 0) {
        pdl_wait();
        __threadfence();
        sm.flag = atomicAdd(p.done, 1) == (int)gridDim.x - 1;
        __threadfence();
    }
    __syncthreads();
    if (sm.flag) {
        const int nt = min(__ldcg(p.plan_hdr + PL_TILES), p.max_tiles);
        for (int t = threadIdx.x; t < nt; t += blockDim.x) p.tile_cnt[t] = p.s_done[t] = 0;
        if (threadIdx.x == 0) {
            *p.cnt = 0;
            *p.done = 0;
        }
    }
    if (threadIdx.x == 0) tstamp(p, 1, 31);
}

// ===========================================================================
// host side
// ===========================================================================
size_t stream_plan_bytes(int32_t max_tiles)
{
    const size_t a = 256 + (size_t)max_tiles * sizeof(TileRec) + 2 * ((size_t)kStreamMaxGrid + 1) * 8;
    return (a + 255) / 256 * 256;
}

int stream_grid(int sms) { return sms < kStreamMaxGrid ? sms : kStreamMaxGrid; }

cudaError_t launch_stream(const StreamParams &p, cudaStream_t s, bool pdl)
{
    static int attr_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_dev != dev) {   // the attributes are per device; the first launch on each sets them
        e = cudaFuncSetAttribute(shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(ShrinkSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sizeof(ExpandSmem));
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    if (p.grid_s > kStreamMaxGrid || p.grid_e > kStreamMaxGrid) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;

    // the shrink waits twice for every block of its grid: a cooperative launch keeps them all resident
    cfg.attrs = pdl ? attr : attr + 1;
    cfg.numAttrs = pdl ? 2 : 1;
    cfg.gridDim = dim3(p.grid_s);
    cfg.blockDim = dim3(kShThreads);
    cfg.dynamicSmemBytes = sizeof(ShrinkSmem);
    e = cudaLaunchKernelEx(&cfg, shrink_kernel, p);
    if (e != cudaSuccess) return e;

    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3(p.grid_e);
    cfg.blockDim = dim3(kExThreads);
    cfg.dynamicSmemBytes = sizeof(ExpandSmem);
    return cudaLaunchKernelEx(&cfg, expand_kernel, p);
}

}  // namespace lora
