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
//   * CUDA-core path (at most LORA_OPT_TC_MIN_ROWS rows, decode-sized):
//     tiles of up to 16 rows; shrink item = (tile, K-chunk of about 32 KB of
//     A), fp32 partial by FMA; the expand item sums the published partials in
//     K order itself.
//   * tensor-core path (more rows, prefill-sized): tiles of up to 128 rows;
//     shrink item = (tile, 512-wide K-chunk) on tcgen05 with the accumulator
//     in tensor memory; the last shrink item of a tile sums the partials in K
//     order and writes S in bf16; the expand runs D = S B^T on tcgen05 with a
//     double-buffered accumulator and adds scale * D in the epilogue.
// An expand item is a run of output-column units of one slice of one tile;
// its units stream through a three-stage ring of {B rows, output rows}
// buffers, and items are sized so each CTA gets about two of them.
// Shrink items publish their fp32 partials to L2 and bump the tile's counter
// with release semantics; expand items put their first operands in flight
// and then wait (bounded) for the tile.  CTA b takes shrink items b, b+grid,
// ... before any expand item, and the whole grid is co-resident, so every
// wait ends.  Operand chunks are contiguous runs of the packed table or whole
// input/output rows and move by bulk async copies on mbarriers; the
// tensor-core gathers of token rows use 16-byte cp.async.  The summation
// order never depends on timing or on which rows share a tile, so the same
// inputs always give the same bits.
#include "common.cuh"
#include "tc.cuh"

namespace lora {

constexpr int kT = kEngineThreads;
constexpr int kGroupCap = 2048;                     // groups per launch held in shared memory
constexpr int kGroupCache = 512;                    // group records cached in shared memory
constexpr int kRankCache = 1024;                    // stored ranks cached in shared memory
// CUDA-core path
constexpr int kChunkBytes = 32 * 1024;              // target bytes of one A chunk / one B unit
constexpr int kMaxKc = 1024;                        // K elements of a chunk at the smallest R
constexpr int kMaxBgUnit = 512;                     // output columns of one CUDA-core expand unit, at most
// tensor-core path
constexpr int kTcRows = 128;                        // MMA M: rows of one tile
constexpr int kTcKc = 512;                          // K elements of one shrink item
constexpr int kTcStageK = 64;                       // K elements of one shrink pipeline stage
constexpr int kTcCols = 128;                        // output columns of one expand unit (MMA N)
constexpr int kTcMaxDepth = 4;                      // shrink pipeline stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemExpandCol = 256;            // shrink accumulator: [0, R); expand: [256, 384), [384, 512)
// shared-memory pool: the shrink work uses [0, 96K); the expand ring grows down from the top
constexpr int kShrinkBytes = 96 * 1024;
constexpr int kExpandBytes = 72 * 1024;
constexpr int kPool = kShrinkBytes + kExpandBytes;
constexpr int kBgA = 0, kBgX = 32 * 1024, kBgRed = 64 * 1024;   // CUDA-core shrink carve-up
constexpr int kSOff = 0;                            // an expand item's S: fp32 [16][64] or bf16 [rp/8][128][8]
constexpr int kEsBytes = 48 * 1024;                 // one expand stage: B rows at 0, output rows after them
constexpr int kEsDepth = 3;
constexpr int kEsYbg = 32 * 1024, kEsYtc = 16 * 1024;
constexpr int kItemsPerCta = 2;                     // expand items per CTA the work list aims for
// trace slots (lora_set_trace): first shrink item, first expand item, first units
enum {
    TS_ENTRY = 0, TS_WORKLIST = 1, TS_SH_START = 2, TS_SH_STAGE = 3 /* 8 slots: stage s MMAs issued */,
    TS_SH_MMA_DONE = 11, TS_SH_STORED = 12, TS_SH_PUBLISHED = 13, TS_EX_READY = 14, TS_EX_S = 15,
    TS_EX_UNIT = 16 /* 4 units x (landed, epilogue done) */, TS_EXIT = 31
};

__device__ __forceinline__ int kc_for(int R)
{
    int kc = (kChunkBytes / (2 * R)) / 64 * 64;
    return kc < 64 ? 64 : (kc > kMaxKc ? kMaxKc : kc);
}
// CUDA-core expand unit: about 32 KB of B, a multiple of the 256-row B tile, at most 512 columns
__device__ __forceinline__ int bg_unit_for(int rp)
{
    int w = (kChunkBytes / (2 * rp)) / kNTile * kNTile;
    return w < kNTile ? kNTile : (w > kMaxBgUnit ? kMaxBgUnit : w);
}
__device__ __forceinline__ int es_off(int st) { return kPool - (st + 1) * kEsBytes; }

struct __align__(1024) EngineSmem {
    __align__(1024) unsigned char pool[kPool];
    uint64_t bar_shrink;                 // CUDA-core shrink copies
    uint64_t bar_es[kEsDepth];           // expand stage copies
    uint64_t bar_s;                      // tensor-core expand: S copy
    uint64_t bar_stage[kTcMaxDepth];     // tensor-core shrink stage: A chunk landed
    uint64_t bar_mma[kTcMaxDepth];       // tensor-core shrink stage: consumed by the MMAs
    uint64_t bar_mmae[2];                // tensor-core expand MMAs done, per accumulator buffer
    uint32_t tmem_base;
    int32_t G, flag, fin, ue;
    int32_t row_src[kTcRows];
    int32_t row_dst[kTcRows];
    float row_w[kTcRows];
    int32_t sh_pre[kGroupCap + 1];       // shrink items before group g
    int32_t ex_pre[kGroupCap + 1];       // expand items before group g
    int32_t tile_pre[kGroupCap + 1];     // tiles before group g
    int32_t part_pre[kGroupCap + 1];     // scratch floats before group g
    int4 grp[kGroupCache];               // (adapter, expert, rows_off, count) of the first groups
    int32_t rp_cache[kRankCache];        // stored rank of the first adapters
};

size_t engine_smem_bytes(int) { return sizeof(EngineSmem); }

struct GroupDims {
    int a, e, rows_off, count;
    int rp, R;
    bool tc;
    int tile_rows, kc, n_kc, tiles;
    int uw;        // output columns of one expand unit
    int units;     // expand units of one tile over all slices
    int ipt;       // expand items of one tile (needs the launch-wide units per item; 0 before it is known)
    int scratch;   // floats of hand-off scratch: partials (+ bf16 S of each tile on the tensor-core path)
};

__device__ __forceinline__ GroupDims group_dims(const EngineParams &p, const EngineSmem &sm, int g, int ue)
{
    GroupDims d;
    const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
    d.a = gr.x;
    d.e = gr.y;
    d.rows_off = gr.z;
    d.count = gr.w;
    d.rp = d.a < kRankCache ? sm.rp_cache[d.a] : p.rpad[d.a];
    d.R = p.n_a * d.rp;
    d.tc = p.path == 2 || (p.path == 0 && d.count > p.tc_min_rows);
    d.tile_rows = d.tc ? kTcRows : kBgmvRows;
    d.kc = d.tc ? kTcKc : kc_for(d.R);
    d.n_kc = (p.K + d.kc - 1) / d.kc;
    d.tiles = (d.count + d.tile_rows - 1) / d.tile_rows;
    d.uw = d.tc ? kTcCols : bg_unit_for(d.rp);
    int units = 0, items = 0;
    for (int s = 0; s < p.n_slices; ++s) {
        const int us = (p.slice_n[s] + d.uw - 1) / d.uw;
        units += us;
        if (ue > 0) items += (us + ue - 1) / ue;
    }
    d.units = units;
    d.ipt = items;
    d.scratch = d.n_kc * d.count * d.R + (d.tc ? d.tiles * (kTcRows / 2) * d.R : 0);
    return d;
}

__device__ __forceinline__ int find_group(const int32_t *pre, int G, int item)
{
    int lo = 0, hi = G;   // pre[lo] <= item < pre[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
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
__device__ __forceinline__ bool wait_counter(const int32_t *ctr, int target, const EngineParams &p)
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

// Phase stamps for lora_set_trace (slot k of this block, kTraceSlots per block).
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
       PH_MMAE = 13 /* 2 bits */ };

// ===========================================================================
// CUDA-core path
// ===========================================================================
// Shrink partial for up to ROWS rows: thread (ks, j) accumulates row j of the
// A chunk against every row over K-groups ks, ks + nks, ... and leaves its
// sums in red[ks][i][j].
template <int ROWS>
__device__ __forceinline__ void bg_shrink_rows(EngineSmem &sm, int R, int kw, int xstride, int nrows)
{
    const int tid = threadIdx.x;
    const int nks = kT / R;
    const int j = tid % R, ks = tid / R;
    if (ks >= nks) return;
    const uint4 *A = reinterpret_cast<const uint4 *>(sm.pool + kBgA);
    const uint4 *X = reinterpret_cast<const uint4 *>(sm.pool + kBgX);
    float *red = reinterpret_cast<float *>(sm.pool + kBgRed);
    float acc[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i) acc[i] = 0.f;
    const int kgs = kw / 8;
    for (int kg = ks; kg < kgs; kg += nks) {
        float af[8];
        bf16x8_to_f32(A[kg * R + j], af);
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            if (i < nrows) {
                float xf[8];
                bf16x8_to_f32(X[i * xstride + kg], xf);
                float s = acc[i];
#pragma unroll
                for (int u = 0; u < 8; ++u) s = fmaf(xf[u], af[u], s);
                acc[i] = s;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
        if (i < nrows) red[(ks * kBgmvRows + i) * R + j] = acc[i];
}


// ===========================================================================
// tensor-core path
// ===========================================================================
__device__ __forceinline__ int tc_stage_bytes(int R) { return kTcRows * kTcStageK * 2 + R * kTcStageK * 2; }
__device__ __forceinline__ int tc_depth(int R)
{
    const int d = kShrinkBytes / tc_stage_bytes(R);
    return d > kTcMaxDepth ? kTcMaxDepth : d;
}

// Scratch layout of a tensor-core tile: [n_kc][nrows][R] fp32 partials for
// every tile of the group, then one bf16 S [R/8][128][8] per tile.
__device__ __forceinline__ const __nv_bfloat16 *tc_S(const EngineParams &p, const EngineSmem &sm, const GroupDims &d,
                                                     int g, int tile)
{
    return reinterpret_cast<const __nv_bfloat16 *>(p.partials + sm.part_pre[g] + (int64_t)d.n_kc * d.count * d.R +
                                                   (int64_t)tile * (kTcRows / 2) * d.R);
}

// Put one shrink pipeline stage in flight: 128 token rows x 64 K in the
// 128-byte swizzled K-major layout, and the matching A chunk (one bulk copy).
// When the tile's rows are one run of consecutive rows of x with the whole
// 128-row box inside x, a single TMA tile load brings them; otherwise every
// thread gathers 16-byte pieces with cp.async into the same swizzled places
// (zero for rows past the tile or columns past K).
__device__ __forceinline__ void tc_issue_stage(const EngineParams &p, EngineSmem &sm, const GroupDims &d, int nrows,
                                               int k0, int kw, int s, int depth, bool run)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = s % depth;
    unsigned char *Xs = sm.pool + slot * tc_stage_bytes(d.R);
    unsigned char *As = Xs + kTcRows * kTcStageK * 2;
    const int kb = k0 + s * kTcStageK;
    const int vkg = min(8, (kw - s * kTcStageK) / 8);       // K-groups of 8 present in this stage
    const int need = ((vkg + 1) / 2) * 2;                   // K-groups the MMAs read (whole K=16 steps)
    if (vkg < need) {   // odd K-group count at the end of K: the last A K-group reads as zero
        uint4 *z = reinterpret_cast<uint4 *>(As + vkg * d.R * 16);
        for (int i = tid; i < d.R; i += kT) z[i] = make_uint4(0u, 0u, 0u, 0u);
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
        const __nv_bfloat16 *ablk =
            reinterpret_cast<const __nv_bfloat16 *>(p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)]);
        const uint32_t bytes = (uint32_t)vkg * d.R * 16;
        mbar_arrive_expect_tx(&sm.bar_stage[slot], bytes + (run ? kTcRows * kTcStageK * 2 : 0));
        bulk_g2s(As, ablk + (int64_t)(kb / 8) * d.R * 8, bytes, &sm.bar_stage[slot]);
        if (run) tc::tma_tile2d(Xs, &p.x_map, kb, sm.row_src[0], &sm.bar_stage[slot]);
    }
}

template <int N>
__device__ __forceinline__ void cp_wait_n() { tc::cp_async_wait<N>(); }
__device__ __forceinline__ void cp_wait_pending(int pending)
{
    if (pending <= 0) cp_wait_n<0>();
    else if (pending == 1) cp_wait_n<1>();
    else if (pending == 2) cp_wait_n<2>();
    else cp_wait_n<3>();
}


// Tensor-core shrink item: partial = X_rows[:, K-chunk] A[:, K-chunk]^T into
// tensor memory, then out to the tile's scratch slot.  A pipeline stage is
// refilled one iteration after its MMAs were issued, so the refill rarely
// waits.  Returns false if a wait ran out.
__device__ bool tc_shrink_item(const EngineParams &p, EngineSmem &sm, const GroupDims &d, int g, int tile, int chunk,
                               Phases &ph, bool first)
{
    if (first) stamp(p, TS_SH_START);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = tile * kTcRows;
    const int nrows = min(kTcRows, d.count - r0);
    const int k0 = chunk * kTcKc;
    const int kw = min(kTcKc, p.K - k0);
    const int nst = (kw + kTcStageK - 1) / kTcStageK;
    const int depth = min(tc_depth(d.R), nst);
    int my_row = 0;
    if (tid < kTcRows) {
        my_row = tid < nrows ? p.rows[d.rows_off + r0 + tid] / p.src_div : 0;
        sm.row_src[tid] = my_row;
    }
    __syncthreads();
    // one TMA tile per stage when the rows are one run of consecutive rows and the 128-row box stays inside x
    const int x_total = *p.m_ptr * p.m_mult;
    const bool consecutive = tid >= nrows || my_row == sm.row_src[0] + tid;
    const bool run = __syncthreads_and(consecutive ? 1 : 0) != 0 && p.x_rows > 0 && sm.row_src[0] + kTcRows <= x_total;
    for (int s = 0; s < depth; ++s) tc_issue_stage(p, sm, d, nrows, k0, kw, s, depth, run);

    const uint32_t idesc = tc::idesc_bf16(kTcRows, d.R);
    uint32_t pending = 0;   // slots whose MMA commit has not been waited for
    bool ok = true;
    for (int s = 0; s < nst && ok; ++s) {
        const int slot = s % depth;
        if (s >= 1 && s - 1 + depth < nst) {   // refill the previous stage's slot
            const int ps = (s - 1) % depth;
            ok = cta_wait(&sm.bar_mma[ps], ph.get(PH_MMA + ps), p);
            ph.flip(PH_MMA + ps);
            pending &= ~(1u << ps);
            if (!ok) break;
            tc_issue_stage(p, sm, d, nrows, k0, kw, s - 1 + depth, depth, run);
        }
        if (!run) {
            cp_wait_pending(min(nst, s + depth) - (s + 1));
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
                const int vkg = min(8, (kw - s * kTcStageK) / 8);
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
    cp_wait_n<0>();
    if (!ok) return false;
    tc::fence_after_sync();
    if (first) stamp(p, TS_SH_MMA_DONE);

    // tensor memory -> this tile's partial slot: warp w (w < 4) owns rows 32w .. 32w + 31
    if (warp < 4) {
        const int row = warp * 32 + lane;
        float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * d.R + (int64_t)chunk * nrows * d.R +
                     (int64_t)row * d.R;
        for (int c0 = 0; c0 < d.R; c0 += 16) {
            float v[16];
            tc::tmem_ld16(sm.tmem_base + ((uint32_t)(warp * 32) << 16) + c0, v);
            if (row < nrows) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4 *>(dst + c0 + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (first) stamp(p, TS_SH_STORED);
    return true;
}

// Last shrink item of a tensor-core tile: S = sum over K-chunks (ascending) of
// the partials, rounded once to bf16, stored [R/8][128][8] (rows past the tile
// are zero).
__device__ void tc_finish_tile(const EngineParams &p, const EngineSmem &sm, const GroupDims &d, int g, int tile)
{
    const int r0 = tile * kTcRows;
    const int nrows = min(kTcRows, d.count - r0);
    const float *part = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * d.R;
    const int64_t stride = (int64_t)nrows * d.R;
    uint4 *S = reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(tc_S(p, sm, d, g, tile)));
    const int kgs = d.R / 8;
    for (int u = threadIdx.x; u < kTcRows * kgs; u += kT) {
        const int i = u % kTcRows, kg = u / kTcRows;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        if (i < nrows) {
            const float *src = part + (int64_t)i * d.R + kg * 8;
            for (int c0 = 0; c0 < d.n_kc; c0 += 4) {
                float4 v[4][2];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c0 + c < d.n_kc) {
                        v[c][0] = __ldcg(reinterpret_cast<const float4 *>(src + (c0 + c) * stride));
                        v[c][1] = __ldcg(reinterpret_cast<const float4 *>(src + (c0 + c) * stride + 4));
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c0 + c < d.n_kc) {
                        acc[0] += v[c][0].x; acc[1] += v[c][0].y; acc[2] += v[c][0].z; acc[3] += v[c][0].w;
                        acc[4] += v[c][1].x; acc[5] += v[c][1].y; acc[6] += v[c][1].z; acc[7] += v[c][1].w;
                    }
                }
            }
        }
        __align__(16) __nv_bfloat16 o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __float2bfloat16_rn(acc[e]);
        S[kg * kTcRows + i] = *reinterpret_cast<const uint4 *>(o);
    }
}


// ===========================================================================
// expand items (both paths)
// ===========================================================================
struct ExpandItem {
    int g, tile, s, u0, nu, r0, nrows, sa, tg;
    GroupDims d;
};

__device__ __forceinline__ ExpandItem decode_expand(const EngineParams &p, const EngineSmem &sm, int G, int item)
{
    ExpandItem it;
    const int ue = sm.ue;
    it.g = find_group(sm.ex_pre, G, item);
    it.d = group_dims(p, sm, it.g, ue);
    const int local = item - sm.ex_pre[it.g];
    it.tile = local / it.d.ipt;
    int q = local % it.d.ipt;
    int s = 0;
    for (; s < p.n_slices; ++s) {
        const int is = ((p.slice_n[s] + it.d.uw - 1) / it.d.uw + ue - 1) / ue;
        if (q < is) break;
        q -= is;
    }
    const int us = (p.slice_n[s] + it.d.uw - 1) / it.d.uw;
    it.s = s;
    it.u0 = q * ue;
    it.nu = min(ue, us - it.u0);
    it.r0 = it.tile * it.d.tile_rows;
    it.nrows = min(it.d.tile_rows, it.d.count - it.r0);
    it.sa = (p.n_a == 1) ? 0 : s;
    it.tg = sm.tile_pre[it.g] + it.tile;
    return it;
}

// Put unit k of an expand item in flight into stage k % 3: its B rows and its
// output rows.  Unit 0 also records the item's output rows and row weights.
__device__ __forceinline__ void issue_unit(const EngineParams &p, EngineSmem &sm, const ExpandItem &it, int k)
{
    const int tid = threadIdx.x;
    const GroupDims &d = it.d;
    const int st = k % kEsDepth;
    unsigned char *base = sm.pool + es_off(st);
    const int uu = it.u0 + k;
    const int n0 = p.slice_off[it.s] + uu * d.uw;
    const int nw = min(d.uw, p.slice_n[it.s] - uu * d.uw);
    const int yoff = d.tc ? kEsYtc : kEsYbg;
    if (tid < it.nrows) {
        int row;
        if (k == 0) {
            row = p.rows[d.rows_off + it.r0 + tid];
            sm.row_dst[tid] = row;
            sm.row_w[tid] = p.row_weight ? p.row_weight[row] : 1.0f;
        } else {
            row = sm.row_dst[tid];   // written by this thread when unit 0 was issued
        }
        bulk_g2s(base + yoff + tid * d.uw * 2, p.y + (int64_t)row * p.ldy + n0, (uint32_t)nw * 2, &sm.bar_es[st]);
    }
    if (tid == 0) {
        const __nv_bfloat16 *bblk =
            reinterpret_cast<const __nv_bfloat16 *>(p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)]);
        const uint32_t y_bytes = (uint32_t)it.nrows * nw * 2;
        if (d.tc) {
            // 128 output columns = one half of a 256-row B tile: rp/8 runs of 128 x 16 bytes
            const uint32_t kgs = d.rp / 8;
            const int btile = p.slice_tile_off[it.s] + uu / 2, half = uu & 1;
            mbar_arrive_expect_tx(&sm.bar_es[st], kgs * kTcCols * 16 + y_bytes);
            for (uint32_t kg = 0; kg < kgs; ++kg)
                bulk_g2s(base + kg * kTcCols * 16, bblk + ((int64_t)(btile * kgs + kg) * kNTile + half * kTcCols) * 8,
                         kTcCols * 16, &sm.bar_es[st]);
        } else {
            const int tile0 = p.slice_tile_off[it.s] + uu * (d.uw / kNTile);
            const int ntl = (nw + kNTile - 1) / kNTile;
            const uint32_t b_bytes = (uint32_t)ntl * kNTile * d.rp * 2;
            mbar_arrive_expect_tx(&sm.bar_es[st], b_bytes + y_bytes);
            bulk_g2s(base, bblk + (int64_t)tile0 * kNTile * d.rp, b_bytes, &sm.bar_es[st]);
        }
    }
}

// CUDA-core unit: thread per output column; y = bf16(y_base + scale * w_row * sum_j S[i][j] B[n][j]).
template <int ROWS>
__device__ __forceinline__ void bg_unit(const EngineParams &p, const EngineSmem &sm, const ExpandItem &it, int k)
{
    const GroupDims &d = it.d;
    const int st = k % kEsDepth;
    const unsigned char *base = sm.pool + es_off(st);
    const uint4 *B = reinterpret_cast<const uint4 *>(base);
    const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(base + kEsYbg);
    const float *S = reinterpret_cast<const float *>(sm.pool + kSOff);
    const int uu = it.u0 + k;
    const int n0 = p.slice_off[it.s] + uu * d.uw;
    const int nw = min(d.uw, p.slice_n[it.s] - uu * d.uw);
    const float sc = p.scale[d.a];
    const int kgs = d.rp / 8;
    const int nrows = it.nrows;
    for (int nl = threadIdx.x; nl < nw; nl += kT) {
        float acc[ROWS];
#pragma unroll
        for (int i = 0; i < ROWS; ++i) acc[i] = 0.f;
        const int tl = nl / kNTile, row = nl % kNTile;
        for (int kg = 0; kg < kgs; ++kg) {
            float bfv[8];
            bf16x8_to_f32(B[(tl * kgs + kg) * kNTile + row], bfv);
#pragma unroll
            for (int i = 0; i < ROWS; ++i) {
                if (i < nrows) {
                    float a = acc[i];
#pragma unroll
                    for (int u = 0; u < 8; ++u) a = fmaf(S[i * kMaxRank + kg * 8 + u], bfv[u], a);
                    acc[i] = a;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            if (i < nrows) {
                const float yb = __bfloat162float(ys[i * d.uw + nl]);
                p.y[(int64_t)sm.row_dst[i] * p.ldy + n0 + nl] = __float2bfloat16_rn(fmaf(sc * sm.row_w[i], acc[i], yb));
            }
        }
    }
}

// Tensor-core unit k: D(k & 1) = S B_k^T (one thread issues, commit on bar_mmae).
__device__ __forceinline__ void tc_unit_mma(EngineSmem &sm, const ExpandItem &it, int k)
{
    const GroupDims &d = it.d;
    const unsigned char *base = sm.pool + es_off(k % kEsDepth);
    const uint32_t steps = d.rp / 16;
    const uint32_t acc = sm.tmem_base + kTmemExpandCol + (k & 1) * kTcCols;
    tc::fence_after_sync();
    for (uint32_t j = 0; j < steps; ++j) {
        const uint64_t ad = tc::smem_desc(smem_u32(sm.pool + kSOff) + j * 2 * kTcRows * 16, kTcRows * 16, 128);
        const uint64_t bd = tc::smem_desc(smem_u32(base) + j * 2 * kTcCols * 16, kTcCols * 16, 128);
        tc::mma_bf16(acc, ad, bd, tc::idesc_bf16(kTcRows, kTcCols), j > 0 ? 1u : 0u);
    }
    tc::mma_commit(&sm.bar_mmae[k & 1]);
}

// Tensor-core epilogue of unit k: warp w owns rows 32 (w % 4) + lane and 64
// columns starting at 64 (w / 4); y = bf16(y_base + scale * w_row * D).
__device__ __forceinline__ void tc_unit_epilogue(const EngineParams &p, const EngineSmem &sm, const ExpandItem &it,
                                                 int k)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const GroupDims &d = it.d;
    const int uu = it.u0 + k;
    const int n0 = p.slice_off[it.s] + uu * d.uw;
    const int nw = min(d.uw, p.slice_n[it.s] - uu * d.uw);
    const int row = (warp & 3) * 32 + lane;
    const int cbase = (warp >> 2) * 64;
    const bool live = row < it.nrows;
    const float sc = p.scale[d.a] * (live ? sm.row_w[row] : 0.f);
    const __nv_bfloat16 *ys =
        reinterpret_cast<const __nv_bfloat16 *>(sm.pool + es_off(k % kEsDepth) + kEsYtc) + row * kTcCols;
    __nv_bfloat16 *yg = p.y + (int64_t)(live ? sm.row_dst[row] : 0) * p.ldy + n0;
    const uint32_t acc = sm.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kTmemExpandCol + (k & 1) * kTcCols;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c0 = cbase + h * 32;
        float v[32];
        tc::tmem_ld32(acc + c0, v);
        if (live) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + 8 * q;
                if (c < nw) {
                    float yf[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(ys + c), yf);
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = __float2bfloat16_rn(fmaf(sc, v[8 * q + e], yf[e]));
                    *reinterpret_cast<uint4 *>(yg + c) = *reinterpret_cast<const uint4 *>(o);
                }
            }
        }
    }
}

// One expand item.  Unit 0 may already be in flight (prefetched during the
// shrink work).  Returns false if a wait ran out; *inflight tracks the stages
// whose copies have not been waited for.
__device__ bool expand_item(const EngineParams &p, EngineSmem &sm, const ExpandItem &it, bool unit0_issued,
                            Phases &ph, uint32_t &inflight, bool first)
{
    const int tid = threadIdx.x;
    const GroupDims &d = it.d;
    const int nu = it.nu;
    for (int k = unit0_issued ? 1 : 0; k < min(nu, kEsDepth); ++k) {
        issue_unit(p, sm, it, k);
        inflight |= 1u << (k % kEsDepth);
    }

    // wait until the tile's shrink results are published
    if (tid == 0) {
        const bool ok = d.tc ? wait_counter(&p.sync[it.tg * 4 + 2], 1, p) : wait_counter(&p.sync[it.tg * 4 + 0], d.n_kc, p);
        if (ok && d.tc) {
            // S was written by another CTA through ordinary stores: order them before the async copy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t s_bytes = (uint32_t)(d.rp / 8) * kTcRows * 16;
            const __nv_bfloat16 *S = tc_S(p, sm, d, it.g, it.tile) + (int64_t)it.sa * (d.rp / 8) * kTcRows * 8;
            mbar_arrive_expect_tx(&sm.bar_s, s_bytes);
            bulk_g2s(sm.pool + kSOff, S, s_bytes, &sm.bar_s);
        }
        sm.flag = ok ? 1 : 0;
    }
    if (first) stamp(p, TS_EX_READY);
    __syncthreads();
    bool ready = sm.flag != 0;
    if (ready && !d.tc) {
        // S[i][j] = sum over K-chunks q (ascending) of the published partials; loads first, then the sum
        float *S = reinterpret_cast<float *>(sm.pool + kSOff);
        const int64_t stride = (int64_t)it.nrows * d.R;
        const float *part = p.partials + sm.part_pre[it.g] + (int64_t)d.n_kc * it.r0 * d.R + it.sa * d.rp;
        for (int idx = tid; idx < it.nrows * d.rp; idx += kT) {
            const int i = idx / d.rp, jj = idx % d.rp;
            const float *src = part + (int64_t)i * d.R + jj;
            float acc = 0.f;
            for (int q0 = 0; q0 < d.n_kc; q0 += 16) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = (q0 + u < d.n_kc) ? __ldcg(src + (q0 + u) * stride) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (q0 + u < d.n_kc) acc += v[u];
            }
            S[i * kMaxRank + jj] = acc;
        }
    }
    if (ready && d.tc) {
        ready = cta_wait(&sm.bar_s, ph.get(PH_S), p);
        ph.flip(PH_S);
    }
    __syncthreads();
    if (first) stamp(p, TS_EX_S);
    if (tid == 0 && sm.flag != 0) {
        const int old = atomicAdd(&p.sync[it.tg * 4 + 1], 1);
        if (old == d.ipt - 1) {   // last consumer of this tile resets its counters
            p.sync[it.tg * 4 + 0] = 0;
            p.sync[it.tg * 4 + 1] = 0;
            p.sync[it.tg * 4 + 2] = 0;
        }
    }
    if (!ready) return false;

    for (int k = 0; k < nu; ++k) {
        const int st = k % kEsDepth;
        if (!cta_wait(&sm.bar_es[st], ph.get(PH_ES + st), p)) return false;
        ph.flip(PH_ES + st);
        inflight &= ~(1u << st);
        if (first && k < 4) stamp(p, TS_EX_UNIT + 2 * k);
        if (d.tc) {
            if (tid == 0) tc_unit_mma(sm, it, k);
            if (k > 0) {   // epilogue of the previous unit overlaps this unit's MMAs
                const int pb = (k - 1) & 1;
                if (!cta_wait(&sm.bar_mmae[pb], ph.get(PH_MMAE + pb), p)) return false;
                ph.flip(PH_MMAE + pb);
                tc::fence_after_sync();
                tc_unit_epilogue(p, sm, it, k - 1);
                tc::fence_before_sync();
                __syncthreads();   // stage (k - 1) % 3 is free again
                if (first && k - 1 < 4) stamp(p, TS_EX_UNIT + 2 * (k - 1) + 1);
                if (k - 1 + kEsDepth < nu) {
                    issue_unit(p, sm, it, k - 1 + kEsDepth);
                    inflight |= 1u << ((k - 1) % kEsDepth);
                }
            }
        } else {
            if (it.nrows <= 2) bg_unit<2>(p, sm, it, k);
            else if (it.nrows <= 4) bg_unit<4>(p, sm, it, k);
            else if (it.nrows <= 8) bg_unit<8>(p, sm, it, k);
            else bg_unit<16>(p, sm, it, k);
            __syncthreads();       // stage k % 3 is free again
            if (first && k < 4) stamp(p, TS_EX_UNIT + 2 * k + 1);
            if (k + kEsDepth < nu) {
                issue_unit(p, sm, it, k + kEsDepth);
                inflight |= 1u << st;
            }
        }
    }
    if (d.tc) {
        const int pb = (nu - 1) & 1;
        if (!cta_wait(&sm.bar_mmae[pb], ph.get(PH_MMAE + pb), p)) return false;
        ph.flip(PH_MMAE + pb);
        tc::fence_after_sync();
        tc_unit_epilogue(p, sm, it, nu - 1);
        tc::fence_before_sync();
        __syncthreads();
    }
    return true;
}

// ===========================================================================
// the kernel
// ===========================================================================
__global__ void __launch_bounds__(kEngineThreads, 1) engine_kernel(const __grid_constant__ EngineParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    EngineSmem &sm = *reinterpret_cast<EngineSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (p.trace != nullptr && tid > 0 && tid < kTraceSlots && (int)blockIdx.x < p.trace_ctas)
        p.trace[(size_t)blockIdx.x * kTraceSlots + tid] = 0;
    stamp(p, TS_ENTRY);

    // ---- prologue: one round trip for the count, the first group records and the stored ranks ----
    if (tid == 0) {
        sm.G = *p.num_groups;
        sm.flag = 0;
        mbar_init(&sm.bar_shrink, 1);
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
    const int gpre = min(p.group_capacity, kGroupCache);
    for (int g = tid; g < gpre; g += kT) sm.grp[g] = p.groups[g];
    for (int a = tid; a < min(p.L, kRankCache); a += kT) sm.rp_cache[a] = p.rpad[a];
    __syncthreads();
    const int G = sm.G;
    if (G <= 0) return;
    if (G > p.group_capacity || G > kGroupCap) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    if (warp == 0) {
        // pass 1: validate the groups, count expand units -> units per expand item
        bool bad = false, any_tc = false;
        int units = 0;
        for (int g = lane; g < G; g += 32) {
            const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
            if (gr.x < 0 || gr.x >= p.L || gr.y < 0 || gr.y >= p.num_experts || gr.z < 0 || gr.w < 1 ||
                (int64_t)gr.z + gr.w > p.rows_capacity) {
                bad = true;   // a workspace that lora_build_segments never filled
            } else {
                const GroupDims d = group_dims(p, sm, g, 0);
                units += d.tiles * d.units;
                any_tc |= d.tc;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) units += __shfl_xor_sync(0xffffffffu, units, o);
        bad = __any_sync(0xffffffffu, bad);
        any_tc = __any_sync(0xffffffffu, any_tc);
        const int target = kItemsPerCta * (int)gridDim.x;
        const int ue = max(1, (units + target - 1) / target);
        // pass 2: per-group item counts and their exclusive prefix sums, 32 groups per step
        int4 carry = make_int4(0, 0, 0, 0);
        for (int base = 0; base < G && !bad; base += 32) {
            const int g = base + lane;
            int4 v = make_int4(0, 0, 0, 0);
            if (g < G) {
                const GroupDims d = group_dims(p, sm, g, ue);
                v = make_int4(d.tiles * d.n_kc, d.tiles * d.ipt, d.tiles, d.scratch);
            }
            int4 incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int4 u = make_int4(__shfl_up_sync(0xffffffffu, incl.x, o), __shfl_up_sync(0xffffffffu, incl.y, o),
                                         __shfl_up_sync(0xffffffffu, incl.z, o), __shfl_up_sync(0xffffffffu, incl.w, o));
                if (lane >= o) incl = make_int4(incl.x + u.x, incl.y + u.y, incl.z + u.z, incl.w + u.w);
            }
            if (g < G) {
                sm.sh_pre[g] = carry.x + incl.x - v.x;
                sm.ex_pre[g] = carry.y + incl.y - v.y;
                sm.tile_pre[g] = carry.z + incl.z - v.z;
                sm.part_pre[g] = carry.w + incl.w - v.w;
            }
            carry.x += __shfl_sync(0xffffffffu, incl.x, 31);
            carry.y += __shfl_sync(0xffffffffu, incl.y, 31);
            carry.z += __shfl_sync(0xffffffffu, incl.z, 31);
            carry.w += __shfl_sync(0xffffffffu, incl.w, 31);
        }
        if (lane == 0) {
            sm.sh_pre[G] = carry.x;
            sm.ex_pre[G] = carry.y;
            sm.tile_pre[G] = carry.z;
            sm.part_pre[G] = carry.w;
            sm.ue = ue;
            sm.flag = bad ? 1 : (any_tc ? 2 : 0);
        }
    }
    __syncthreads();
    if (sm.flag == 1) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    const bool use_tc = sm.flag == 2;
    const int n_shrink = sm.sh_pre[G], n_expand = sm.ex_pre[G], n_tiles = sm.tile_pre[G], n_part = sm.part_pre[G];
    if (n_tiles > p.max_tiles || (int64_t)n_part > p.partial_floats) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    if (use_tc && (smem_u32(sm.pool) & 1023u) != 0) {   // swizzled TMA tiles need a 1024-byte aligned pool
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    if (use_tc) {   // one warp allocates the tensor memory this CTA's MMAs accumulate into
        if (warp == 0) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    Phases ph = {0u};
    uint32_t inflight = 0;   // expand stages with copies not yet waited for
    const int grid = gridDim.x;
    bool alive = true;
    stamp(p, TS_WORKLIST);

    // Unit 0 of the first expand item does not depend on any shrink result: it
    // is put in flight (stage 0 lies in the part of the pool the shrink work
    // leaves alone) right after the first shrink item's copies.
    const bool prefetch = (int)blockIdx.x < n_expand;
    bool unit0_issued = false;
    if (prefetch && (int)blockIdx.x >= n_shrink) {
        issue_unit(p, sm, decode_expand(p, sm, G, blockIdx.x), 0);
        unit0_issued = true;
        inflight |= 1u;
    }

    // ------------------------------------------------------------------
    // shrink items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_shrink && alive; item += grid) {
        const int g = find_group(sm.sh_pre, G, item);
        const GroupDims d = group_dims(p, sm, g, sm.ue);
        const int local = item - sm.sh_pre[g];
        const int tile = local / d.n_kc, chunk = local % d.n_kc;
        const int tg = sm.tile_pre[g] + tile;
        if (d.tc) {
            if (prefetch && item == (int)blockIdx.x) {
                issue_unit(p, sm, decode_expand(p, sm, G, blockIdx.x), 0);
                unit0_issued = true;
                inflight |= 1u;
            }
            if (!tc_shrink_item(p, sm, d, g, tile, chunk, ph, item == (int)blockIdx.x)) {
                alive = false;
                break;
            }
            // publish; the last K-chunk of the tile turns the partials into S
            if (tid == 0) {
                int last = 0;
                if (!p.withhold) {
                    asm volatile("fence.acq_rel.gpu;" ::: "memory");
                    last = atom_add_acq_rel_gpu(&p.sync[tg * 4 + 0], 1) == d.n_kc - 1;
                }
                sm.fin = last;
            }
            __syncthreads();
            if (sm.fin) {
                tc_finish_tile(p, sm, d, g, tile);
                __syncthreads();
                if (tid == 0) release_add(&p.sync[tg * 4 + 2], 1);
            }
            if (item == (int)blockIdx.x) stamp(p, TS_SH_PUBLISHED);
            continue;
        }
        const int r0 = tile * kBgmvRows;
        const int nrows = min(kBgmvRows, d.count - r0);
        const int k0 = chunk * d.kc;
        const int kw = min(d.kc, p.K - k0);
        const uint32_t a_bytes = (uint32_t)(kw / 8) * d.R * 16;
        const uint32_t x_bytes = (uint32_t)kw * 2;
        if (tid == 0) {
            const __nv_bfloat16 *ablk =
                reinterpret_cast<const __nv_bfloat16 *>(p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)]);
            mbar_arrive_expect_tx(&sm.bar_shrink, a_bytes + nrows * x_bytes);
            bulk_g2s(sm.pool + kBgA, ablk + (int64_t)(k0 / 8) * d.R * 8, a_bytes, &sm.bar_shrink);
        }
        if (warp == 1 && lane < nrows) {
            const int src = p.rows[d.rows_off + r0 + lane] / p.src_div;
            bulk_g2s(sm.pool + kBgX + (size_t)lane * d.kc * 2, p.x + (int64_t)src * p.ldx + k0, x_bytes,
                     &sm.bar_shrink);
        }
        if (prefetch && item == (int)blockIdx.x) {
            issue_unit(p, sm, decode_expand(p, sm, G, blockIdx.x), 0);
            unit0_issued = true;
            inflight |= 1u;
        }
        const bool ok = cta_wait(&sm.bar_shrink, ph.get(PH_SHRINK), p);
        ph.flip(PH_SHRINK);
        if (!ok) {
            alive = false;
            break;
        }
        if (item == (int)blockIdx.x) stamp(p, TS_SH_STAGE);

        // partial dot products: thread (ks, j) covers row j of A, K-groups ks, ks+nks, ...
        const int R = d.R;
        const int nks = kT / R;
        if (nrows <= 2) bg_shrink_rows<2>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 4) bg_shrink_rows<4>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 8) bg_shrink_rows<8>(sm, R, kw, d.kc / 8, nrows);
        else bg_shrink_rows<16>(sm, R, kw, d.kc / 8, nrows);
        __syncthreads();
        const float *red = reinterpret_cast<const float *>(sm.pool + kBgRed);
        float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * R + (int64_t)chunk * nrows * R;
        for (int idx = tid; idx < nrows * R; idx += kT) {
            const int i = idx / R, jj = idx % R;
            float s = 0.f;
            for (int q = 0; q < nks; ++q) s += red[(q * kBgmvRows + i) * R + jj];
            dst[idx] = s;
        }
        __syncthreads();
        if (tid == 0 && !p.withhold) release_add(&p.sync[tg * 4 + 0], 1);
        if (item == (int)blockIdx.x) stamp(p, TS_SH_PUBLISHED);
    }

    // ------------------------------------------------------------------
    // expand items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_expand && alive; item += grid) {
        const ExpandItem it = decode_expand(p, sm, G, item);
        const bool pre = unit0_issued && item == (int)blockIdx.x;
        if (!expand_item(p, sm, it, pre, ph, inflight, item == (int)blockIdx.x)) alive = false;
        __syncthreads();
    }
    // a CTA that gave up still lets its own copies land before it leaves
    for (int st = 0; st < kEsDepth; ++st)
        if (inflight & (1u << st)) mbar_wait_bounded(&sm.bar_es[st], ph.get(PH_ES + st), p.timeout_ns, p.err);
    stamp(p, TS_EXIT);
    if (use_tc) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(sm.tmem_base, kTmemCols);
    }
}

const void *engine_kernel_ptr() { return reinterpret_cast<const void *>(engine_kernel); }

void launch_engine(const EngineParams &p, int grid, size_t smem, cudaStream_t s, cudaError_t *err)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kEngineThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *err = cudaLaunchKernelEx(&cfg, engine_kernel, p);
}

}  // namespace lora
