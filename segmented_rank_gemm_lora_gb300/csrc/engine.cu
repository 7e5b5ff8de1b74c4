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
//     A), fp32 partial by FMA; expand item = (tile, chunk of about 32 KB of B
//     rows), which sums the published partials in K order itself.
//   * tensor-core path (more rows, prefill-sized): tiles of up to 128 rows;
//     shrink item = (tile, 512-wide K-chunk) on tcgen05 with the accumulator
//     in tensor memory; the last shrink item of a tile sums the partials in K
//     order and writes S in bf16; expand item = (tile, 128 output columns):
//     D = S B^T on tcgen05, then y += scale * D in the epilogue.
// Shrink items publish their fp32 partials to L2 and bump the tile's counter
// with release semantics; expand items put their operands in flight first
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
constexpr int kChunkBytes = 32 * 1024;              // target bytes of one A or B chunk
constexpr int kMaxKc = 1024;                        // K elements of a chunk at the smallest R
constexpr int kMaxNc = 1024;                        // N rows of a chunk at the smallest stored rank
// tensor-core path
constexpr int kTcRows = 128;                        // MMA M: rows of one tile
constexpr int kTcKc = 512;                          // K elements of one shrink item
constexpr int kTcStageK = 64;                       // K elements of one pipeline stage
constexpr int kTcCols = 128;                        // output columns of one expand item (MMA N)
constexpr int kTcMaxDepth = 4;                      // shrink pipeline stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemExpandCol = 256;            // shrink accumulator: columns [0, R); expand: [256, 384)
// shared memory regions (each item kind lays out its own buffers inside them)
constexpr int kShrinkBytes = 96 * 1024;
constexpr int kExpandBytes = 72 * 1024;
// CUDA-core carve-up
constexpr int kBgA = 0, kBgX = 32 * 1024, kBgRed = 64 * 1024;             // shrink region
constexpr int kBgB = 0, kBgY = 32 * 1024, kBgS = 64 * 1024;               // expand region
// tensor-core carve-up of the expand region
constexpr int kTcB = 0, kTcS = 16 * 1024, kTcY = 32 * 1024;

__device__ __forceinline__ int kc_for(int R)
{
    int kc = (kChunkBytes / (2 * R)) / 64 * 64;
    return kc < 64 ? 64 : (kc > kMaxKc ? kMaxKc : kc);
}
__device__ __forceinline__ int nc_for(int rp)
{
    int nc = (kChunkBytes / (2 * rp)) / kNTile * kNTile;
    return nc < kNTile ? kNTile : (nc > kMaxNc ? kMaxNc : nc);
}

struct __align__(1024) EngineSmem {
    __align__(1024) unsigned char shrink[kShrinkBytes];
    __align__(1024) unsigned char expand[kExpandBytes];
    uint64_t bar_shrink;                 // CUDA-core shrink copies
    uint64_t bar_expand;                 // expand copies (both paths)
    uint64_t bar_stage[kTcMaxDepth];     // tensor-core shrink stage: A chunk landed
    uint64_t bar_mma[kTcMaxDepth];       // tensor-core shrink stage: consumed by the MMAs
    uint64_t bar_mma_exp;                // tensor-core expand MMAs done
    uint32_t tmem_base;
    int32_t G, flag, fin;
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
    int tile_rows, kc, n_kc, nc, n_nc, tiles;
    int scratch;   // floats of hand-off scratch: partials (+ bf16 S of each tile on the tensor-core path)
};

__device__ __forceinline__ GroupDims group_dims(const EngineParams &p, const EngineSmem &sm, int g)
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
    d.nc = d.tc ? kTcCols : nc_for(d.rp);
    int n = 0;
    for (int s = 0; s < p.n_slices; ++s) n += (p.slice_n[s] + d.nc - 1) / d.nc;
    d.n_nc = n;
    d.tiles = (d.count + d.tile_rows - 1) / d.tile_rows;
    d.scratch = d.n_kc * d.count * d.R + (d.tc ? d.tiles * (kTcRows / 2) * d.R : 0);
    return d;
}

__device__ __forceinline__ int4 add4(int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

__device__ __forceinline__ int4 shfl_up4(int4 v, int o)
{
    return make_int4(__shfl_up_sync(0xffffffffu, v.x, o), __shfl_up_sync(0xffffffffu, v.y, o),
                     __shfl_up_sync(0xffffffffu, v.z, o), __shfl_up_sync(0xffffffffu, v.w, o));
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

// Phase stamps for lora_set_trace (slot k of this block).
__device__ __forceinline__ void stamp(const EngineParams &p, int k)
{
    if (p.trace != nullptr && threadIdx.x == 0 && (int)blockIdx.x < p.trace_ctas)
        p.trace[(size_t)blockIdx.x * 8 + k] = globaltimer();
}

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
    const uint4 *A = reinterpret_cast<const uint4 *>(sm.shrink + kBgA);
    const uint4 *X = reinterpret_cast<const uint4 *>(sm.shrink + kBgX);
    float *red = reinterpret_cast<float *>(sm.shrink + kBgRed);
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

// One expand item, decoded (both paths).
struct ExpandItem {
    int g, tile, c, s, n0, nw, r0, nrows, sa, tg;
    GroupDims d;
};

__device__ __forceinline__ ExpandItem decode_expand(const EngineParams &p, const EngineSmem &sm, int G, int item)
{
    ExpandItem it;
    it.g = find_group(sm.ex_pre, G, item);
    it.d = group_dims(p, sm, it.g);
    const int local = item - sm.ex_pre[it.g];
    it.tile = local / it.d.n_nc;
    int c = local % it.d.n_nc;
    int s = 0;
    for (; s < p.n_slices; ++s) {
        const int cs = (p.slice_n[s] + it.d.nc - 1) / it.d.nc;
        if (c < cs) break;
        c -= cs;
    }
    it.s = s;
    it.c = c;
    it.n0 = p.slice_off[s] + c * it.d.nc;
    it.nw = min(it.d.nc, p.slice_off[s] + p.slice_n[s] - it.n0);
    it.r0 = it.tile * it.d.tile_rows;
    it.nrows = min(it.d.tile_rows, it.d.count - it.r0);
    it.sa = (p.n_a == 1) ? 0 : s;
    it.tg = sm.tile_pre[it.g] + it.tile;
    return it;
}

// Expand for up to ROWS rows: thread per output column of the chunk;
// y = bf16(y_base + scale * w_row * sum_j S[i][j] B[n][j]).
template <int ROWS>
__device__ __forceinline__ void bg_expand_rows(const EngineParams &p, const EngineSmem &sm, const ExpandItem &it)
{
    const GroupDims &d = it.d;
    const float sc = p.scale[d.a];
    const int kgs = d.rp / 8;
    const int nrows = it.nrows;
    const uint4 *B = reinterpret_cast<const uint4 *>(sm.expand + kBgB);
    const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(sm.expand + kBgY);
    const float *S = reinterpret_cast<const float *>(sm.expand + kBgS);
    for (int nl = threadIdx.x; nl < it.nw; nl += kT) {
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
                const float base = __bfloat162float(ys[i * d.nc + nl]);
                const float v = fmaf(sc * sm.row_w[i], acc[i], base);
                p.y[(int64_t)sm.row_dst[i] * p.ldy + it.n0 + nl] = __float2bfloat16_rn(v);
            }
        }
    }
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

// Put one shrink pipeline stage in flight: 128 token rows x 64 K (cp.async,
// zero for missing rows or K) and the matching A chunk (one bulk copy).
__device__ __forceinline__ void tc_issue_stage(const EngineParams &p, EngineSmem &sm, const GroupDims &d, int nrows,
                                               int k0, int kw, int s, int depth)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = s % depth;
    unsigned char *Xs = sm.shrink + slot * tc_stage_bytes(d.R);
    unsigned char *As = Xs + kTcRows * kTcStageK * 2;
    const int kb = k0 + s * kTcStageK;
    const int vkg = min(8, (kw - s * kTcStageK) / 8);       // K-groups of 8 present in this stage
    const int need = ((vkg + 1) / 2) * 2;                   // K-groups the MMAs read (whole K=16 steps)
    // thread (warp, lane) covers rows 16*warp + (lane & 15), K-groups 2q + (lane >> 4), q = 0..3
    const int row = warp * 16 + (lane & 15);
    const __nv_bfloat16 *xrow = p.x + (int64_t)sm.row_src[row] * p.ldx + kb;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int kg = 2 * q + (lane >> 4);
        if (kg < need) {
            const bool valid = row < nrows && kg < vkg;
            tc::cp_async16(Xs + (kg * kTcRows + row) * 16, valid ? (const void *)(xrow + kg * 8) : (const void *)p.x,
                           valid);
        }
    }
    tc::cp_async_commit();
    if (vkg < need) {   // odd K-group count at the end of K: the last A K-group reads as zero
        uint4 *z = reinterpret_cast<uint4 *>(As + vkg * d.R * 16);
        for (int i = tid; i < d.R; i += kT) z[i] = make_uint4(0u, 0u, 0u, 0u);
        tc::fence_proxy_async_smem();
    }
    if (tid == 0) {
        const __nv_bfloat16 *ablk =
            reinterpret_cast<const __nv_bfloat16 *>(p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)]);
        const uint32_t bytes = (uint32_t)vkg * d.R * 16;
        mbar_arrive_expect_tx(&sm.bar_stage[slot], bytes);
        bulk_g2s(As, ablk + (int64_t)(kb / 8) * d.R * 8, bytes, &sm.bar_stage[slot]);
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

struct TcPhases {
    uint32_t stage, mma, mma_pending, exp;
};

// Tensor-core shrink item: partial = X_rows[:, K-chunk] A[:, K-chunk]^T into
// tensor memory, then out to the tile's scratch slot.  Returns false if a wait
// ran out.
__device__ bool tc_shrink_item(const EngineParams &p, EngineSmem &sm, const GroupDims &d, int g, int tile, int chunk,
                               TcPhases &ph)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = tile * kTcRows;
    const int nrows = min(kTcRows, d.count - r0);
    const int k0 = chunk * kTcKc;
    const int kw = min(kTcKc, p.K - k0);
    const int nst = (kw + kTcStageK - 1) / kTcStageK;
    const int depth = min(tc_depth(d.R), nst);
    if (tid < kTcRows) sm.row_src[tid] = tid < nrows ? p.rows[d.rows_off + r0 + tid] / p.src_div : 0;
    __syncthreads();
    for (int s = 0; s < depth; ++s) tc_issue_stage(p, sm, d, nrows, k0, kw, s, depth);

    const uint32_t idesc = tc::idesc_bf16(kTcRows, d.R);
    bool ok = true;
    for (int s = 0; s < nst && ok; ++s) {
        const int slot = s % depth;
        const int issued = min(nst, s + depth);
        cp_wait_pending(issued - (s + 1));
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bool landed = mbar_wait_bounded(&sm.bar_stage[slot], (ph.stage >> slot) & 1u, p.timeout_ns, p.err);
            sm.flag = landed ? 1 : 0;
            if (landed) {
                tc::fence_after_sync();
                const unsigned char *Xs = sm.shrink + slot * tc_stage_bytes(d.R);
                const unsigned char *As = Xs + kTcRows * kTcStageK * 2;
                const int vkg = min(8, (kw - s * kTcStageK) / 8);
                const int steps = (vkg + 1) / 2;
                for (int j = 0; j < steps; ++j) {
                    const uint64_t ad = tc::smem_desc(smem_u32(Xs) + j * 2 * kTcRows * 16, kTcRows * 16, 128);
                    const uint64_t bd = tc::smem_desc(smem_u32(As) + j * 2 * d.R * 16, d.R * 16, 128);
                    tc::mma_bf16(sm.tmem_base, ad, bd, idesc, (s > 0 || j > 0) ? 1u : 0u);
                }
                tc::mma_commit(&sm.bar_mma[slot]);
            }
        }
        ph.stage ^= 1u << slot;
        __syncthreads();
        ok = sm.flag != 0;
        if (!ok) break;
        ph.mma_pending |= 1u << slot;
        if (s + depth < nst) {   // the slot is refilled: its MMAs must be done reading it
            ok = cta_wait(&sm.bar_mma[slot], (ph.mma >> slot) & 1u, p);
            ph.mma ^= 1u << slot;
            ph.mma_pending &= ~(1u << slot);
            if (ok) tc_issue_stage(p, sm, d, nrows, k0, kw, s + depth, depth);
        }
    }
    // every commit completes in order, so the last one covers all MMAs; retire the rest
    for (int slot = 0; slot < kTcMaxDepth; ++slot) {
        if (ph.mma_pending & (1u << slot)) {
            const bool done = cta_wait(&sm.bar_mma[slot], (ph.mma >> slot) & 1u, p);
            ph.mma ^= 1u << slot;
            ph.mma_pending &= ~(1u << slot);
            ok = ok && done;
        }
    }
    cp_wait_n<0>();
    if (!ok) return false;
    tc::fence_after_sync();

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

// Put a tensor-core expand item's B rows and output rows in flight (the S
// bytes are part of the expected count; they are copied once S is published).
__device__ __forceinline__ void tc_issue_expand(const EngineParams &p, EngineSmem &sm, const ExpandItem &it)
{
    const int tid = threadIdx.x;
    const GroupDims &d = it.d;
    const uint32_t kgs = d.rp / 8;
    const uint32_t b_bytes = kgs * kTcCols * 16;
    const uint32_t s_bytes = kgs * kTcRows * 16;
    if (tid < it.nrows) {
        const int row = p.rows[d.rows_off + it.r0 + tid];
        sm.row_dst[tid] = row;
        sm.row_w[tid] = p.row_weight ? p.row_weight[row] : 1.0f;
        bulk_g2s(sm.expand + kTcY + tid * kTcCols * 2, p.y + (int64_t)row * p.ldy + it.n0, (uint32_t)it.nw * 2,
                 &sm.bar_expand);
    }
    if (tid == 0) {
        const __nv_bfloat16 *bblk =
            reinterpret_cast<const __nv_bfloat16 *>(p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)]);
        // 128 output columns = one half of a 256-row B tile: rp/8 runs of 128 x 16 bytes
        const int btile = p.slice_tile_off[it.s] + it.c / 2, half = it.c & 1;
        mbar_arrive_expect_tx(&sm.bar_expand, b_bytes + s_bytes + (uint32_t)it.nrows * it.nw * 2);
        for (uint32_t kg = 0; kg < kgs; ++kg)
            bulk_g2s(sm.expand + kTcB + kg * kTcCols * 16,
                     bblk + ((int64_t)(btile * kgs + kg) * kNTile + half * kTcCols) * 8, kTcCols * 16,
                     &sm.bar_expand);
    }
}

__device__ __forceinline__ void issue_expand(const EngineParams &p, EngineSmem &sm, const ExpandItem &it)
{
    if (it.d.tc) {
        tc_issue_expand(p, sm, it);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupDims &d = it.d;
    if (warp == 1 && lane < it.nrows) {
        const int row = p.rows[d.rows_off + it.r0 + lane];
        sm.row_dst[lane] = row;
        sm.row_w[lane] = p.row_weight ? p.row_weight[row] : 1.0f;
        bulk_g2s(sm.expand + kBgY + (size_t)lane * d.nc * 2, p.y + (int64_t)row * p.ldy + it.n0, (uint32_t)it.nw * 2,
                 &sm.bar_expand);
    }
    if (tid == 0) {
        const __nv_bfloat16 *bblk =
            reinterpret_cast<const __nv_bfloat16 *>(p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)]);
        const int tile0 = p.slice_tile_off[it.s] + it.c * (d.nc / kNTile);
        const int ntl = (it.nw + kNTile - 1) / kNTile;
        const uint32_t b_bytes = (uint32_t)ntl * kNTile * d.rp * 2;
        mbar_arrive_expect_tx(&sm.bar_expand, b_bytes + it.nrows * (uint32_t)it.nw * 2);
        bulk_g2s(sm.expand + kBgB, bblk + (int64_t)tile0 * kNTile * d.rp, b_bytes, &sm.bar_expand);
    }
}

// Tensor-core expand: D[128 x 128] = S[:, slice block] B_half^T, then
// y = bf16(y_base + scale * w_row * D) for the tile's rows.
__device__ bool tc_expand_item(const EngineParams &p, EngineSmem &sm, const ExpandItem &it, TcPhases &ph)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupDims &d = it.d;
    if (tid == 0) {
        const uint32_t steps = d.rp / 16;
        tc::fence_after_sync();
        for (uint32_t j = 0; j < steps; ++j) {
            const uint64_t ad = tc::smem_desc(smem_u32(sm.expand + kTcS) + j * 2 * kTcRows * 16, kTcRows * 16, 128);
            const uint64_t bd = tc::smem_desc(smem_u32(sm.expand + kTcB) + j * 2 * kTcCols * 16, kTcCols * 16, 128);
            tc::mma_bf16(sm.tmem_base + kTmemExpandCol, ad, bd, tc::idesc_bf16(kTcRows, kTcCols), j > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.bar_mma_exp);
    }
    const bool ok = cta_wait(&sm.bar_mma_exp, ph.exp, p);
    ph.exp ^= 1u;
    if (!ok) return false;
    tc::fence_after_sync();
    // warp w: rows 32 (w % 4) + lane, columns 64 (w / 4) .. + 64
    const int row = (warp & 3) * 32 + lane;
    const int cbase = (warp >> 2) * 64;
    const float sc = p.scale[d.a] * (row < it.nrows ? sm.row_w[row] : 0.f);
    const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(sm.expand + kTcY) + row * kTcCols;
    __nv_bfloat16 *yg = p.y + (int64_t)(row < it.nrows ? sm.row_dst[row] : 0) * p.ldy + it.n0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c0 = cbase + h * 32;
        float v[32];
        tc::tmem_ld32(sm.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kTmemExpandCol + c0, v);
        if (row < it.nrows) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + 8 * q;
                if (c < it.nw) {
                    const uint4 yb = *reinterpret_cast<const uint4 *>(ys + c);
                    float yf[8];
                    bf16x8_to_f32(yb, yf);
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = __float2bfloat16_rn(fmaf(sc, v[8 * q + e], yf[e]));
                    *reinterpret_cast<uint4 *>(yg + c) = *reinterpret_cast<const uint4 *>(o);
                }
            }
        }
    }
    tc::fence_before_sync();
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
    if (p.trace != nullptr && tid > 0 && tid < 8 && (int)blockIdx.x < p.trace_ctas)
        p.trace[(size_t)blockIdx.x * 8 + tid] = 0;
    stamp(p, 0);

    // ---- prologue: one round trip for the count, the first group records and the stored ranks ----
    if (tid == 0) {
        sm.G = *p.num_groups;
        sm.flag = 0;
        mbar_init(&sm.bar_shrink, 1);
        mbar_init(&sm.bar_expand, 1);
        for (int i = 0; i < kTcMaxDepth; ++i) {
            mbar_init(&sm.bar_stage[i], 1);
            mbar_init(&sm.bar_mma[i], 1);
        }
        mbar_init(&sm.bar_mma_exp, 1);
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
        // per-group item counts and their exclusive prefix sums, 32 groups per step
        int4 carry = make_int4(0, 0, 0, 0);
        bool bad = false, any_tc = false;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int4 v = make_int4(0, 0, 0, 0);
            if (g < G) {
                const int4 gr = g < kGroupCache ? sm.grp[g] : p.groups[g];
                if (gr.x < 0 || gr.x >= p.L || gr.y < 0 || gr.y >= p.num_experts || gr.z < 0 || gr.w < 1 ||
                    (int64_t)gr.z + gr.w > p.rows_capacity) {
                    bad = true;   // a workspace that lora_build_segments never filled
                } else {
                    const GroupDims d = group_dims(p, sm, g);
                    v = make_int4(d.tiles * d.n_kc, d.tiles * d.n_nc, d.tiles, d.scratch);
                    any_tc |= d.tc;
                }
            }
            int4 incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int4 u = shfl_up4(incl, o);
                if (lane >= o) incl = add4(incl, u);
            }
            if (g < G) {
                sm.sh_pre[g] = carry.x + incl.x - v.x;
                sm.ex_pre[g] = carry.y + incl.y - v.y;
                sm.tile_pre[g] = carry.z + incl.z - v.z;
                sm.part_pre[g] = carry.w + incl.w - v.w;
            }
            carry = add4(carry, make_int4(__shfl_sync(0xffffffffu, incl.x, 31), __shfl_sync(0xffffffffu, incl.y, 31),
                                          __shfl_sync(0xffffffffu, incl.z, 31), __shfl_sync(0xffffffffu, incl.w, 31)));
        }
        bad = __any_sync(0xffffffffu, bad);
        any_tc = __any_sync(0xffffffffu, any_tc);
        if (lane == 0) {
            sm.sh_pre[G] = carry.x;
            sm.ex_pre[G] = carry.y;
            sm.tile_pre[G] = carry.z;
            sm.part_pre[G] = carry.w;
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
    if (use_tc) {   // one warp allocates the tensor memory this CTA's MMAs accumulate into
        if (warp == 0) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    uint32_t ph_shrink = 0, ph_expand = 0;
    TcPhases tph = {0u, 0u, 0u, 0u};
    const int grid = gridDim.x;
    bool alive = true;
    stamp(p, 1);

    // The first expand item's operands do not depend on any shrink result: they
    // are put in flight right after the first shrink item's copies, so they
    // arrive while this CTA does its shrink work.
    const bool prefetched = blockIdx.x < n_expand;
    bool expand_in_flight = false;
    if (prefetched && (int)blockIdx.x >= n_shrink) {
        issue_expand(p, sm, decode_expand(p, sm, G, blockIdx.x));
        expand_in_flight = true;
    }

    // ------------------------------------------------------------------
    // shrink items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_shrink && alive; item += grid) {
        const int g = find_group(sm.sh_pre, G, item);
        const GroupDims d = group_dims(p, sm, g);
        const int local = item - sm.sh_pre[g];
        const int tile = local / d.n_kc, chunk = local % d.n_kc;
        const int tg = sm.tile_pre[g] + tile;
        if (d.tc) {
            if (prefetched && item == (int)blockIdx.x) {
                issue_expand(p, sm, decode_expand(p, sm, G, blockIdx.x));
                expand_in_flight = true;
            }
            if (!tc_shrink_item(p, sm, d, g, tile, chunk, tph)) {
                alive = false;
                break;
            }
            if (item == (int)blockIdx.x) stamp(p, 2);
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
            stamp(p, 3);
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
            bulk_g2s(sm.shrink + kBgA, ablk + (int64_t)(k0 / 8) * d.R * 8, a_bytes, &sm.bar_shrink);
        }
        if (warp == 1 && lane < nrows) {
            const int src = p.rows[d.rows_off + r0 + lane] / p.src_div;
            bulk_g2s(sm.shrink + kBgX + (size_t)lane * d.kc * 2, p.x + (int64_t)src * p.ldx + k0, x_bytes,
                     &sm.bar_shrink);
        }
        if (prefetched && item == (int)blockIdx.x) {
            issue_expand(p, sm, decode_expand(p, sm, G, blockIdx.x));
            expand_in_flight = true;
        }
        const bool ok = cta_wait(&sm.bar_shrink, ph_shrink, p);
        ph_shrink ^= 1;
        if (!ok) {
            alive = false;
            break;
        }
        if (item == (int)blockIdx.x) stamp(p, 2);

        // partial dot products: thread (ks, j) covers row j of A, K-groups ks, ks+nks, ...
        const int R = d.R;
        const int nks = kT / R;
        if (nrows <= 2) bg_shrink_rows<2>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 4) bg_shrink_rows<4>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 8) bg_shrink_rows<8>(sm, R, kw, d.kc / 8, nrows);
        else bg_shrink_rows<16>(sm, R, kw, d.kc / 8, nrows);
        __syncthreads();
        const float *red = reinterpret_cast<const float *>(sm.shrink + kBgRed);
        float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * R + (int64_t)chunk * nrows * R;
        for (int idx = tid; idx < nrows * R; idx += kT) {
            const int i = idx / R, jj = idx % R;
            float s = 0.f;
            for (int q = 0; q < nks; ++q) s += red[(q * kBgmvRows + i) * R + jj];
            dst[idx] = s;
        }
        __syncthreads();
        if (tid == 0 && !p.withhold) release_add(&p.sync[tg * 4 + 0], 1);
        stamp(p, 3);
    }

    // ------------------------------------------------------------------
    // expand items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_expand && alive; item += grid) {
        const ExpandItem it = decode_expand(p, sm, G, item);
        const GroupDims &d = it.d;
        if (!(prefetched && item == (int)blockIdx.x)) issue_expand(p, sm, it);
        expand_in_flight = true;

        // wait until the tile's shrink results are published
        if (tid == 0) {
            const bool ok = d.tc ? wait_counter(&p.sync[it.tg * 4 + 2], 1, p)
                                 : wait_counter(&p.sync[it.tg * 4 + 0], d.n_kc, p);
            if (d.tc) {
                const uint32_t s_bytes = (uint32_t)(d.rp / 8) * kTcRows * 16;
                if (ok) {
                    // S was written by another CTA through ordinary stores: order them before the async copy
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    const __nv_bfloat16 *S = tc_S(p, sm, d, it.g, it.tile) + (int64_t)it.sa * (d.rp / 8) * kTcRows * 8;
                    bulk_g2s(sm.expand + kTcS, S, s_bytes, &sm.bar_expand);
                } else {
                    mbar_complete_tx(&sm.bar_expand, s_bytes);   // the S bytes will never come
                }
            }
            sm.flag = ok ? 1 : 0;
        }
        if (item == (int)blockIdx.x) stamp(p, 4);
        __syncthreads();
        const bool ready = sm.flag != 0;
        if (ready && !d.tc) {
            // S[i][j] = sum over K-chunks q (ascending) of the published partials; loads first, then the sum
            float *S = reinterpret_cast<float *>(sm.expand + kBgS);
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
        __syncthreads();
        if (item == (int)blockIdx.x) stamp(p, 5);
        if (tid == 0 && ready) {
            const int old = atomicAdd(&p.sync[it.tg * 4 + 1], 1);
            if (old == d.n_nc - 1) {   // last consumer of this tile resets its counters
                p.sync[it.tg * 4 + 0] = 0;
                p.sync[it.tg * 4 + 1] = 0;
                p.sync[it.tg * 4 + 2] = 0;
            }
        }
        const bool landed = cta_wait(&sm.bar_expand, ph_expand, p);
        ph_expand ^= 1;
        expand_in_flight = false;
        if (!landed) {
            alive = false;
            break;
        }
        if (item == (int)blockIdx.x) stamp(p, 6);
        if (!ready) {
            __syncthreads();
            continue;
        }
        if (d.tc) {
            if (!tc_expand_item(p, sm, it, tph)) {
                alive = false;
                break;
            }
        } else if (it.nrows <= 2) bg_expand_rows<2>(p, sm, it);
        else if (it.nrows <= 4) bg_expand_rows<4>(p, sm, it);
        else if (it.nrows <= 8) bg_expand_rows<8>(p, sm, it);
        else bg_expand_rows<16>(p, sm, it);
        __syncthreads();
    }
    // a CTA that gave up still lets its own copies land before it leaves
    if (expand_in_flight) mbar_wait_bounded(&sm.bar_expand, ph_expand, p.timeout_ns, p.err);
    stamp(p, 7);
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
