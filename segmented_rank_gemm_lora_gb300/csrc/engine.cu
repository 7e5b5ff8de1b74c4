// The fused shrink -> expand -> add engine behind lora_apply and lora_moe_delta.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 2.3: every segment is a
// shrink X_seg A_i^T followed by an expand with B_i^T added to the base rows,
// and all segments run in one operator instance, spread over the cores;
// section 2.4: tile the token dimension first, then the rank/K dimension so a
// piece of A fits on chip, accumulating the pieces; section 4.2: the
// rank-sized intermediate S accumulates in fp32.
//
// GB300 form.  One persistent grid (one CTA per SM) walks a work list that
// every CTA derives, identically, from the segment table:
//   tile         = up to 16 rows of one group (segment, or MoE adapter/expert);
//   shrink item  = (tile, K-chunk): fp32 partial S = X_rows[:, chunk] A[:, chunk]^T,
//                  written to an L2-resident scratch slot; the tile's counter is
//                  then bumped with release semantics;
//   expand item  = (tile, N-chunk of one slice): waits (bounded) until all
//                  K-chunks of the tile are published, sums the partials in a
//                  fixed order, multiplies by the B rows of the chunk and adds
//                  scale * result into the output rows.
// CTA b takes shrink items b, b+grid, ... and then expand items b, b+grid, ...;
// it finishes all of its shrink items before it waits on anything, and the
// whole grid is co-resident (cooperative launch), so every wait ends.
// Operand chunks are single contiguous runs in the packed table and land in
// shared memory through bulk async copies completing on mbarriers, so one
// thread puts a CTA's whole chunk in flight at once.
// The sum order never depends on timing or on which rows share a tile, so the
// same inputs always give the same bits.
#include "common.cuh"

namespace lora {

constexpr int kGroupCap = 2048;                     // groups per launch held in shared memory
constexpr int kChunkBytes = 32 * 1024;              // target bytes of one A or B chunk
constexpr int kMaxKc = 1024;                        // K elements of a chunk at the smallest R
constexpr int kMaxNc = 1024;                        // N rows of a chunk at the smallest stored rank

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

constexpr int kGroupCache = 512;                    // group records cached in shared memory
constexpr int kRankCache = 1024;                    // stored ranks cached in shared memory

struct __align__(128) EngineSmem {
    uint64_t bar_shrink, bar_expand;
    int32_t row_dst[kBgmvRows];
    float row_w[kBgmvRows];
    int32_t flag;
    int32_t G;
    int32_t sh_pre[kGroupCap + 1];     // shrink items before group g
    int32_t ex_pre[kGroupCap + 1];     // expand items before group g
    int32_t tile_pre[kGroupCap + 1];   // tiles before group g
    int32_t part_pre[kGroupCap + 1];   // partial floats before group g
    int4 grp[kGroupCache];             // (adapter, expert, rows_off, count) of the first groups
    int32_t rp_cache[kRankCache];      // stored rank of the first adapters
    __align__(128) uint4 A[kChunkBytes / 16];          // packed A chunk [kc/8][R][8]
    __align__(128) uint4 X[kBgmvRows * kMaxKc / 8];     // input rows [16][kc]
    __align__(128) uint4 B[kChunkBytes / 16];          // packed B tiles [nc/256][rp/8][256][8]
    __align__(128) uint4 Y[kBgmvRows * kMaxNc / 8];     // output rows [16][nc]
    float red[kEngineThreads * kBgmvRows];              // [nks][16][R]
    float S[kBgmvRows * kMaxRank];                      // reduced S of one slice block
};

size_t engine_smem_bytes(int) { return sizeof(EngineSmem); }

struct GroupDims {
    int a, e, rows_off, count;
    int rp, R, kc, n_kc, nc, n_nc, tiles;
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
    d.kc = kc_for(d.R);
    d.n_kc = (p.K + d.kc - 1) / d.kc;
    d.nc = nc_for(d.rp);
    int n = 0;
    for (int s = 0; s < p.n_slices; ++s) n += (p.slice_n[s] + d.nc - 1) / d.nc;
    d.n_nc = n;
    d.tiles = (d.count + kBgmvRows - 1) / kBgmvRows;
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

// One expand item, decoded.
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
    it.n0 = p.slice_off[s] + c * it.d.nc;
    it.nw = min(it.d.nc, p.slice_off[s] + p.slice_n[s] - it.n0);
    it.r0 = it.tile * kBgmvRows;
    it.nrows = min(kBgmvRows, it.d.count - it.r0);
    it.sa = (p.n_a == 1) ? 0 : s;
    it.tg = sm.tile_pre[it.g] + it.tile;
    it.c = c;
    return it;
}

// Put the B chunk and the output rows of an expand item in flight (no waiting).
__device__ __forceinline__ void issue_expand(const EngineParams &p, EngineSmem &sm, const ExpandItem &it)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupDims &d = it.d;
    if (warp == 1 && lane < it.nrows) {
        const int row = p.rows[d.rows_off + it.r0 + lane];
        sm.row_dst[lane] = row;
        sm.row_w[lane] = p.row_weight ? p.row_weight[row] : 1.0f;
        bulk_g2s(reinterpret_cast<unsigned char *>(sm.Y) + (size_t)lane * d.nc * 2, p.y + (int64_t)row * p.ldy + it.n0,
                 (uint32_t)it.nw * 2, &sm.bar_expand);
    }
    if (tid == 0) {
        const __nv_bfloat16 *bblk =
            reinterpret_cast<const __nv_bfloat16 *>(p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)]);
        const int tile0 = p.slice_tile_off[it.s] + it.c * (d.nc / kNTile);
        const int ntl = (it.nw + kNTile - 1) / kNTile;
        const uint32_t b_bytes = (uint32_t)ntl * kNTile * d.rp * 2;
        mbar_arrive_expect_tx(&sm.bar_expand, b_bytes + it.nrows * (uint32_t)it.nw * 2);
        bulk_g2s(sm.B, bblk + (int64_t)tile0 * kNTile * d.rp, b_bytes, &sm.bar_expand);
    }
}

// Shrink partial for up to ROWS rows: thread (ks, j) accumulates row j of the
// A chunk against every row over K-groups ks, ks + nks, ... and leaves its
// sums in red[ks][i][j].
template <int ROWS>
__device__ __forceinline__ void shrink_rows(EngineSmem &sm, int R, int kw, int xstride, int nrows)
{
    const int tid = threadIdx.x;
    const int nks = kEngineThreads / R;
    const int j = tid % R, ks = tid / R;
    if (ks >= nks) return;
    float acc[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i) acc[i] = 0.f;
    const int kgs = kw / 8;
    for (int kg = ks; kg < kgs; kg += nks) {
        float af[8];
        bf16x8_to_f32(sm.A[kg * R + j], af);
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            if (i < nrows) {
                float xf[8];
                bf16x8_to_f32(sm.X[i * xstride + kg], xf);
                float s = acc[i];
#pragma unroll
                for (int u = 0; u < 8; ++u) s = fmaf(xf[u], af[u], s);
                acc[i] = s;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
        if (i < nrows) sm.red[(ks * kBgmvRows + i) * R + j] = acc[i];
}

// Expand for up to ROWS rows: thread per output column of the chunk;
// y = bf16(y_base + scale * w_row * sum_j S[i][j] B[n][j]).
template <int ROWS>
__device__ __forceinline__ void expand_rows(const EngineParams &p, const EngineSmem &sm, const GroupDims &d,
                                            const ExpandItem &it)
{
    const float sc = p.scale[d.a];
    const int kgs = d.rp / 8;
    const int nrows = it.nrows;
    const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(sm.Y);
    for (int nl = threadIdx.x; nl < it.nw; nl += kEngineThreads) {
        float acc[ROWS];
#pragma unroll
        for (int i = 0; i < ROWS; ++i) acc[i] = 0.f;
        const int tl = nl / kNTile, row = nl % kNTile;
        for (int kg = 0; kg < kgs; ++kg) {
            float bfv[8];
            bf16x8_to_f32(sm.B[(tl * kgs + kg) * kNTile + row], bfv);
#pragma unroll
            for (int i = 0; i < ROWS; ++i) {
                if (i < nrows) {
                    float a = acc[i];
#pragma unroll
                    for (int u = 0; u < 8; ++u) a = fmaf(sm.S[i * kMaxRank + kg * 8 + u], bfv[u], a);
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

// Phase stamps for lora_set_trace (slot k of this block); the callers stamp
// the once-only phases on their first pass.
__device__ __forceinline__ void stamp(const EngineParams &p, int k)
{
    if (p.trace != nullptr && threadIdx.x == 0 && (int)blockIdx.x < p.trace_ctas)
        p.trace[(size_t)blockIdx.x * 8 + k] = globaltimer();
}

__global__ void __launch_bounds__(kEngineThreads, 1) engine_kernel(const __grid_constant__ EngineParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
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
        fence_mbar_init();
    }
    const int gpre = min(p.group_capacity, kGroupCache);
    for (int g = tid; g < gpre; g += kEngineThreads) sm.grp[g] = p.groups[g];
    for (int a = tid; a < min(p.L, kRankCache); a += kEngineThreads) sm.rp_cache[a] = p.rpad[a];
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
        bool bad = false;
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
                    v = make_int4(d.tiles * d.n_kc, d.tiles * d.n_nc, d.tiles, d.n_kc * d.count * d.R);
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
        if (lane == 0) {
            sm.sh_pre[G] = carry.x;
            sm.ex_pre[G] = carry.y;
            sm.tile_pre[G] = carry.z;
            sm.part_pre[G] = carry.w;
            sm.flag = bad ? 1 : 0;
        }
    }
    __syncthreads();
    if (sm.flag) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    const int n_shrink = sm.sh_pre[G], n_expand = sm.ex_pre[G], n_tiles = sm.tile_pre[G], n_part = sm.part_pre[G];
    if (n_tiles > p.max_tiles || (int64_t)n_part > p.partial_floats) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }

    uint32_t ph_shrink = 0, ph_expand = 0;
    const int grid = gridDim.x;
    stamp(p, 1);

    // The first expand item's operands do not depend on any shrink result: they
    // are put in flight right after the first shrink item's copies, so they
    // arrive while this CTA does its shrink work.
    const bool prefetched = blockIdx.x < n_expand;
    if (prefetched && (int)blockIdx.x >= n_shrink) issue_expand(p, sm, decode_expand(p, sm, G, blockIdx.x));

    // ------------------------------------------------------------------
    // shrink items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_shrink; item += grid) {
        const int g = find_group(sm.sh_pre, G, item);
        const GroupDims d = group_dims(p, sm, g);
        const int local = item - sm.sh_pre[g];
        const int tile = local / d.n_kc, chunk = local % d.n_kc;
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
            bulk_g2s(sm.A, ablk + (int64_t)(k0 / 8) * d.R * 8, a_bytes, &sm.bar_shrink);
        }
        if (warp == 1 && lane < nrows) {
            const int src = p.rows[d.rows_off + r0 + lane] / p.src_div;
            bulk_g2s(reinterpret_cast<unsigned char *>(sm.X) + (size_t)lane * d.kc * 2,
                     p.x + (int64_t)src * p.ldx + k0, x_bytes, &sm.bar_shrink);
        }
        if (prefetched && item == (int)blockIdx.x) issue_expand(p, sm, decode_expand(p, sm, G, blockIdx.x));
        const bool ok = cta_wait(&sm.bar_shrink, ph_shrink, p);
        ph_shrink ^= 1;
        if (!ok) return;   // copies never land only if the GPU is wedged; nothing else waits on us
        if (item == (int)blockIdx.x) stamp(p, 2);

        // partial dot products: thread (ks, j) covers row j of A, K-groups ks, ks+nks, ...
        const int R = d.R;
        const int nks = kEngineThreads / R;
        if (nrows <= 2) shrink_rows<2>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 4) shrink_rows<4>(sm, R, kw, d.kc / 8, nrows);
        else if (nrows <= 8) shrink_rows<8>(sm, R, kw, d.kc / 8, nrows);
        else shrink_rows<16>(sm, R, kw, d.kc / 8, nrows);
        __syncthreads();
        const int tg = sm.tile_pre[g] + tile;
        float *dst = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * R + (int64_t)chunk * nrows * R;
        for (int idx = tid; idx < nrows * R; idx += kEngineThreads) {
            const int i = idx / R, jj = idx % R;
            float s = 0.f;
            for (int q = 0; q < nks; ++q) s += sm.red[(q * kBgmvRows + i) * R + jj];
            dst[idx] = s;
        }
        __syncthreads();
        if (tid == 0 && !p.withhold) release_add(&p.sync[tg * 4 + 0], 1);
        stamp(p, 3);
    }

    // ------------------------------------------------------------------
    // expand items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_expand; item += grid) {
        const ExpandItem it = decode_expand(p, sm, G, item);
        const GroupDims &d = it.d;
        if (!(prefetched && item == blockIdx.x)) issue_expand(p, sm, it);

        // wait until every K-chunk of this tile is published
        if (tid == 0) {
            int ok = 1;
            const int32_t *cnt = &p.sync[it.tg * 4 + 0];
            if (ld_acquire_gpu(cnt) < d.n_kc) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_gpu(cnt) < d.n_kc) {
                    if (globaltimer() - t0 > p.timeout_ns) {
                        atomicOr(p.err, kErrTimeout);
                        ok = 0;
                        break;
                    }
                    nanosleep_ns(32);
                }
            }
            sm.flag = ok;
        }
        if (item == (int)blockIdx.x) stamp(p, 4);
        __syncthreads();
        const bool ready = sm.flag != 0;
        if (ready) {
            // S[i][j] = sum over K-chunks q (ascending) of the published partials; loads first, then the sum
            const int64_t stride = (int64_t)it.nrows * d.R;
            const float *part = p.partials + sm.part_pre[it.g] + (int64_t)d.n_kc * it.r0 * d.R + it.sa * d.rp;
            for (int idx = tid; idx < it.nrows * d.rp; idx += kEngineThreads) {
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
                sm.S[i * kMaxRank + jj] = acc;
            }
        }
        __syncthreads();
        if (item == (int)blockIdx.x) stamp(p, 5);
        if (tid == 0 && ready) {
            const int old = atomicAdd(&p.sync[it.tg * 4 + 1], 1);
            if (old == d.n_nc - 1) {   // last consumer of this tile resets its counters
                p.sync[it.tg * 4 + 0] = 0;
                p.sync[it.tg * 4 + 1] = 0;
            }
        }
        const bool landed = cta_wait(&sm.bar_expand, ph_expand, p);
        ph_expand ^= 1;
        if (!landed) return;
        if (item == (int)blockIdx.x) stamp(p, 6);
        if (!ready) {
            __syncthreads();
            continue;
        }

        const float sc = p.scale[d.a];
        if (it.nrows <= 2) expand_rows<2>(p, sm, d, it);
        else if (it.nrows <= 4) expand_rows<4>(p, sm, d, it);
        else if (it.nrows <= 8) expand_rows<8>(p, sm, d, it);
        else expand_rows<16>(p, sm, d, it);
        (void)sc;
        __syncthreads();
    }
    stamp(p, 7);
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
