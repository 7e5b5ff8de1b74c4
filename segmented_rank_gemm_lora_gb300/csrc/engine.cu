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

struct __align__(128) EngineSmem {
    uint64_t bar_shrink, bar_expand;
    int32_t row_src[kBgmvRows];
    int32_t row_dst[kBgmvRows];
    float row_w[kBgmvRows];
    int32_t flag;
    int32_t totals[4];
    int32_t scan_tmp[40];
    int32_t sh_pre[kGroupCap + 1];     // shrink items before group g
    int32_t ex_pre[kGroupCap + 1];     // expand items before group g
    int32_t tile_pre[kGroupCap + 1];   // tiles before group g
    int32_t part_pre[kGroupCap + 1];   // partial floats before group g
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

__device__ __forceinline__ GroupDims group_dims(const EngineParams &p, int g)
{
    GroupDims d;
    const int4 gr = p.groups[g];
    d.a = gr.x;
    d.e = gr.y;
    d.rows_off = gr.z;
    d.count = gr.w;
    d.rp = p.rpad[d.a];
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

// exclusive block scan (256 threads) of a[0..n) in place, returns the total
__device__ int32_t scan256(int32_t *a, int n, int32_t *tmp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kEngineThreads - 1) / kEngineThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    int32_t v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) tmp[warp] = v;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int w = 0; w < kEngineThreads / 32; ++w) {
            int32_t c = tmp[w];
            tmp[w] = run;
            run += c;
        }
        tmp[kEngineThreads / 32] = run;
    }
    __syncthreads();
    int32_t run = tmp[warp] + v - local;
    for (int i = lo; i < hi; ++i) {
        int32_t c = a[i];
        a[i] = run;
        run += c;
    }
    const int32_t total = tmp[kEngineThreads / 32];
    __syncthreads();
    return total;
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

__global__ void __launch_bounds__(kEngineThreads, 1) engine_kernel(const __grid_constant__ EngineParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    EngineSmem &sm = *reinterpret_cast<EngineSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int G = *p.num_groups;
    if (G <= 0) return;
    if (G > p.group_capacity || G > kGroupCap) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }

    if (tid == 0) {
        mbar_init(&sm.bar_shrink, 1);
        mbar_init(&sm.bar_expand, 1);
        fence_mbar_init();
    }

    // ---- work list, derived identically by every CTA ----
    if (tid == 0) sm.flag = 0;
    __syncthreads();
    for (int g = tid; g < G; g += kEngineThreads) {
        const int4 gr = p.groups[g];
        if (gr.x < 0 || gr.x >= p.L || gr.y < 0 || gr.y >= p.num_experts || gr.z < 0 || gr.w < 1 ||
            (int64_t)gr.z + gr.w > p.rows_capacity)
            sm.flag = 1;   // a workspace that lora_build_segments never filled
    }
    __syncthreads();
    if (sm.flag) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }
    for (int g = tid; g < G; g += kEngineThreads) {
        const GroupDims d = group_dims(p, g);
        sm.sh_pre[g] = d.tiles * d.n_kc;
        sm.ex_pre[g] = d.tiles * d.n_nc;
        sm.tile_pre[g] = d.tiles;
        sm.part_pre[g] = d.n_kc * d.count * d.R;
    }
    __syncthreads();
    const int n_shrink = scan256(sm.sh_pre, G, sm.scan_tmp);
    const int n_expand = scan256(sm.ex_pre, G, sm.scan_tmp);
    const int n_tiles = scan256(sm.tile_pre, G, sm.scan_tmp);
    const int n_part = scan256(sm.part_pre, G, sm.scan_tmp);
    if (tid == 0) {
        sm.sh_pre[G] = n_shrink;
        sm.ex_pre[G] = n_expand;
        sm.tile_pre[G] = n_tiles;
        sm.part_pre[G] = n_part;
    }
    __syncthreads();
    if (n_tiles > p.max_tiles || (int64_t)n_part > p.partial_floats) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, kErrWorkspace);
        return;
    }

    uint32_t ph_shrink = 0, ph_expand = 0;
    const int grid = gridDim.x;

    // ------------------------------------------------------------------
    // shrink items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_shrink; item += grid) {
        const int g = find_group(sm.sh_pre, G, item);
        const GroupDims d = group_dims(p, g);
        const int local = item - sm.sh_pre[g];
        const int tile = local / d.n_kc, chunk = local % d.n_kc;
        const int r0 = tile * kBgmvRows;
        const int nrows = min(kBgmvRows, d.count - r0);
        const int k0 = chunk * d.kc;
        const int kw = min(d.kc, p.K - k0);
        if (tid < nrows) sm.row_src[tid] = p.rows[d.rows_off + r0 + tid] / p.src_div;
        __syncthreads();

        const __nv_bfloat16 *ablk =
            reinterpret_cast<const __nv_bfloat16 *>(p.a_ptr[d.a * p.E_A + (p.E_A == 1 ? 0 : d.e)]);
        const uint32_t a_bytes = (uint32_t)(kw / 8) * d.R * 16;
        const uint32_t x_bytes = (uint32_t)kw * 2;
        if (tid == 0) {
            mbar_arrive_expect_tx(&sm.bar_shrink, a_bytes + nrows * x_bytes);
            bulk_g2s(sm.A, ablk + (int64_t)(k0 / 8) * d.R * 8, a_bytes, &sm.bar_shrink);
        }
        if (warp == 1 && lane < nrows) {
            bulk_g2s(reinterpret_cast<unsigned char *>(sm.X) + (size_t)lane * d.kc * 2,
                     p.x + (int64_t)sm.row_src[lane] * p.ldx + k0, x_bytes, &sm.bar_shrink);
        }
        const bool ok = cta_wait(&sm.bar_shrink, ph_shrink, p);
        ph_shrink ^= 1;
        if (!ok) return;   // copies never land only if the GPU is wedged; nothing else waits on us

        // partial dot products: thread (ks, j) covers row j of A, K-groups ks, ks+nks, ...
        const int R = d.R;
        const int nks = kEngineThreads / R;
        const int j = tid % R, ks = tid / R;
        float acc[kBgmvRows];
#pragma unroll
        for (int i = 0; i < kBgmvRows; ++i) acc[i] = 0.f;
        if (ks < nks) {
            const int kgs = kw / 8;
            const int xstride = d.kc / 8;
            for (int kg = ks; kg < kgs; kg += nks) {
                float af[8];
                bf16x8_to_f32(sm.A[kg * R + j], af);
#pragma unroll
                for (int i = 0; i < kBgmvRows; ++i) {
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
            for (int i = 0; i < kBgmvRows; ++i)
                if (i < nrows) sm.red[(ks * kBgmvRows + i) * R + j] = acc[i];
        }
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
        if (tid == 0 && !p.withhold) {
            __threadfence();
            atom_add_release_gpu(&p.sync[tg * 4 + 0], 1);
        }
    }

    // ------------------------------------------------------------------
    // expand items
    // ------------------------------------------------------------------
    for (int item = blockIdx.x; item < n_expand; item += grid) {
        const int g = find_group(sm.ex_pre, G, item);
        const GroupDims d = group_dims(p, g);
        const int local = item - sm.ex_pre[g];
        const int tile = local / d.n_nc;
        int c = local % d.n_nc;
        int s = 0;
        for (; s < p.n_slices; ++s) {
            const int cs = (p.slice_n[s] + d.nc - 1) / d.nc;
            if (c < cs) break;
            c -= cs;
        }
        const int n0 = p.slice_off[s] + c * d.nc;
        const int nw = min(d.nc, p.slice_off[s] + p.slice_n[s] - n0);
        const int r0 = tile * kBgmvRows;
        const int nrows = min(kBgmvRows, d.count - r0);
        const int sa = (p.n_a == 1) ? 0 : s;
        const int tg = sm.tile_pre[g] + tile;
        if (tid < nrows) {
            const int row = p.rows[d.rows_off + r0 + tid];
            sm.row_dst[tid] = row;
            sm.row_w[tid] = p.row_weight ? p.row_weight[row] : 1.0f;
        }
        __syncthreads();

        const __nv_bfloat16 *bblk =
            reinterpret_cast<const __nv_bfloat16 *>(p.b_ptr[d.a * p.E_B + (p.E_B == 1 ? 0 : d.e)]);
        const int tile0 = p.slice_tile_off[s] + c * (d.nc / kNTile);
        const int ntl = (nw + kNTile - 1) / kNTile;
        const uint32_t b_bytes = (uint32_t)ntl * kNTile * d.rp * 2;
        const uint32_t y_bytes = (uint32_t)nw * 2;
        if (tid == 0) {
            mbar_arrive_expect_tx(&sm.bar_expand, b_bytes + nrows * y_bytes);
            bulk_g2s(sm.B, bblk + (int64_t)tile0 * kNTile * d.rp, b_bytes, &sm.bar_expand);
        }
        if (warp == 1 && lane < nrows) {
            bulk_g2s(reinterpret_cast<unsigned char *>(sm.Y) + (size_t)lane * d.nc * 2,
                     p.y + (int64_t)sm.row_dst[lane] * p.ldy + n0, y_bytes, &sm.bar_expand);
        }

        // wait until every K-chunk of this tile is published
        if (tid == 0) {
            int ok = 1;
            const int32_t *cnt = &p.sync[tg * 4 + 0];
            if (ld_acquire_gpu(cnt) < d.n_kc) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_gpu(cnt) < d.n_kc) {
                    if (globaltimer() - t0 > p.timeout_ns) {
                        atomicOr(p.err, kErrTimeout);
                        ok = 0;
                        break;
                    }
                    nanosleep_ns(64);
                }
            }
            sm.flag = ok;
        }
        __syncthreads();
        const bool ready = sm.flag != 0;
        if (ready) {
            const float *part = p.partials + sm.part_pre[g] + (int64_t)d.n_kc * r0 * d.R;
            for (int idx = tid; idx < nrows * d.rp; idx += kEngineThreads) {
                const int i = idx / d.rp, jj = idx % d.rp;
                float acc = 0.f;
                for (int q = 0; q < d.n_kc; ++q)
                    acc += __ldcg(part + ((int64_t)q * nrows + i) * d.R + sa * d.rp + jj);
                sm.S[i * kMaxRank + jj] = acc;
            }
        }
        __syncthreads();
        if (tid == 0 && ready) {
            const int old = atomicAdd(&p.sync[tg * 4 + 1], 1);
            if (old == d.n_nc - 1) {   // last consumer of this tile resets its counters
                p.sync[tg * 4 + 0] = 0;
                p.sync[tg * 4 + 1] = 0;
            }
        }
        const bool landed = cta_wait(&sm.bar_expand, ph_expand, p);
        ph_expand ^= 1;
        if (!landed) return;
        if (!ready) {
            __syncthreads();
            continue;
        }

        const float sc = p.scale[d.a];
        const int kgs = d.rp / 8;
        for (int nl = tid; nl < nw; nl += kEngineThreads) {
            float acc[kBgmvRows];
#pragma unroll
            for (int i = 0; i < kBgmvRows; ++i) acc[i] = 0.f;
            const int tl = nl / kNTile, row = nl % kNTile;
            for (int kg = 0; kg < kgs; ++kg) {
                float bfv[8];
                bf16x8_to_f32(sm.B[(tl * kgs + kg) * kNTile + row], bfv);
#pragma unroll
                for (int i = 0; i < kBgmvRows; ++i) {
                    if (i < nrows) {
                        float a = acc[i];
#pragma unroll
                        for (int u = 0; u < 8; ++u) a = fmaf(sm.S[i * kMaxRank + kg * 8 + u], bfv[u], a);
                        acc[i] = a;
                    }
                }
            }
            const __nv_bfloat16 *ys = reinterpret_cast<const __nv_bfloat16 *>(sm.Y);
#pragma unroll
            for (int i = 0; i < kBgmvRows; ++i) {
                if (i < nrows) {
                    const float base = __bfloat162float(ys[i * d.nc + nl]);
                    const float v = fmaf(sc * sm.row_w[i], acc[i], base);
                    p.y[(int64_t)sm.row_dst[i] * p.ldy + n0 + nl] = __float2bfloat16_rn(v);
                }
            }
        }
        __syncthreads();
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
