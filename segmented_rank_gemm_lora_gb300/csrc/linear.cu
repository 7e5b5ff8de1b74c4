// The LoRA linear layer in one kernel: y = x W^T + scale_i (x A_i^T) B_i^T.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 3.3: each linear layer
// that carries LoRA (qkv, o_proj, gate/up, down) becomes a custom layer that
// takes the whole input and runs the base matmul and the LoRA operator, which
// may be merged into one larger fused operator; section 2.3: tokens bucketed
// into segments by adapter; section 4.2: S accumulates in fp32.
//
// One CTA per (token tile, output tile): a token tile is up to 128 tokens of
// one segment (or of the tokens without an adapter), taken through the
// segment table's permutation; an output tile is up to 256 columns of one
// slice (two of the table's 128-column B tiles).
// The K loop streams, through a ring of stages,
//   x: the tile's rows gathered with 16-byte cp.async into the no-swizzle
//      K-major layout ([8][128][8] per 64-column stage);
//   W: one 2-D TMA box (64 K x 256 rows, 128-byte swizzle);
//   A: for a segment's tile, the adapter's packed A chunk ([8][R][8], one
//      bulk copy of a contiguous run);
// and one thread issues tcgen05 MMAs into two tensor-memory accumulators,
// D = x W^T (128 x 256) and S = x A^T (128 x R): x is read once for both.
// After the loop the epilogue warps read S, scale it, round it once to bf16
// and store it to shared memory as an MMA operand; one more pass of MMAs adds
// S_slice B^T to D (one MMA pass per B tile); D is rounded to bf16 and
// written to y once (the
// layer's output replaces y: no base output is read).
#include "linear.h"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kT = kLinearThreads;
constexpr int kXBytes = kLinearRows * kLinearK * 2;   // x stage: [8][128][8] bf16
constexpr int kWBytes = kLinearCols * kLinearK * 2;   // W stage: 256 rows x 128 B, swizzled
constexpr uint32_t kTmemCols = 512;                   // D: columns [0, 256); S: [256, 256 + R)
constexpr int kMaxStages = kLinearMaxStages;
static_assert(kLinearRows == 128 && kLinearCols == 2 * kLinearBCols && kLinearK == 64, "tile shape");
static_assert(kLinearBTileBytes == 2 * kMaxRank * kLinearBCols * 2, "two B tiles [rp/8][128][8] at the largest rank");

struct LinSmem {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t bbar, acc, sready, fin;
    uint64_t a_blk, b_blk;
    float sc;
    uint32_t tmem;
    int32_t adapter, slot0, rows, rp, xtma;
    int32_t rowsrc[kLinearRows];
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const LinearParams &p)
{
    return mbar_wait_bounded(bar, parity, p.timeout_ns, p.err);
}

__global__ void __launch_bounds__(kT, 1) linear_kernel(const __grid_constant__ LinearParams p)
{
    extern __shared__ unsigned char dsm_raw[];
    __shared__ LinSmem sm;
    // the stages start on a 1024-byte boundary (the swizzled W boxes need it)
    unsigned char *const dsm = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
    unsigned char *const bst = dsm + p.stages * p.stage_bytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = blockIdx.x;    // output tile (256 columns)
    const int rt = blockIdx.y;   // token tile
    pdl_wait();   // the segment table and x may come from the kernels before
    pdl_trigger();

    // ---- the token tile: tile rt of the segments (each cut into 128-row tiles), then of the tokens
    // without an adapter (the tail of the permutation) ----
    if (warp == 0) {
        const int nG = p.header[H_NUM_SEGMENTS], M = p.header[H_M], nv = p.header[H_NUM_VALID];
        int base = 0;
        bool found = false;
        for (int c = 0; c < nG && !found; c += 32) {
            const int g = c + lane;
            const int4 seg = g < nG ? p.segments[g] : make_int4(0, 0, 0, 0);
            const int tl = (seg.w + kLinearRows - 1) >> 7;
            int incl = tl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (rt < base + total) {
                const int first = base + incl - tl;
                if (rt >= first && rt < base + incl) {
                    sm.adapter = seg.x;
                    sm.slot0 = seg.z + (rt - first) * kLinearRows;
                    sm.rows = min(kLinearRows, seg.w - (rt - first) * kLinearRows);
                }
                found = true;
            }
            base += total;
        }
        if (!found && lane == 0) {
            const int t0 = rt - base, nn = M - nv;
            const bool in = t0 >= 0 && t0 * kLinearRows < nn;
            sm.adapter = -1;
            sm.slot0 = nv + t0 * kLinearRows;
            sm.rows = in ? min(kLinearRows, nn - t0 * kLinearRows) : 0;
        }
    }
    __syncthreads();
    const int rows = sm.rows;
    if (rows <= 0) return;
    if (tid < rows) sm.rowsrc[tid] = p.perm[sm.slot0 + tid];
    {
        // x moves as TMA boxes when the box's 128 rows are the tile's rows in order (or rows past a short
        // tile's end, whose products are not stored) and lie inside the last build's tokens
        const int r0 = p.perm[sm.slot0];
        const bool run = tid >= rows || p.perm[sm.slot0 + tid] == r0 + tid;
        const int all = __syncthreads_and(run);
        if (tid == 0) sm.xtma = all && r0 + kLinearRows <= p.header[H_M];
    }
    if (tid == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&sm.full[i], 1 + 128);   // the TMA issuer's expect_tx, then one arrival per x gatherer
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.bbar, 1);
        mbar_init(&sm.acc, 1);
        mbar_init(&sm.sready, 128);
        mbar_init(&sm.fin, 1);
        const int a = sm.adapter;
        const bool ok = a >= 0 && a < p.L;
        sm.rp = ok ? p.rpad[a] : 0;
        sm.a_blk = ok ? p.a_ptr[a] : 0;
        sm.b_blk = ok ? p.b_ptr[a] : 0;
        sm.sc = ok ? p.scale[a] : 0.f;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&sm.tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem;
    const int rp = sm.rp, R = p.n_a * rp;
    const bool lora = rp > 0, xtma = sm.xtma != 0;
    int s = 0;
    while (s + 1 < p.n_slices && j >= p.slice_ctile_off[s + 1]) ++s;
    const int lt = j - p.slice_ctile_off[s];
    const int col0 = p.slice_off[s] + lt * kLinearCols, width = min(kLinearCols, p.slice_n[s] - lt * kLinearCols);
    const int jb = p.slice_tile_off[s] + 2 * lt;              // the tile's first B tile
    const int nb = width > kLinearBCols ? 2 : 1;              // and its B tiles
    const int nK = (p.K + kLinearK - 1) / kLinearK;
    const int S = p.stages;

    if (warp < 4) {
        // ---- producers: thread t gathers x row t; thread 0 also requests W and A (and the B tile) ----
        const int t = tid;
        const __nv_bfloat16 *xrow = p.x + (int64_t)(t < rows ? sm.rowsrc[t] : sm.rowsrc[0]) * p.ldx;
        const unsigned char *ablk = reinterpret_cast<const unsigned char *>(sm.a_blk);
        if (t == 0 && lora) {
            const uint32_t bbytes = (uint32_t)(nb * rp * 256);
            mbar_arrive_expect_tx(&sm.bbar, bbytes);
            bulk_g2s(bst, reinterpret_cast<const unsigned char *>(sm.b_blk) + (int64_t)jb * rp * 256, bbytes, &sm.bbar);
        }
        for (int kb = 0; kb < nK; ++kb) {
            const int st = kb % S;
            unsigned char *sb = dsm + st * p.stage_bytes;
            if (kb >= S) wait_bar(&sm.empty[st], ((kb / S) - 1) & 1, p);
            const int k0 = kb * kLinearK, kk = min(kLinearK, p.K - k0);
            if (t == 0) {
                const uint32_t abytes = lora ? (uint32_t)((kk >> 3) * R * 16) : 0u;
                mbar_arrive_expect_tx(&sm.full[st], (uint32_t)kWBytes + abytes + (xtma ? (uint32_t)kXBytes : 0u));
                tc::tma_tile2d(sb + kXBytes, &p.w_map, k0, col0, &sm.full[st]);
                if (xtma) tc::tma_tile2d(sb, &p.x_map, k0, sm.rowsrc[0], &sm.full[st]);
                if (lora) bulk_g2s(sb + kXBytes + kWBytes, ablk + (int64_t)(k0 >> 3) * R * 16, abytes, &sm.full[st]);
            }
            if (!xtma) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    tc::cp_async16(sb + (c * kLinearRows + t) * 16, xrow + k0 + c * 8, t < rows && c * 8 < kk);
            }
            // a last K step of 8 columns: the A rows of its other 8 columns are zero
            if (lora && (kk & 8))
                for (int i = t; i < R; i += 128)
                    tc::cp_async16(sb + kXBytes + kWBytes + ((kk >> 3) * R + i) * 16, ablk, false);
            tc::cp_async_arrive_noinc(&sm.full[st]);
        }
        tc::cp_async_wait_all();
    } else if (warp == 4 && lane == 0) {
        // ---- MMA issuer: D += x W^T and S += x A^T, stage by stage ----
        const uint32_t id_d = tc::idesc_bf16(kLinearRows, kLinearCols);
        const uint32_t id_s = lora ? tc::idesc_bf16(kLinearRows, R) : 0u;
        for (int kb = 0; kb < nK; ++kb) {
            const int st = kb % S;
            wait_bar(&sm.full[st], (kb / S) & 1, p);
            // the producers' cp.async pieces (gathered x rows, a zeroed K tail), seen through the barrier, to the
            // tensor core; a stage of TMA and bulk copies alone needs no proxy fence
            if (!xtma || (lora && ((p.K - kb * kLinearK) & 8) && p.K - kb * kLinearK < kLinearK)) tc::fence_proxy_async_smem();
            tc::fence_after_sync();
            const uint32_t xs = smem_u32(dsm + st * p.stage_bytes), ws = xs + kXBytes, as = ws + kWBytes;
            const int nks = (min(kLinearK, p.K - kb * kLinearK) + 15) >> 4;
            for (int ks = 0; ks < nks; ++ks) {
                const uint64_t xd = xtma ? tc::smem_desc_sw128(xs + ks * 32)
                                         : tc::smem_desc(xs + ks * 2 * kLinearRows * 16, kLinearRows * 16, 128);
                const uint32_t accum = (kb | ks) != 0;
                tc::mma_bf16(tmem, xd, tc::smem_desc_sw128(ws + ks * 32), id_d, accum);
                if (lora) tc::mma_bf16(tmem + kLinearCols, xd, tc::smem_desc(as + ks * 2 * R * 16, R * 16, 128), id_s, accum);
            }
            tc::mma_commit(&sm.empty[st]);
        }
        tc::mma_commit(&sm.acc);
    }
    __syncwarp();

    if (warp >= 4) {
        // ---- epilogue: thread t owns token row t (tensor-memory lane t) ----
        const int t = tid - 128;
        const uint32_t lane_tm = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        wait_bar(&sm.acc, 0, p);
        tc::fence_after_sync();
        if (lora) {
            // S row t, scaled and rounded to bf16, into the stage area as the operand [R/8][128][8]
            const float sc = sm.sc;
            for (int c0 = 0; c0 < R; c0 += 16) {
                float v[16];
                tc::tmem_ld16(lane_tm + kLinearCols + c0, v);
                uint4 q[2];
                uint32_t *w = reinterpret_cast<uint32_t *>(q);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(sc * v[2 * i], sc * v[2 * i + 1]);
                    w[i] = *reinterpret_cast<const uint32_t *>(&h);
                }
                *reinterpret_cast<uint4 *>(dsm + ((c0 >> 3) * kLinearRows + t) * 16) = q[0];
                *reinterpret_cast<uint4 *>(dsm + (((c0 >> 3) + 1) * kLinearRows + t) * 16) = q[1];
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(&sm.sready);
            if (warp == 4 && lane == 0) {
                // D += S_slice B_tile^T (K = the stored rank)
                wait_bar(&sm.sready, 0, p);
                wait_bar(&sm.bbar, 0, p);
                tc::fence_after_sync();
                const int scol = p.n_a == 1 ? 0 : s * rp;
                const uint32_t ss = smem_u32(dsm) + (scol >> 3) * kLinearRows * 16, bs = smem_u32(bst);
                const uint32_t id_b = tc::idesc_bf16(kLinearRows, kLinearBCols);
                for (int b = 0; b < nb; ++b)
                    for (int ks = 0; ks < (rp >> 4); ++ks)
                        tc::mma_bf16(tmem + b * kLinearBCols, tc::smem_desc(ss + ks * 2 * kLinearRows * 16, kLinearRows * 16, 128),
                                     tc::smem_desc(bs + b * rp * 256 + ks * 2 * kLinearBCols * 16, kLinearBCols * 16, 128),
                                     id_b, 1u);
                tc::mma_commit(&sm.fin);
            }
            __syncwarp();
            wait_bar(&sm.fin, 0, p);
            tc::fence_after_sync();
        }
        // D row t -> bf16 -> y (256 columns of one slice, `width` of them inside it)
        __nv_bfloat16 *yrow = t < rows ? p.y + (int64_t)sm.rowsrc[t] * p.ldy + col0 : nullptr;
        for (int c0 = 0; c0 < kLinearCols; c0 += 32) {
            float v[32];
            tc::tmem_ld32(lane_tm + c0, v);
            if (yrow == nullptr) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + q * 8;
                if (c >= width) break;
                uint4 o;
                uint32_t *w = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(v[q * 8 + 2 * i], v[q * 8 + 2 * i + 1]);
                    w[i] = *reinterpret_cast<const uint32_t *>(&h);
                }
                *reinterpret_cast<uint4 *>(yrow + c) = o;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

const void *linear_kernel_ptr() { return reinterpret_cast<const void *>(&linear_kernel); }

cudaError_t launch_linear(const LinearParams &p, dim3 grid, size_t smem, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, linear_kernel, p);
}

}  // namespace lora
