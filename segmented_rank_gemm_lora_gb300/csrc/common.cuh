// Internal definitions shared by the library's translation units: workspace
// layout, kernel parameter blocks and small sm_103a PTX wrappers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/lora.h"

namespace lora {

// ---------------------------------------------------------------------------
// sizes
// ---------------------------------------------------------------------------
constexpr int kMaxRank = 64;           // largest true rank
constexpr int kMaxSlices = 4;
constexpr int kNTile = 128;            // B is stored in tiles of 128 output rows
constexpr int kBgmvRows = 16;          // rows of one small tile
// Keys the segment build sorts by, at most: adapters + 1 (the "none" key), or adapters x experts + 1.  The
// block-wide build keeps three counters per key in its shared memory, which holds a little over 17000.
constexpr int kMaxBuildKeys = 16000;
constexpr int kEngineThreads = 256;
constexpr int kHeaderInts = 16;
constexpr int kTraceSlots = 32;        // uint64 phase stamps per thread block (lora_set_trace)

// device error word bits (sticky, cleared by lora_get_status)
constexpr uint32_t kErrBadId = 1u << 0;
constexpr uint32_t kErrBadExpert = 1u << 1;
constexpr uint32_t kErrTimeout = 1u << 2;
constexpr uint32_t kErrWorkspace = 1u << 3;

// header slots
enum HeaderSlot {
    H_M = 0, H_NUM_SEGMENTS = 1, H_NUM_VALID = 2, H_NUM_MOE_GROUPS = 3, H_TOPK = 4, H_E = 5,
    H_BLOCK_M = 6, H_P_MAX = 7, H_B_MAX = 8, H_ERR = 12
};

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout, derived on the host from the lora_workspace fields.
struct WsLayout {
    size_t header, perm, segments, sorted_ids, expert_ids, ntpp, moe_groups;
    size_t sync, partials, total;
    int32_t seg_capacity, moe_group_capacity, P_max_cap, B_max_cap;
    int32_t max_tiles;
    int64_t partial_floats;
};
bool ws_layout(int32_t max_M, int32_t L, int32_t topk, int32_t E, int32_t block_m, WsLayout *out);

// ---------------------------------------------------------------------------
// engine parameters (one launch of the shrink/expand kernel)
// ---------------------------------------------------------------------------
struct EngineParams {
    // 2-D tensor map over the shrink input (bf16 [x_rows][K], row stride ldx; box 64 columns x
    // 128 rows, 128-byte swizzle): the tensor-core path loads runs of 128 consecutive rows through it
    CUtensorMap x_map;
    int32_t x_rows;          // rows the map spans; 0 = no map (every load takes the cp.async gather)
    const int32_t *m_ptr;    // token count of the last build (device)
    int32_t m_mult;          // rows of x per token (topk for the per-pair MoE input, else 1)
    // 2-D tensor maps over the output (bf16 [y_rows][N], row stride ldy; 128-byte swizzle): 128-column
    // units of 128-row tiles whose rows are one run of consecutive rows load through a 64 x 128 box and
    // store through 64 x 32 boxes
    CUtensorMap y_map_ld;
    CUtensorMap y_map_st;
    int32_t y_rows;          // rows the maps span; 0 = no maps (every unit takes per-row bulk copies)
    int32_t y_mult;          // rows of y per token
    // weight table
    const uint64_t *a_ptr;   // [L * E_A] packed A block addresses
    const uint64_t *b_ptr;   // [L * E_B] packed B block addresses
    const int32_t *rpad;     // [L] stored rank (multiple of 16)
    const float *scale;      // [L]
    int32_t L, E_A, E_B, K, n_slices, n_a;
    int32_t slice_n[kMaxSlices], slice_off[kMaxSlices], slice_tile_off[kMaxSlices];
    // work description written by lora_build_segments
    const int4 *groups;      // (adapter, expert, index into rows, count)
    const int32_t *num_groups;
    int32_t group_capacity;
    int32_t num_experts;     // experts a group may name (1 for dense)
    int64_t rows_capacity;   // entries of the row list
    const int32_t *rows;     // row list
    int32_t src_div;         // shrink input row = rows[i] / src_div
    // operands
    const __nv_bfloat16 *x;  int64_t ldx;
    __nv_bfloat16 *y;        int64_t ldy;
    const float *row_weight; // optional, indexed by rows[i]
    // scratch
    int32_t *sync;           // [max_tiles][4] counters
    float *partials;
    int64_t partial_floats;
    int32_t max_tiles;
    uint32_t *err;
    uint64_t timeout_ns;
    int32_t withhold;        // test hook: do not publish shrink results
    int32_t path;            // 0 auto, 1 every group on small tiles, 2 every group on 128-row tiles
    int32_t tc_min_rows;     // groups with more rows take 128-row tiles
    uint64_t *trace;         // optional [trace_ctas][32] phase stamps
    int32_t trace_ctas;
    // segment build fused into the launch (dense, at most 32 tokens): every CTA sorts ids itself and
    // CTA 0 also writes the segment table to the workspace; ids == nullptr reads the last build's table
    const int32_t *ids;
    int32_t ids_M;
    int32_t *ws_header, *ws_perm;
    int4 *ws_segments;
};

void launch_engine(const EngineParams &p, int grid, size_t smem, cudaStream_t s, bool pdl, cudaError_t *err);
size_t engine_smem_bytes(int group_capacity);
const void *engine_kernel_ptr();

// ---------------------------------------------------------------------------
// streaming path (csrc/stream.cu): shrink (with the plan) -> expand, two kernels chained on the stream
// ---------------------------------------------------------------------------
// One row tile of a group, as the plan lays it out.  The tile's shrink is cut into n_kc K-chunks of kc
// columns (the same cut for every tile of a group), each streamed in stages of ks columns; its expand is
// cut into n_units units of W output columns of one slice.
struct TileRec {
    int32_t a, e, row0, m;          // adapter, expert, first entry in the row list, rows
    int32_t rp, R, n_pad, kc;       // stored rank, A-block rows (n_a * rp), rows rounded up to 16, chunk K
    int32_t n_kc, ks, W, n_units;   // chunks, stage K, expand unit width, expand units
    int32_t p_off, s_off;           // fp32 partial offset (floats), S offset (bytes)
    int32_t c0, u0;                 // launch-wide index of the tile's first chunk / first unit
};
static_assert(sizeof(TileRec) == 64, "tile record");

// Plan header slots (int32)
enum PlanSlot {
    PL_TILES = 0,    // tiles
    PL_UNITS = 1,    // expand units of the launch
    PL_POOL_U = 2,   // first unit of the expand's claimed tail (units before it are split ahead of time)
    PL_CLAIM = 3,    // units of that tail claimed so far
};

struct StreamParams {
    // weight table
    const uint64_t *a_ptr, *b_ptr;   // [L * E_A], [L * E_B] packed block addresses
    const int32_t *rpad;             // [L] stored rank
    const float *scale;              // [L]
    int32_t L, E_A, E_B, K, n_slices, n_a;
    int32_t slice_n[kMaxSlices], slice_off[kMaxSlices], slice_tile_off[kMaxSlices];
    // groups written by lora_build_segments: (adapter, expert, index into rows, count)
    const int4 *groups;
    const int32_t *num_groups;
    int32_t group_capacity;
    const int32_t *rows;             // row list: y row of each entry; the x row is rows[i] / src_div
    int32_t src_div;
    // operands
    const __nv_bfloat16 *x;  int64_t ldx;
    __nv_bfloat16 *y;        int64_t ldy;
    const float *row_weight;         // optional, indexed by the y row
    // plan area (caller's workspace)
    int32_t *plan_hdr;               // [16]
    TileRec *tiles;                  // [max_tiles]
    int2 *ex_start;                  // [grid + 1] first (tile, unit) of every expand block
    int2 *rd_start;                  // [grid + 1] first (tile, S chunk) of every expand block's S sums
    int32_t *cnt;                    // shrink blocks whose share of the launch's tile records is out
    int32_t *done;                   // expand blocks that have ended (the last one resets the counters)
    int32_t *tile_cnt;               // [max_tiles] per tile: its K-chunks whose partials are out
    int32_t *s_done;                 // [max_tiles] per tile: its S chunks summed
    int32_t *ex_claim;               // plan_hdr + PL_CLAIM (reset by the shrink)
    float *partials;                 // fp32 chunk partials
    int64_t partial_cap;             // floats
    unsigned char *s_area;           // finished S, bf16, per tile [n_a][rp / 8][n_pad][8]
    int64_t s_cap;                   // bytes
    int32_t max_tiles;
    int32_t grid_s, grid_e;          // blocks of the shrink and of the expand launch
    int32_t tile_max;                // rows of a tile at most (128; smaller values force more tiles)
    uint32_t *err;
    uint64_t timeout_ns;
    int32_t withhold;                // test hook: the expand never loads S, so its waits run out
    uint64_t *trace;                 // optional phase stamps: [3][trace_ctas][32] (shrink, expand, plan)
    int32_t trace_ctas;
};

cudaError_t launch_stream(const StreamParams &p, cudaStream_t s, bool pdl);
// Bytes of the plan area (header, tiles, prefixes, block starts) for max_tiles tiles and grids up to
// kStreamMaxGrid blocks; the S area and the partials follow it.
constexpr int kStreamMaxGrid = 1024;
size_t stream_plan_bytes(int32_t max_tiles);
int stream_grid(int sms);

struct BuildParams {
    const int32_t *ids;
    const int32_t *topk_ids;      // nullable
    const uint8_t *enabled;       // nullable
    int32_t M, L, topk, E, block_m;
    int32_t *header, *perm;
    int4 *segments;
    int32_t *sorted_ids, *expert_ids, *ntpp;
    int4 *moe_groups;
    int32_t seg_capacity, moe_group_capacity;
    int32_t *sync;                // zeroed
    int32_t sync_ints;
};
cudaError_t launch_build(const BuildParams &p, cudaStream_t s, bool pdl);

cudaError_t launch_pack_a(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int32_t K, int32_t n_a, int32_t rank,
                          int32_t rpad, cudaStream_t s);
cudaError_t launch_pack_b(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int32_t rank, int32_t rpad,
                          int32_t n_slices, const int32_t *slice_n, cudaStream_t s);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier with a time limit.  Returns false
// (and sets the timeout bit) when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns, uint32_t *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Wait for phase `parity` of an mbarrier with a time limit, letting the hardware suspend the thread until
// the phase completes (up to 20 us per try) instead of polling, so a waiting thread takes no issue slots from
// the warps that work beside it.  Returns false (and sets the timeout bit) when the limit ran out.
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t *bar, uint32_t parity, uint64_t limit_ns, uint32_t *err)
{
    auto try_wait = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
            : "memory");
        return ok != 0;
    };
    if (try_wait()) return true;
    const uint64_t t0 = globaltimer();
    while (!try_wait()) {
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// Retire `bytes` of an mbarrier's expected transactions that will never arrive.
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Bulk (non-tensor) async copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk async copy shared -> global in this thread's bulk group (same alignment rules).
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int atom_add_release_gpu(int32_t *p, int v)
{
    int old;
    asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t *p, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start
// while the kernel before it on the stream still runs; it must wait here before it reads anything that
// kernel (or any earlier work) wrote.  Outside such a launch the wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel on the stream (if launched with programmatic serialization) start launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void nanosleep_ns(uint32_t ns)
{
    asm volatile("nanosleep.u32 %0;" ::"r"(ns));
}

// Dense batches of at most 32 tokens, one token per lane of one warp: each token's slot in the stable
// counting sort on key = adapter id, or L for tokens without one (-1, bad or disabled ids; lanes past M
// take L + 1).  The key bits are compared from the top, one ballot per bit: a lane counts the lanes that
// share its higher bits and have a 0 where it has a 1 (the smaller keys) and narrows its set of equal
// lanes; the slot is the smaller keys plus the equal keys on lower lanes.
struct WarpRank {
    int key;        // this lane's key
    int rank;       // its slot in the sorted order
    int count;      // lanes with the same key
    int seg;        // on the first lane of a key: keys smaller than it (the segment's index)
    bool first;     // the lowest lane of its key
    bool bad;       // the id is neither -1 nor in [0, L)
};
__device__ __forceinline__ WarpRank warp_rank_ids(const int32_t *ids, const uint8_t *enabled, int M, int L)
{
    const int lane = threadIdx.x & 31;
    const uint32_t below = (1u << lane) - 1u;
    WarpRank r;
    r.key = L + 1;
    r.bad = false;
    if (lane < M) {
        const int32_t i = ids[lane];
        r.bad = i < -1 || i >= L;
        r.key = (i >= 0 && i < L && (enabled == nullptr || enabled[i])) ? i : L;
    }
    uint32_t same = 0xffffffffu;
    int less = 0;
#pragma unroll 1
    for (int b = 31 - __clz(L + 1); b >= 0; --b) {
        const uint32_t ones = __ballot_sync(0xffffffffu, (r.key >> b) & 1);
        if ((r.key >> b) & 1) {
            less += __popc(same & ~ones);
            same &= ones;
        } else {
            same &= ~ones;
        }
    }
    r.rank = less + __popc(same & below);
    r.count = __popc(same);
    r.first = (same & below) == 0;
    // first lanes hold the smallest slot of their key: the keys below this one are the first lanes on lower
    // slots
    const uint32_t first_slots = __reduce_or_sync(0xffffffffu, r.first ? 1u << r.rank : 0u);
    r.seg = __popc(first_slots & ((1u << r.rank) - 1u));
    return r;
}

// 8 bf16 (one uint4) -> 8 floats
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float f[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
#endif

}  // namespace lora
