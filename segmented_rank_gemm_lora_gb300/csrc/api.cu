// Host side of the C ABI declared in include/lora.h.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "linear.h"
#include "embedding.h"
#include "table_entry.h"

using namespace lora;

namespace {

constexpr int64_t kPartialFloatsPerRow = 16384;   // L2 scratch for rank-sized partials, per row of work
constexpr int64_t kMaxRows = 65536;               // tokens (or token/expert pairs) per build

std::atomic<int64_t> g_opt_path{0};
std::atomic<int64_t> g_opt_tc_min_rows{32};
std::atomic<int64_t> g_opt_timeout_ns{1000000000LL};
std::atomic<int64_t> g_opt_grid{0};
std::atomic<int64_t> g_opt_withhold{0};
std::atomic<int64_t> g_opt_pdl{1};
std::atomic<void *> g_trace{nullptr};
std::atomic<int64_t> g_trace_bytes{0};

struct DeviceInfo {
    int sms = 0;
    int engine_blocks_per_sm = 0;
    int max_dyn_smem = 0;               // opt-in shared memory per block
    bool attr_done = false;
};
std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

lora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_encode_mu;
encode_tiled_fn g_encode = nullptr;

// 2-D map over a bf16 [rows][K] matrix with row stride ld: box 64 columns x 128 rows, 128-byte swizzle,
// reads outside the matrix return zero.
static lora_status encode_2d(const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
                             CUtensorMap *out);

lora_status encode_rows_map(const void *base, int64_t rows, int32_t K, int64_t ld, CUtensorMap *out)
{
    // the kernel only issues boxes that lie inside the rows of x, so the row extent may be rounded up to one box
    return encode_2d(base, std::max<int64_t>(rows, 128), K, ld, 128, out);
}

// bf16 [rows][cols] with row stride ld elements; boxes of 64 columns x box_rows rows, 128-byte swizzle
static lora_status encode_2d(const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
                             CUtensorMap *out)
{
    {
        std::lock_guard<std::mutex> lk(g_encode_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                cudaGetLastError();
                return LORA_ERR_CUDA;
            }
            g_encode = reinterpret_cast<encode_tiled_fn>(fn);
        }
    }
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LORA_OK : LORA_ERR_UNSUPPORTED;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lora_status device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.attr_done) {
        const size_t smem = engine_smem_bytes(0);
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LORA_ERR_CUDA;
        if (cudaFuncSetAttribute(engine_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return LORA_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.engine_blocks_per_sm, engine_kernel_ptr(),
                                                          kEngineThreads, smem) != cudaSuccess)
            return LORA_ERR_CUDA;
        if (d.engine_blocks_per_sm < 1) return LORA_ERR_UNSUPPORTED;
        int optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, linear_kernel_ptr()) != cudaSuccess)
            return LORA_ERR_CUDA;
        d.max_dyn_smem = optin - (int)fa.sharedSizeBytes;   // what the fused linear kernel may take
        if (cudaFuncSetAttribute(linear_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_dyn_smem) !=
            cudaSuccess)
            return LORA_ERR_CUDA;
        d.attr_done = true;
    }
    *out = d;
    return LORA_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// table
// ---------------------------------------------------------------------------
struct lora_table_s {
    int32_t L = 0, K = 0, N = 0, n_slices = 0, n_a = 0, E_A = 1, E_B = 1;
    int32_t slice_n[kMaxSlices] = {0}, slice_off[kMaxSlices] = {0}, slice_tile_off[kMaxSlices] = {0};
    int32_t b_tiles = 0;                // n-tiles per B block
    std::vector<int32_t> rank, rpad;
    std::vector<float> scale;
    std::vector<uint64_t> a_ptr, b_ptr; // host copies of the device pointer tables
    std::vector<void *> group_mem;      // one allocation per stored rank
    int64_t device_bytes = 0;
    uint64_t *d_a_ptr = nullptr, *d_b_ptr = nullptr;
    int32_t *d_rpad = nullptr;
    float *d_scale = nullptr;
    int32_t max_R = 0;
    // the pool of adapter blocks per stored rank ("vLLM-Ascend dynamic LoRA fused operator", section 3.1):
    // an adapter's A blocks (E_A of them, contiguous) and B blocks (E_B), taken whole and returned whole
    struct Slot {
        char *a, *b;
    };
    std::map<int32_t, std::vector<Slot>> free_slots;               // stored rank -> free blocks
    struct Retiring {
        cudaEvent_t done;                                          // recorded after the entries were replaced
        int32_t rp;
        Slot slot;
    };
    std::vector<Retiring> retiring;                                // replaced blocks still readable by queued work
    uint32_t magic = 0x4c6f5241u;
};

static bool valid_table(lora_table t) { return t != nullptr && t->magic == 0x4c6f5241u; }

extern "C" int32_t lora_rank_padded(int32_t rank)
{
    if (rank < 1 || rank > kMaxRank) return -1;
    return (int32_t)round_up(rank, 16);
}

static void free_table(lora_table t)
{
    for (auto &r : t->retiring) cudaEventDestroy(r.done);
    for (void *m : t->group_mem) cudaFree(m);
    cudaFree(t->d_a_ptr);
    cudaFree(t->d_b_ptr);
    cudaFree(t->d_rpad);
    cudaFree(t->d_scale);
    t->magic = 0;
    delete t;
}

extern "C" lora_status lora_pack_weights(const lora_adapter_desc *adapters, int32_t L, const lora_proj_shape *shape,
                                         lora_stream_t stream, lora_table *out)
{
    if (!adapters || !shape || !out || L < 1) return LORA_ERR_INVALID_ARG;
    *out = nullptr;
    const lora_proj_shape &sh = *shape;
    if (sh.K < 8 || sh.K % 8 != 0 || sh.K > (1 << 20)) return LORA_ERR_INVALID_ARG;
    if (sh.n_slices < 1 || sh.n_slices > kMaxSlices) return LORA_ERR_INVALID_ARG;
    if (!(sh.n_a == 1 || sh.n_a == sh.n_slices)) return LORA_ERR_INVALID_ARG;
    if (sh.E_A < 1 || sh.E_B < 1) return LORA_ERR_INVALID_ARG;
    int64_t N = 0;
    for (int s = 0; s < sh.n_slices; ++s) {
        if (sh.slice_n[s] < 8 || sh.slice_n[s] % 8 != 0) return LORA_ERR_INVALID_ARG;
        N += sh.slice_n[s];
    }
    if (N > (1 << 30)) return LORA_ERR_UNSUPPORTED;
    for (int i = 0; i < L; ++i) {
        if (lora_rank_padded(adapters[i].rank) < 0) return LORA_ERR_INVALID_ARG;
        if (!adapters[i].A || !adapters[i].B) return LORA_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    lora_table t = new (std::nothrow) lora_table_s();
    if (!t) return LORA_ERR_OOM;
    t->L = L;
    t->K = sh.K;
    t->N = (int32_t)N;
    t->n_slices = sh.n_slices;
    t->n_a = sh.n_a;
    t->E_A = sh.E_A;
    t->E_B = sh.E_B;
    int32_t col = 0, tiles = 0;
    for (int i = 0; i < sh.n_slices; ++i) {
        t->slice_n[i] = sh.slice_n[i];
        t->slice_off[i] = col;
        t->slice_tile_off[i] = tiles;
        col += sh.slice_n[i];
        tiles += (int32_t)ceil_div(sh.slice_n[i], kNTile);
    }
    t->b_tiles = tiles;
    t->rank.resize(L);
    t->rpad.resize(L);
    t->scale.resize(L);
    t->a_ptr.assign((size_t)L * sh.E_A, 0);
    t->b_ptr.assign((size_t)L * sh.E_B, 0);
    for (int i = 0; i < L; ++i) {
        t->rank[i] = adapters[i].rank;
        t->rpad[i] = lora_rank_padded(adapters[i].rank);
        t->scale[i] = adapters[i].scale;
        t->max_R = std::max(t->max_R, sh.n_a * t->rpad[i]);
    }

    // one contiguous allocation per stored rank: all A blocks of that rank, then all B blocks
    std::vector<int32_t> ranks_present(t->rpad);
    std::sort(ranks_present.begin(), ranks_present.end());
    ranks_present.erase(std::unique(ranks_present.begin(), ranks_present.end()), ranks_present.end());
    lora_status st = LORA_OK;
    for (int32_t rp : ranks_present) {
        const int64_t a_block = round_up((int64_t)sh.K * sh.n_a * rp * 2, 256);
        const int64_t b_block = round_up((int64_t)tiles * kNTile * rp * 2, 256);
        std::vector<int> members;
        for (int i = 0; i < L; ++i)
            if (t->rpad[i] == rp) members.push_back(i);
        const int64_t bytes = (int64_t)members.size() * (sh.E_A * a_block + sh.E_B * b_block);
        void *mem = nullptr;
        if (cudaMalloc(&mem, (size_t)bytes) != cudaSuccess) {
            cudaGetLastError();
            st = LORA_ERR_OOM;
            break;
        }
        t->group_mem.push_back(mem);
        t->device_bytes += bytes;
        char *base = static_cast<char *>(mem);
        int64_t off = 0;
        for (int i : members) {
            for (int e = 0; e < sh.E_A; ++e) {
                t->a_ptr[(size_t)i * sh.E_A + e] = reinterpret_cast<uint64_t>(base + off);
                off += a_block;
            }
        }
        for (int i : members) {
            for (int e = 0; e < sh.E_B; ++e) {
                t->b_ptr[(size_t)i * sh.E_B + e] = reinterpret_cast<uint64_t>(base + off);
                off += b_block;
            }
        }
    }
    if (st == LORA_OK) {
        for (int i = 0; i < L && st == LORA_OK; ++i) {
            const int32_t r = t->rank[i], rp = t->rpad[i];
            const auto *A = static_cast<const __nv_bfloat16 *>(adapters[i].A);
            const auto *B = static_cast<const __nv_bfloat16 *>(adapters[i].B);
            for (int e = 0; e < sh.E_A && st == LORA_OK; ++e)
                st = cuda_status(launch_pack_a(A + (int64_t)e * sh.n_a * r * sh.K,
                                               reinterpret_cast<__nv_bfloat16 *>(t->a_ptr[(size_t)i * sh.E_A + e]),
                                               sh.K, sh.n_a, r, rp, s));
            for (int e = 0; e < sh.E_B && st == LORA_OK; ++e)
                st = cuda_status(launch_pack_b(B + (int64_t)e * N * r,
                                               reinterpret_cast<__nv_bfloat16 *>(t->b_ptr[(size_t)i * sh.E_B + e]),
                                               r, rp, sh.n_slices, sh.slice_n, s));
        }
    }
    if (st == LORA_OK) {
        const size_t na = t->a_ptr.size() * 8, nb = t->b_ptr.size() * 8;
        if (cudaMalloc(&t->d_a_ptr, na) != cudaSuccess || cudaMalloc(&t->d_b_ptr, nb) != cudaSuccess ||
            cudaMalloc(&t->d_rpad, (size_t)L * 4) != cudaSuccess || cudaMalloc(&t->d_scale, (size_t)L * 4) != cudaSuccess) {
            cudaGetLastError();
            st = LORA_ERR_OOM;
        }
    }
    if (st == LORA_OK) {
        // the host vectors live as long as the table, so async copies from them are safe
        if (cudaMemcpyAsync(t->d_a_ptr, t->a_ptr.data(), t->a_ptr.size() * 8, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(t->d_b_ptr, t->b_ptr.data(), t->b_ptr.size() * 8, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(t->d_rpad, t->rpad.data(), (size_t)L * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(t->d_scale, t->scale.data(), (size_t)L * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
            st = LORA_ERR_CUDA;
    }
    if (st != LORA_OK) {
        cudaStreamSynchronize(s);
        free_table(t);
        return st;
    }
    *out = t;
    return LORA_OK;
}

// Bytes of one adapter's A region (E_A blocks) and B region (E_B blocks) at stored rank rp, as the pack lays them.
static int64_t slot_a_bytes(lora_table t, int32_t rp) { return t->E_A * round_up((int64_t)t->K * t->n_a * rp * 2, 256); }
static int64_t slot_b_bytes(lora_table t, int32_t rp)
{
    return t->E_B * round_up((int64_t)t->b_tiles * kNTile * rp * 2, 256);
}

constexpr int kPoolChunkSlots = 4;   // blocks a new pool chunk of one stored rank holds

extern "C" lora_status lora_table_set_adapter(lora_table t, int32_t index, const lora_adapter_desc *adapter,
                                              lora_stream_t stream)
{
    if (!valid_table(t) || !adapter || index < 0 || index >= t->L) return LORA_ERR_INVALID_ARG;
    const int32_t rp = lora_rank_padded(adapter->rank);
    if (rp < 0 || !adapter->A || !adapter->B) return LORA_ERR_INVALID_ARG;
    if (t->E_A > kMaxEntryBlocks || t->E_B > kMaxEntryBlocks) return LORA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // blocks whose replacement every earlier launch has passed go back to the pool
    for (size_t i = 0; i < t->retiring.size();) {
        const cudaError_t q = cudaEventQuery(t->retiring[i].done);
        if (q == cudaSuccess) {
            t->free_slots[t->retiring[i].rp].push_back(t->retiring[i].slot);
            cudaEventDestroy(t->retiring[i].done);
            t->retiring.erase(t->retiring.begin() + (long)i);
        } else {
            if (q != cudaErrorNotReady) return LORA_ERR_CUDA;
            ++i;
        }
    }
    std::vector<lora_table_s::Slot> &pool = t->free_slots[rp];
    const int64_t abytes = slot_a_bytes(t, rp), bbytes = slot_b_bytes(t, rp);
    if (pool.empty()) {
        // a new chunk of blocks of this stored rank (the pool grows by whole chunks, never per adapter)
        void *mem = nullptr;
        if (cudaMalloc(&mem, (size_t)(kPoolChunkSlots * (abytes + bbytes))) != cudaSuccess) {
            cudaGetLastError();
            return LORA_ERR_OOM;
        }
        t->group_mem.push_back(mem);
        t->device_bytes += kPoolChunkSlots * (abytes + bbytes);
        char *base = static_cast<char *>(mem);
        for (int i = kPoolChunkSlots - 1; i >= 0; --i)
            pool.push_back({base + i * (abytes + bbytes), base + i * (abytes + bbytes) + abytes});
    }
    const lora_table_s::Slot slot = pool.back();
    // the new weights into the free block (the adapter's current block stays intact for queued launches)
    const int32_t r = adapter->rank;
    const auto *A = static_cast<const __nv_bfloat16 *>(adapter->A);
    const auto *B = static_cast<const __nv_bfloat16 *>(adapter->B);
    const int64_t a_block = abytes / t->E_A, b_block = bbytes / t->E_B;
    lora_status st = LORA_OK;
    for (int e = 0; e < t->E_A && st == LORA_OK; ++e)
        st = cuda_status(launch_pack_a(A + (int64_t)e * t->n_a * r * t->K,
                                       reinterpret_cast<__nv_bfloat16 *>(slot.a + e * a_block), t->K, t->n_a, r, rp, s));
    for (int e = 0; e < t->E_B && st == LORA_OK; ++e)
        st = cuda_status(launch_pack_b(B + (int64_t)e * t->N * r, reinterpret_cast<__nv_bfloat16 *>(slot.b + e * b_block),
                                       r, rp, t->n_slices, t->slice_n, s));
    if (st != LORA_OK) return st;
    pool.pop_back();
    // then the lookup entries, in stream order
    TableEntry e{};
    e.index = index;
    e.E_A = t->E_A;
    e.E_B = t->E_B;
    e.rpad = rp;
    e.scale = adapter->scale;
    for (int i = 0; i < t->E_A; ++i) e.a[i] = reinterpret_cast<uint64_t>(slot.a + i * a_block);
    for (int i = 0; i < t->E_B; ++i) e.b[i] = reinterpret_cast<uint64_t>(slot.b + i * b_block);
    st = cuda_status(launch_set_entry(e, t->d_a_ptr, t->d_b_ptr, t->d_rpad, t->d_scale, s));
    if (st != LORA_OK) return st;
    // the replaced block retires once the stream has passed the new entries
    lora_table_s::Retiring ret{};
    ret.rp = t->rpad[index];
    ret.slot = {reinterpret_cast<char *>(t->a_ptr[(size_t)index * t->E_A]),
                reinterpret_cast<char *>(t->b_ptr[(size_t)index * t->E_B])};
    if (cudaEventCreateWithFlags(&ret.done, cudaEventDisableTiming) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaEventRecord(ret.done, s) != cudaSuccess) {
        cudaEventDestroy(ret.done);
        return LORA_ERR_CUDA;
    }
    t->retiring.push_back(ret);
    // host copies of the entries
    t->rank[index] = r;
    t->rpad[index] = rp;
    t->scale[index] = adapter->scale;
    for (int i = 0; i < t->E_A; ++i) t->a_ptr[(size_t)index * t->E_A + i] = e.a[i];
    for (int i = 0; i < t->E_B; ++i) t->b_ptr[(size_t)index * t->E_B + i] = e.b[i];
    t->max_R = std::max(t->max_R, t->n_a * rp);
    return LORA_OK;
}

extern "C" lora_status lora_table_destroy(lora_table table)
{
    if (!valid_table(table)) return LORA_ERR_INVALID_ARG;
    free_table(table);
    return LORA_OK;
}

extern "C" lora_status lora_table_info(lora_table t, lora_table_info_t *info)
{
    if (!valid_table(t) || !info) return LORA_ERR_INVALID_ARG;
    info->L = t->L;
    info->K = t->K;
    info->N = t->N;
    info->n_slices = t->n_slices;
    info->n_a = t->n_a;
    info->E_A = t->E_A;
    info->E_B = t->E_B;
    std::vector<int32_t> stored(t->rpad);
    std::sort(stored.begin(), stored.end());
    info->num_rank_groups = (int32_t)(std::unique(stored.begin(), stored.end()) - stored.begin());
    info->device_bytes = t->device_bytes;
    int32_t best = 0, best_rank = -1;
    for (int i = 0; i < t->L; ++i)
        if (t->rank[i] > best_rank) best_rank = t->rank[i], best = t->rpad[i];
    info->stored_rank_of_max = best;
    return LORA_OK;
}

extern "C" int32_t lora_table_stored_rank(lora_table t, int32_t adapter)
{
    if (!valid_table(t) || adapter < 0 || adapter >= t->L) return -1;
    return t->rpad[adapter];
}

// ---------------------------------------------------------------------------
// workspace
// ---------------------------------------------------------------------------
bool lora::ws_layout(int32_t max_M, int32_t L, int32_t topk, int32_t E, int32_t block_m, WsLayout *o)
{
    if (max_M < 1 || L < 1 || block_m < 0) return false;
    if (block_m > 0 && (topk < 1 || E < 1)) return false;
    if (L + 1 > kMaxBuildKeys) return false;
    if (block_m > 0 && (int64_t)L * E + 1 > kMaxBuildKeys) return false;
    WsLayout w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (size_t)round_up((int64_t)(off + bytes), 256);
        return at;
    };
    w.header = take(kHeaderInts * 4);
    w.perm = take((size_t)max_M * 4);
    w.seg_capacity = std::max(1, std::min(L, max_M));
    w.segments = take((size_t)w.seg_capacity * 16);
    int64_t max_rows = max_M;
    w.moe_group_capacity = 0;
    if (block_m > 0) {
        const int64_t P = (int64_t)max_M * topk;
        const int64_t P_max = round_up(P + (int64_t)E * (block_m - 1), block_m);
        if (P_max > (1LL << 30)) return false;
        w.P_max_cap = (int32_t)P_max;
        w.B_max_cap = (int32_t)(P_max / block_m);
        w.sorted_ids = take((size_t)L * P_max * 4);
        w.expert_ids = take((size_t)L * w.B_max_cap * 4);
        w.ntpp = take((size_t)L * 4);
        w.moe_group_capacity = (int32_t)std::max<int64_t>(1, std::min<int64_t>((int64_t)L * E, P));
        w.moe_groups = take((size_t)w.moe_group_capacity * 16);
        max_rows = std::max<int64_t>(max_rows, P);
    } else {
        w.sorted_ids = w.expert_ids = w.ntpp = w.moe_groups = off;
    }
    if (max_rows > kMaxRows) return false;   // keeps every scratch offset inside int32
    const int64_t groups = std::max<int64_t>(w.seg_capacity, w.moe_group_capacity);
    w.max_tiles = (int32_t)(ceil_div(max_rows, kBgmvRows) + groups);
    w.sync = take((size_t)w.max_tiles * 16);
    w.partial_floats = max_rows * kPartialFloatsPerRow;
    w.partials = take((size_t)w.partial_floats * 4);
    w.total = off;
    *o = w;
    return true;
}

extern "C" size_t lora_workspace_bytes(int32_t max_M, int32_t L, int32_t topk, int32_t num_experts, int32_t block_m)
{
    WsLayout w;
    if (!ws_layout(max_M, L, topk, num_experts, block_m, &w)) return 0;
    return w.total;
}

static lora_status check_ws(const lora_workspace *ws, WsLayout *w)
{
    if (!ws || !ws->d_ptr || (reinterpret_cast<uintptr_t>(ws->d_ptr) & 255u) != 0) return LORA_ERR_INVALID_ARG;
    if (!ws_layout(ws->max_M, ws->L, ws->topk, ws->num_experts, ws->block_m, w)) return LORA_ERR_INVALID_ARG;
    if (ws->bytes < w->total) return LORA_ERR_WORKSPACE;
    return LORA_OK;
}

extern "C" lora_status lora_workspace_layout(const lora_workspace *ws, lora_workspace_layout_t *out)
{
    WsLayout w;
    if (!out) return LORA_ERR_INVALID_ARG;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    out->header = w.header;
    out->perm = w.perm;
    out->segments = w.segments;
    out->sorted_ids = w.sorted_ids;
    out->expert_ids = w.expert_ids;
    out->ntpp = w.ntpp;
    out->moe_groups = w.moe_groups;
    out->scratch = w.sync;
    out->seg_capacity = w.seg_capacity;
    out->moe_group_capacity = w.moe_group_capacity;
    return LORA_OK;
}

template <class T>
static T *at(const lora_workspace *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<char *>(ws->d_ptr) + off);
}

extern "C" lora_status lora_build_segments(const lora_workspace *ws, const int32_t *d_ids, int32_t M,
                                           const int32_t *d_topk_ids, const uint8_t *d_enabled, lora_stream_t stream)
{
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (M < 0 || (M > 0 && !d_ids)) return LORA_ERR_INVALID_ARG;
    if (M > ws->max_M) return LORA_ERR_WORKSPACE;
    if (d_topk_ids && ws->block_m <= 0) return LORA_ERR_INVALID_ARG;
    BuildParams p{};
    p.ids = d_ids;
    p.topk_ids = d_topk_ids;
    p.enabled = d_enabled;
    p.M = M;
    p.L = ws->L;
    p.topk = ws->topk;
    p.E = ws->num_experts;
    p.block_m = d_topk_ids ? ws->block_m : 0;
    p.header = at<int32_t>(ws, w.header);
    p.perm = at<int32_t>(ws, w.perm);
    p.segments = at<int4>(ws, w.segments);
    p.sorted_ids = at<int32_t>(ws, w.sorted_ids);
    p.expert_ids = at<int32_t>(ws, w.expert_ids);
    p.ntpp = at<int32_t>(ws, w.ntpp);
    p.moe_groups = at<int4>(ws, w.moe_groups);
    p.seg_capacity = w.seg_capacity;
    p.moe_group_capacity = w.moe_group_capacity;
    p.sync = at<int32_t>(ws, w.sync);
    p.sync_ints = w.max_tiles * 4;
    return cuda_status(launch_build(p, reinterpret_cast<cudaStream_t>(stream), g_opt_pdl.load() != 0));
}

// The streaming path (plan -> shrink -> expand) over the groups of the last build on `ws`.  Its plan, tile
// records, S and fp32 partials live in the workspace's scratch area, its tile counters in the sync area.
// The persistent engine's small-tile K-chunk when a block's share of the launch's A bytes is a staging
// slot or more: the largest chunk of a 16-row tile (A chunk <= 40 KB, x rows <= 15 KB), in multiples of
// 64 columns.  With smaller shares its chunks shrink, down to kEngineMinKc columns.
constexpr int64_t kEngineMinKc = 64;
static int64_t engine_small_kc(int64_t R)
{
    return std::max<int64_t>(kEngineMinKc, std::min<int64_t>(448, (20480 / R) / 64 * 64));
}
// Fp32 scratch the engine needs per row of small-tile work at A-block rows R, depth K and K-chunk kc: the
// chunks' partials and the row's finished S.
static int64_t engine_partials_per_row(int64_t R, int64_t K, int64_t kc) { return R * (ceil_div(K, kc) + 1); }

static lora_status run_stream(lora_table t, const lora_workspace *ws, const WsLayout &w, bool moe, int32_t src_div,
                              const void *x, int64_t ldx, void *y, int64_t ldy, const float *row_weight,
                              int32_t tile_max, lora_stream_t stream)
{
    DeviceInfo di;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    StreamParams p{};
    p.a_ptr = t->d_a_ptr;
    p.b_ptr = t->d_b_ptr;
    p.rpad = t->d_rpad;
    p.scale = t->d_scale;
    p.L = t->L;
    p.E_A = t->E_A;
    p.E_B = t->E_B;
    p.K = t->K;
    p.n_slices = t->n_slices;
    p.n_a = t->n_a;
    for (int s = 0; s < kMaxSlices; ++s) {
        p.slice_n[s] = t->slice_n[s];
        p.slice_off[s] = t->slice_off[s];
        p.slice_tile_off[s] = t->slice_tile_off[s];
    }
    int32_t *header = at<int32_t>(ws, w.header);
    if (moe) {
        p.groups = at<int4>(ws, w.moe_groups);
        p.num_groups = header + H_NUM_MOE_GROUPS;
        p.group_capacity = w.moe_group_capacity;
        p.rows = at<int32_t>(ws, w.sorted_ids);
    } else {
        p.groups = at<int4>(ws, w.segments);
        p.num_groups = header + H_NUM_SEGMENTS;
        p.group_capacity = w.seg_capacity;
        p.rows = at<int32_t>(ws, w.perm);
    }
    p.src_div = src_div;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.ldx = ldx;
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.ldy = ldy;
    p.row_weight = row_weight;
    // the scratch area: plan (header, tiles, prefixes, block starts), S, then the fp32 partials
    const int64_t max_rows = w.partial_floats / kPartialFloatsPerRow;
    const size_t plan_bytes = stream_plan_bytes(w.max_tiles);
    const size_t s_cap = (size_t)round_up(512 * (max_rows + 16 * (int64_t)w.max_tiles), 256);
    if (plan_bytes + s_cap >= (size_t)w.partial_floats * 4) return LORA_ERR_WORKSPACE;
    unsigned char *area = at<unsigned char>(ws, w.partials);
    p.plan_hdr = reinterpret_cast<int32_t *>(area);
    p.tiles = reinterpret_cast<TileRec *>(area + 256);
    p.ex_start = reinterpret_cast<int2 *>(area + 256 + (size_t)w.max_tiles * sizeof(TileRec));
    p.rd_start = p.ex_start + (kStreamMaxGrid + 1);
    p.s_area = area + plan_bytes;
    p.s_cap = (int64_t)s_cap;
    p.partials = reinterpret_cast<float *>(area + plan_bytes + s_cap);
    p.partial_cap = ((int64_t)w.partial_floats * 4 - (int64_t)plan_bytes - (int64_t)s_cap) / 4;
    p.max_tiles = w.max_tiles;
    // counters in the sync area (4 max_tiles ints), which the build zeroes and every launch leaves zeroed (as
    // the persistent engine expects it): the shrink's arrival count, the expand's exit count, then two counts
    // per tile (K-chunks done, S chunks summed)
    if (4 + 2 * (int64_t)w.max_tiles > 4 * (int64_t)w.max_tiles) return LORA_ERR_WORKSPACE;
    int32_t *sync = at<int32_t>(ws, w.sync);
    p.cnt = sync;
    p.done = sync + 1;
    p.tile_cnt = sync + 4;
    p.s_done = p.tile_cnt + w.max_tiles;
    p.ex_claim = p.plan_hdr + PL_CLAIM;
    const int grid = stream_grid(di.sms);
    const int64_t want = g_opt_grid.load();
    p.grid_s = p.grid_e = (want > 0 && want < grid) ? (int)want : grid;
    p.tile_max = tile_max;
    p.err = reinterpret_cast<uint32_t *>(header + H_ERR);
    p.timeout_ns = (uint64_t)g_opt_timeout_ns.load();
    p.withhold = g_opt_withhold.load() != 0;
    p.trace = static_cast<uint64_t *>(g_trace.load());
    p.trace_ctas = p.trace ? (int32_t)(g_trace_bytes.load() / (3 * 8 * kTraceSlots)) : 0;
    return cuda_status(launch_stream(p, reinterpret_cast<cudaStream_t>(stream), g_opt_pdl.load() != 0));
}

static lora_status run_engine(lora_table t, const lora_workspace *ws, const WsLayout &w, bool moe, int32_t src_div,
                              const void *x, int64_t ldx, int64_t x_rows, void *y, int64_t ldy,
                              const float *row_weight, lora_stream_t stream, const int32_t *fused_ids = nullptr,
                              int32_t fused_M = 0)
{
    // the streaming path serves every batch but the dense ones of at most 32 tokens, where one launch of
    // the persistent engine (small tiles, the segment build fused in) is faster
    {
        const int64_t path = g_opt_path.load();
        if (!fused_ids && (path == 3 || (path == 0 && (moe || ws->max_M > 32))))
            return run_stream(t, ws, w, moe, src_div, x, ldx, y, ldy, row_weight, path == 3 ? 16 : 128, stream);
    }
    // scratch per row of work at the K-chunk the engine's small tiles take whenever a block's share of A is
    // a staging slot or more; with smaller shares the engine may cut shorter chunks, finds the scratch
    // short and reports LORA_ERR_WORKSPACE through the status word
    if (engine_partials_per_row(t->max_R, t->K, engine_small_kc(t->max_R)) > kPartialFloatsPerRow)
        return LORA_ERR_UNSUPPORTED;
    DeviceInfo di;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    EngineParams p{};
    if (t->K >= 64) {   // narrower inputs always take the cp.async gather
        st = encode_rows_map(x, x_rows, t->K, ldx, &p.x_map);
        if (st != LORA_OK) return st;
        p.x_rows = (int32_t)x_rows;
    }
    p.m_ptr = at<int32_t>(ws, w.header) + H_M;
    p.m_mult = (moe && src_div == 1) ? ws->topk : 1;
    p.y_mult = moe ? ws->topk : 1;
    if (t->N >= 128) {   // output tiles move as 2-D boxes only inside rows the last build produced
        const int64_t y_rows = (int64_t)ws->max_M * p.y_mult;
        st = encode_2d(y, std::max<int64_t>(y_rows, 128), t->N, ldy, 128, &p.y_map_ld);
        if (st == LORA_OK) st = encode_2d(y, std::max<int64_t>(y_rows, 128), t->N, ldy, 32, &p.y_map_st);
        if (st != LORA_OK) return st;
        p.y_rows = (int32_t)y_rows;
    }
    p.a_ptr = t->d_a_ptr;
    p.b_ptr = t->d_b_ptr;
    p.rpad = t->d_rpad;
    p.scale = t->d_scale;
    p.L = t->L;
    p.E_A = t->E_A;
    p.E_B = t->E_B;
    p.K = t->K;
    p.n_slices = t->n_slices;
    p.n_a = t->n_a;
    for (int s = 0; s < kMaxSlices; ++s) {
        p.slice_n[s] = t->slice_n[s];
        p.slice_off[s] = t->slice_off[s];
        p.slice_tile_off[s] = t->slice_tile_off[s];
    }
    int32_t *header = at<int32_t>(ws, w.header);
    if (moe) {
        p.groups = at<int4>(ws, w.moe_groups);
        p.num_groups = header + H_NUM_MOE_GROUPS;
        p.group_capacity = w.moe_group_capacity;
        p.num_experts = ws->num_experts;
        p.rows_capacity = (int64_t)ws->L * w.P_max_cap;
        p.rows = at<int32_t>(ws, w.sorted_ids);
    } else {
        p.groups = at<int4>(ws, w.segments);
        p.num_groups = header + H_NUM_SEGMENTS;
        p.group_capacity = w.seg_capacity;
        p.num_experts = 1;
        p.rows_capacity = ws->max_M;
        p.rows = at<int32_t>(ws, w.perm);
    }
    p.src_div = src_div;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.ldx = ldx;
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.ldy = ldy;
    p.row_weight = row_weight;
    p.sync = at<int32_t>(ws, w.sync);
    p.partials = at<float>(ws, w.partials);
    p.partial_floats = w.partial_floats;
    p.max_tiles = w.max_tiles;
    p.err = reinterpret_cast<uint32_t *>(header + H_ERR);
    p.timeout_ns = (uint64_t)g_opt_timeout_ns.load();
    p.withhold = g_opt_withhold.load() != 0;
    p.path = (int32_t)g_opt_path.load();
    p.tc_min_rows = (int32_t)g_opt_tc_min_rows.load();
    p.trace = static_cast<uint64_t *>(g_trace.load());
    p.trace_ctas = p.trace ? (int32_t)(g_trace_bytes.load() / (8 * kTraceSlots)) : 0;
    if (fused_ids) {
        p.ids = fused_ids;
        p.ids_M = fused_M;
        p.ws_header = header;
        p.ws_perm = at<int32_t>(ws, w.perm);
        p.ws_segments = at<int4>(ws, w.segments);
    }
    int grid = di.sms * di.engine_blocks_per_sm;
    const int64_t want = g_opt_grid.load();
    if (want > 0 && want < grid) grid = (int)want;
    cudaError_t e;
    // Early scheduling only behind the one-warp build (dense workspaces of at most 32 tokens): an engine
    // block fits beside it, while the block-wide build holds its SM's shared memory, so behind it one
    // engine block would start late and hold up the whole grid.
    const bool pdl = g_opt_pdl.load() != 0 && !moe && ws->max_M <= 32;
    launch_engine(p, grid, engine_smem_bytes(0), reinterpret_cast<cudaStream_t>(stream), pdl, &e);
    return cuda_status(e);
}

extern "C" lora_status lora_apply(lora_table t, const lora_workspace *ws, const void *d_x, int64_t ldx, void *d_y,
                                  int64_t ldy, lora_stream_t stream)
{
    if (!valid_table(t) || !d_x || !d_y) return LORA_ERR_INVALID_ARG;
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (ws->L != t->L) return LORA_ERR_INVALID_ARG;
    if (t->E_A != 1 || t->E_B != 1) return LORA_ERR_INVALID_ARG;
    if (ldx < t->K || ldy < t->N || ldx % 8 || ldy % 8 || !aligned16(d_x) || !aligned16(d_y)) return LORA_ERR_INVALID_ARG;
    return run_engine(t, ws, w, false, 1, d_x, ldx, ws->max_M, d_y, ldy, nullptr, stream);
}

extern "C" lora_status lora_build_and_apply(lora_table t, const lora_workspace *ws, const int32_t *d_ids, int32_t M,
                                            const void *d_x, int64_t ldx, void *d_y, int64_t ldy,
                                            lora_stream_t stream)
{
    if (!valid_table(t) || !d_x || !d_y) return LORA_ERR_INVALID_ARG;
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (ws->L != t->L) return LORA_ERR_INVALID_ARG;
    if (t->E_A != 1 || t->E_B != 1) return LORA_ERR_INVALID_ARG;
    if (ldx < t->K || ldy < t->N || ldx % 8 || ldy % 8 || !aligned16(d_x) || !aligned16(d_y)) return LORA_ERR_INVALID_ARG;
    if (M < 0 || (M > 0 && !d_ids)) return LORA_ERR_INVALID_ARG;
    if (M > ws->max_M) return LORA_ERR_WORKSPACE;
    // one launch when every group is sure to run on small tiles (no group can exceed the tensor-core
    // threshold), else the two calls it stands for
    const int64_t path = g_opt_path.load(), thr = g_opt_tc_min_rows.load();
    const bool all_small = path == 1 || (path == 0 && ws->max_M <= 32 && M <= (t->max_R > 128 ? thr / 2 : thr));
    if (M == 0 || M > 32 || !all_small) {
        st = lora_build_segments(ws, d_ids, M, nullptr, nullptr, stream);
        if (st != LORA_OK) return st;
        return lora_apply(t, ws, d_x, ldx, d_y, ldy, stream);
    }
    return run_engine(t, ws, w, false, 1, d_x, ldx, ws->max_M, d_y, ldy, nullptr, stream, d_ids, M);
}

extern "C" lora_status lora_moe_delta(lora_table t, int32_t stage, const lora_workspace *ws, const void *d_in,
                                      int64_t ld_in, void *d_cache, int64_t ld_cache, const float *d_topk_weights,
                                      lora_stream_t stream)
{
    if (!valid_table(t) || !d_in || !d_cache) return LORA_ERR_INVALID_ARG;
    if (stage != LORA_MOE_GATE_UP && stage != LORA_MOE_DOWN) return LORA_ERR_INVALID_ARG;
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (ws->L != t->L || ws->block_m <= 0) return LORA_ERR_INVALID_ARG;
    if ((t->E_A != 1 && t->E_A != ws->num_experts) || (t->E_B != 1 && t->E_B != ws->num_experts))
        return LORA_ERR_INVALID_ARG;
    if (ld_in < t->K || ld_cache < t->N || ld_in % 8 || ld_cache % 8 || !aligned16(d_in) || !aligned16(d_cache))
        return LORA_ERR_INVALID_ARG;
    const int32_t src_div = stage == LORA_MOE_GATE_UP ? ws->topk : 1;
    const int64_t in_rows = stage == LORA_MOE_GATE_UP ? (int64_t)ws->max_M : (int64_t)ws->max_M * ws->topk;
    return run_engine(t, ws, w, true, src_div, d_in, ld_in, in_rows, d_cache, ld_cache, d_topk_weights, stream);
}

extern "C" lora_status lora_linear(lora_table t, const lora_workspace *ws, const void *d_x, int64_t ldx, const void *d_w,
                                   int64_t ldw, void *d_y, int64_t ldy, lora_stream_t stream)
{
    if (!valid_table(t) || !d_x || !d_w || !d_y) return LORA_ERR_INVALID_ARG;
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (ws->L != t->L || t->E_A != 1 || t->E_B != 1) return LORA_ERR_INVALID_ARG;
    if (ldx < t->K || ldw < t->K || ldy < t->N || ldx % 8 || ldw % 8 || ldy % 8 || !aligned16(d_x) ||
        !aligned16(d_w) || !aligned16(d_y))
        return LORA_ERR_INVALID_ARG;
    DeviceInfo di;
    st = device_info(&di);
    if (st != LORA_OK) return st;
    // token tiles: every segment cut into 128-row tiles, then the tokens without an adapter
    const int64_t row_tiles = ceil_div(ws->max_M, kLinearRows) + w.seg_capacity + 1;
    int32_t ctile_off[kMaxSlices] = {0};
    int64_t col_tiles = 0;
    for (int s = 0; s < t->n_slices; ++s) {
        ctile_off[s] = (int32_t)col_tiles;
        col_tiles += ceil_div(t->slice_n[s], kLinearCols);
    }
    if (row_tiles > 65535 || col_tiles < 1 || col_tiles > INT32_MAX) return LORA_ERR_UNSUPPORTED;
    const int stage = linear_stage_bytes(t->max_R);
    const int budget = di.max_dyn_smem - kLinearBTileBytes - 1024;   // the B tile and the stages' alignment
    const int stages = std::min(kLinearMaxStages, budget / stage);
    if (stages < 2) return LORA_ERR_UNSUPPORTED;
    LinearParams p{};
    st = encode_2d(d_w, t->N, t->K, ldw, kLinearCols, &p.w_map);
    if (st == LORA_OK) st = encode_2d(d_x, std::max<int64_t>(ws->max_M, kLinearRows), t->K, ldx, kLinearRows, &p.x_map);
    if (st != LORA_OK) return st;
    p.x = static_cast<const __nv_bfloat16 *>(d_x);
    p.ldx = ldx;
    p.y = static_cast<__nv_bfloat16 *>(d_y);
    p.ldy = ldy;
    p.a_ptr = t->d_a_ptr;
    p.b_ptr = t->d_b_ptr;
    p.rpad = t->d_rpad;
    p.scale = t->d_scale;
    p.L = t->L;
    p.K = t->K;
    p.n_a = t->n_a;
    p.n_slices = t->n_slices;
    p.tiles = (int32_t)col_tiles;
    for (int s = 0; s < kMaxSlices; ++s) {
        p.slice_n[s] = t->slice_n[s];
        p.slice_off[s] = t->slice_off[s];
        p.slice_tile_off[s] = t->slice_tile_off[s];
        p.slice_ctile_off[s] = ctile_off[s];
    }
    int32_t *header = at<int32_t>(ws, w.header);
    p.header = header;
    p.perm = at<int32_t>(ws, w.perm);
    p.segments = at<int4>(ws, w.segments);
    p.stages = stages;
    p.stage_bytes = stage;
    p.err = reinterpret_cast<uint32_t *>(header + H_ERR);
    p.timeout_ns = (uint64_t)g_opt_timeout_ns.load();
    const size_t smem = (size_t)stages * stage + kLinearBTileBytes + 1024;
    return cuda_status(launch_linear(p, dim3((unsigned)col_tiles, (unsigned)row_tiles), smem,
                                     reinterpret_cast<cudaStream_t>(stream), g_opt_pdl.load() != 0));
}

extern "C" lora_status lora_embedding_apply(lora_table t, const lora_workspace *ws, const int32_t *d_vocab, void *d_y,
                                            int64_t ldy, lora_stream_t stream)
{
    if (!valid_table(t) || !d_vocab || !d_y) return LORA_ERR_INVALID_ARG;
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    if (ws->L != t->L || t->E_A != 1 || t->E_B != 1 || t->n_a != 1) return LORA_ERR_INVALID_ARG;
    if (ldy < t->N || ldy % 8 || !aligned16(d_y)) return LORA_ERR_INVALID_ARG;
    const int64_t row_tiles = ceil_div(ws->max_M, kEmbedRows) + w.seg_capacity + 1;
    if (row_tiles > 65535) return LORA_ERR_UNSUPPORTED;
    EmbedParams p{};
    p.a_ptr = t->d_a_ptr;
    p.b_ptr = t->d_b_ptr;
    p.rpad = t->d_rpad;
    p.scale = t->d_scale;
    p.L = t->L;
    p.V = t->K;
    p.n_slices = t->n_slices;
    for (int s = 0; s < kMaxSlices; ++s) {
        p.slice_n[s] = t->slice_n[s];
        p.slice_off[s] = t->slice_off[s];
        p.slice_tile_off[s] = t->slice_tile_off[s];
    }
    int32_t *header = at<int32_t>(ws, w.header);
    p.header = header;
    p.perm = at<int32_t>(ws, w.perm);
    p.segments = at<int4>(ws, w.segments);
    p.vocab = d_vocab;
    p.y = static_cast<__nv_bfloat16 *>(d_y);
    p.ldy = ldy;
    p.err = reinterpret_cast<uint32_t *>(header + H_ERR);
    return cuda_status(launch_embedding(p, dim3((unsigned)t->b_tiles, (unsigned)row_tiles),
                                        reinterpret_cast<cudaStream_t>(stream), g_opt_pdl.load() != 0));
}

extern "C" lora_status lora_get_status(const lora_workspace *ws, lora_stream_t stream)
{
    WsLayout w;
    lora_status st = check_ws(ws, &w);
    if (st != LORA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ERR_CUDA;
    uint32_t word = 0;
    uint32_t *dev = reinterpret_cast<uint32_t *>(at<int32_t>(ws, w.header) + H_ERR);
    if (cudaMemcpy(&word, dev, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ERR_CUDA;
    if (word != 0 && cudaMemset(dev, 0, 4) != cudaSuccess) return LORA_ERR_CUDA;
    if (word & kErrTimeout) return LORA_ERR_TIMEOUT;
    if (word & kErrWorkspace) return LORA_ERR_WORKSPACE;
    if (word & kErrBadId) return LORA_ERR_BAD_ADAPTER_ID;
    if (word & kErrBadExpert) return LORA_ERR_BAD_EXPERT_ID;
    return LORA_OK;
}

extern "C" const char *lora_status_string(lora_status s)
{
    switch (s) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID_ARG: return "invalid argument";
    case LORA_ERR_CUDA: return "CUDA runtime error";
    case LORA_ERR_OOM: return "out of device memory";
    case LORA_ERR_BAD_ADAPTER_ID: return "adapter id out of range";
    case LORA_ERR_BAD_EXPERT_ID: return "expert id out of range";
    case LORA_ERR_TIMEOUT: return "in-kernel wait timed out";
    case LORA_ERR_WORKSPACE: return "workspace too small";
    case LORA_ERR_UNSUPPORTED: return "unsupported shape";
    }
    return "unknown status";
}

extern "C" lora_status lora_set_option(int32_t option, int64_t value)
{
    switch (option) {
    case LORA_OPT_PATH:
        if (value < 0 || value > 3) return LORA_ERR_INVALID_ARG;
        g_opt_path = value;
        return LORA_OK;
    case LORA_OPT_TC_MIN_ROWS:
        if (value < 0) return LORA_ERR_INVALID_ARG;
        g_opt_tc_min_rows = value;
        return LORA_OK;
    case LORA_OPT_WAIT_TIMEOUT_NS:
        if (value < 1000) return LORA_ERR_INVALID_ARG;
        g_opt_timeout_ns = value;
        return LORA_OK;
    case LORA_OPT_GRID_CTAS:
        if (value < 0) return LORA_ERR_INVALID_ARG;
        g_opt_grid = value;
        return LORA_OK;
    case LORA_OPT_TEST_WITHHOLD_HANDOFF:
        g_opt_withhold = value != 0;
        return LORA_OK;
    case LORA_OPT_PDL:
        if (value < 0 || value > 1) return LORA_ERR_INVALID_ARG;
        g_opt_pdl = value;
        return LORA_OK;
    }
    return LORA_ERR_INVALID_ARG;
}

extern "C" lora_status lora_set_trace(void *d_trace, size_t bytes)
{
    if (d_trace && (bytes < 8 * kTraceSlots || (reinterpret_cast<uintptr_t>(d_trace) & 7u))) return LORA_ERR_INVALID_ARG;
    g_trace_bytes = d_trace ? (int64_t)bytes : 0;
    g_trace = d_trace;
    return LORA_OK;
}

extern "C" int64_t lora_get_option(int32_t option)
{
    switch (option) {
    case LORA_OPT_PATH: return g_opt_path.load();
    case LORA_OPT_TC_MIN_ROWS: return g_opt_tc_min_rows.load();
    case LORA_OPT_WAIT_TIMEOUT_NS: return g_opt_timeout_ns.load();
    case LORA_OPT_GRID_CTAS: return g_opt_grid.load();
    case LORA_OPT_TEST_WITHHOLD_HANDOFF: return g_opt_withhold.load();
    case LORA_OPT_PDL: return g_opt_pdl.load();
    }
    return -1;
}

// ---------------------------------------------------------------------------
// lora_apply_static_scratch: the whole step (segment table + fused apply) with
// every byte of scratch in one fixed device array, for callers that cannot
// allocate device memory.
// ---------------------------------------------------------------------------
namespace {

constexpr int32_t kStaticMaxM = 4096;                        // tokens per call
constexpr int32_t kStaticMaxTiles = kStaticMaxM / kBgmvRows + kStaticMaxM;
constexpr int64_t kStaticPartialFloats = 8 * 1024 * 1024;   // 32 MiB of hand-off partials
constexpr size_t kStaticHeader = 0;
constexpr size_t kStaticPerm = 256;
constexpr size_t kStaticSegments = kStaticPerm + (size_t)kStaticMaxM * 4;
constexpr size_t kStaticSync = kStaticSegments + (size_t)kStaticMaxM * 16;
constexpr size_t kStaticPartials = kStaticSync + (size_t)kStaticMaxTiles * 16;
constexpr size_t kStaticBytes = kStaticPartials + (size_t)kStaticPartialFloats * 4;

// Shared by every call on a device and kept until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

std::mutex g_static_mu;
std::map<int, unsigned char *> g_static_addr;   // device -> address of g_static_scratch

// Device address of g_static_scratch on the current device (looked up once per device).
lora_status static_scratch_address(unsigned char **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    auto it = g_static_addr.find(dev);
    if (it == g_static_addr.end()) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return LORA_ERR_CUDA;
        }
        it = g_static_addr.emplace(dev, static_cast<unsigned char *>(ptr)).first;
    }
    *out = it->second;
    return LORA_OK;
}

}  // namespace

extern "C" lora_status lora_apply_static_scratch(lora_table t, const int32_t *d_ids, int32_t M, const void *d_x,
                                                 int64_t ldx, void *d_y, int64_t ldy, lora_stream_t stream)
{
    if (!valid_table(t) || M < 0 || (M > 0 && (!d_ids || !d_x || !d_y))) return LORA_ERR_INVALID_ARG;
    if (t->E_A != 1 || t->E_B != 1) return LORA_ERR_INVALID_ARG;
    if (t->L + 1 > kMaxBuildKeys) return LORA_ERR_UNSUPPORTED;   // the segment build's key limit
    if (M > 0 && (ldx < t->K || ldy < t->N || ldx % 8 || ldy % 8 || !aligned16(d_x) || !aligned16(d_y)))
        return LORA_ERR_INVALID_ARG;
    if (M > kStaticMaxM) return LORA_ERR_WORKSPACE;
    // the hand-off scratch of M rows at this table's largest A block must fit the fixed array at the
    // shortest K-chunk the engine can cut (this entry point has no status word to report a shortfall),
    // plus the S padding of up to one 64-row tile per group
    {
        const int64_t R = t->max_R;
        const int64_t need = (int64_t)M * engine_partials_per_row(R, t->K, kEngineMinKc) +
                             R * 64 * std::min<int64_t>(M, t->L);
        if (need > kStaticPartialFloats) return LORA_ERR_WORKSPACE;
    }
    unsigned char *base = nullptr;
    lora_status st = static_scratch_address(&base);
    if (st != LORA_OK) return st;
    DeviceInfo di;
    st = device_info(&di);
    if (st != LORA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t *header = reinterpret_cast<int32_t *>(base + kStaticHeader);
    // this call's device-side status starts clean (the array keeps the last call's contents)
    if (cudaMemsetAsync(header + H_ERR, 0, 4, s) != cudaSuccess) return LORA_ERR_CUDA;

    BuildParams b{};
    b.ids = d_ids;
    b.M = M;
    b.L = t->L;
    b.header = header;
    b.perm = reinterpret_cast<int32_t *>(base + kStaticPerm);
    b.segments = reinterpret_cast<int4 *>(base + kStaticSegments);
    b.seg_capacity = kStaticMaxM;
    b.sync = reinterpret_cast<int32_t *>(base + kStaticSync);   // zeroed by the build kernel
    b.sync_ints = kStaticMaxTiles * 4;
    if (launch_build(b, s, g_opt_pdl.load() != 0) != cudaSuccess) return LORA_ERR_CUDA;

    EngineParams p{};
    if (M > 0 && t->K >= 64) {
        st = encode_rows_map(d_x, M, t->K, ldx, &p.x_map);
        if (st != LORA_OK) return st;
        p.x_rows = M;
    }
    p.m_ptr = header + H_M;
    p.m_mult = 1;
    p.y_mult = 1;
    if (M > 0 && t->N >= 128) {   // output tiles move as 2-D boxes only inside rows the build produced
        st = encode_2d(d_y, std::max<int32_t>(M, 128), t->N, ldy, 128, &p.y_map_ld);
        if (st == LORA_OK) st = encode_2d(d_y, std::max<int32_t>(M, 128), t->N, ldy, 32, &p.y_map_st);
        if (st != LORA_OK) return st;
        p.y_rows = M;
    }
    p.a_ptr = t->d_a_ptr;
    p.b_ptr = t->d_b_ptr;
    p.rpad = t->d_rpad;
    p.scale = t->d_scale;
    p.L = t->L;
    p.E_A = 1;
    p.E_B = 1;
    p.K = t->K;
    p.n_slices = t->n_slices;
    p.n_a = t->n_a;
    for (int i = 0; i < kMaxSlices; ++i) {
        p.slice_n[i] = t->slice_n[i];
        p.slice_off[i] = t->slice_off[i];
        p.slice_tile_off[i] = t->slice_tile_off[i];
    }
    p.groups = b.segments;
    p.num_groups = header + H_NUM_SEGMENTS;
    p.group_capacity = kStaticMaxM;
    p.num_experts = 1;
    p.rows_capacity = kStaticMaxM;
    p.rows = b.perm;
    p.src_div = 1;
    p.x = static_cast<const __nv_bfloat16 *>(d_x);
    p.ldx = ldx;
    p.y = static_cast<__nv_bfloat16 *>(d_y);
    p.ldy = ldy;
    p.row_weight = nullptr;
    p.sync = b.sync;
    p.partials = reinterpret_cast<float *>(base + kStaticPartials);
    p.partial_floats = kStaticPartialFloats;
    p.max_tiles = kStaticMaxTiles;
    p.err = reinterpret_cast<uint32_t *>(header + H_ERR);
    p.timeout_ns = (uint64_t)g_opt_timeout_ns.load();
    p.withhold = 0;
    p.path = (int32_t)g_opt_path.load();
    p.tc_min_rows = (int32_t)g_opt_tc_min_rows.load();
    p.trace = nullptr;
    p.trace_ctas = 0;
    int grid = di.sms * di.engine_blocks_per_sm;
    const int64_t want = g_opt_grid.load();
    if (want > 0 && want < grid) grid = (int)want;
    cudaError_t e;
    launch_engine(p, grid, engine_smem_bytes(0), s, g_opt_pdl.load() != 0 && M <= 32, &e);
    return cuda_status(e);
}
