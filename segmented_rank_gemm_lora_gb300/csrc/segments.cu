// Device-side segment table and MoE alignment.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 2.3: tokens are bucketed
// by lora_id so equal ids become contiguous, giving one segment per adapter
// (id, token range, rank); section 2.4: the per-core work is fixed before the
// compute starts.  "[SGLang] LoRA + MoE fusion", MoE LoRA Alignment: token /
// expert pairs sorted by (adapter, expert), each group padded to block_size_m.
//
// Both are one stable counting sort, run by a single 1024-thread CTA:
//   1. W warps each own a contiguous run of items and count keys into their
//      own shared-memory histogram row;
//   2. per key, an exclusive prefix over the warp rows (in warp order) and the
//      key totals;
//   3. the caller places every key's first slot (compact, or padded for MoE);
//   4. each warp walks its run in order 32 items at a time; match.any gives
//      each lane its rank among equal keys of the step, and the warp's running
//      per-key counters give the rest, so every key keeps the items' order.
#include "common.cuh"

namespace lora {

constexpr int kBuildThreads = 1024;
constexpr int kBuildSmemBytes = 200 * 1024;

// In-place exclusive scan of a[0..n) by the whole block; returns the total.
__device__ int32_t block_exclusive_scan(int32_t *a, int32_t n, int32_t *warp_tmp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kBuildThreads - 1) / kBuildThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    // inclusive warp scan of the per-thread sums
    int32_t v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_tmp[lane];
        int32_t x = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t u = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += u;
        }
        warp_tmp[lane] = x - w;       // exclusive prefix of warp sums
        if (lane == 31) warp_tmp[32] = x;
    }
    __syncthreads();
    int32_t run = warp_tmp[warp] + v - local;
    for (int i = lo; i < hi; ++i) {
        int32_t c = a[i];
        a[i] = run;
        run += c;
    }
    const int32_t total = warp_tmp[32];
    __syncthreads();
    return total;
}

struct SortSmem {
    int32_t *hist;   // [W][nkeys]
    int32_t *tot;    // [nkeys]
    int32_t *base;   // [nkeys]
    int32_t W, nkeys;
};

__device__ __forceinline__ SortSmem carve(int32_t *smem, int32_t nkeys)
{
    SortSmem s;
    const int32_t budget = kBuildSmemBytes / 4 - 64;
    int32_t W = (budget - 2 * nkeys) / nkeys;
    W = W > 32 ? 32 : (W < 1 ? 1 : W);
    s.W = W;
    s.nkeys = nkeys;
    s.tot = smem + 64;
    s.base = s.tot + nkeys;
    s.hist = s.base + nkeys;
    return s;
}

// Phases 1-2: per-warp histograms and per-key totals.
template <class KeyFn>
__device__ void sort_count(const SortSmem &s, int32_t n, KeyFn key)
{
    for (int i = threadIdx.x; i < s.W * s.nkeys; i += kBuildThreads) s.hist[i] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t chunk = (n + s.W - 1) / s.W;
    if (warp < s.W) {
        const int32_t lo = warp * chunk, hi = min(n, lo + chunk);
        for (int32_t i = lo + lane; i < hi; i += 32) atomicAdd(&s.hist[warp * s.nkeys + key(i)], 1);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < s.nkeys; k += kBuildThreads) {
        int32_t run = 0;
        for (int w = 0; w < s.W; ++w) {
            const int32_t c = s.hist[w * s.nkeys + k];
            s.hist[w * s.nkeys + k] = run;
            run += c;
        }
        s.tot[k] = run;
    }
    __syncthreads();
}

// Phase 4: stable placement; place(i, key, base[key] + rank within key).
template <class KeyFn, class PlaceFn>
__device__ void sort_place(const SortSmem &s, int32_t n, KeyFn key, PlaceFn place)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t chunk = (n + s.W - 1) / s.W;
    if (warp < s.W) {
        const int32_t lo = warp * chunk, hi = min(n, lo + chunk);
        int32_t *row = s.hist + warp * s.nkeys;
        for (int32_t i0 = lo; i0 < hi; i0 += 32) {
            const int32_t i = i0 + lane;
            const bool live = i < hi;
            const int32_t k = live ? key(i) : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, k);
            const uint32_t lt = (1u << lane) - 1u;
            int32_t slot = 0;
            if (live) slot = row[k] + __popc(peers & lt);
            __syncwarp();
            if (live && (peers & lt) == 0) row[k] += __popc(peers);
            __syncwarp();
            if (live) place(i, k, s.base[k] + slot);
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kBuildThreads, 1) build_kernel(BuildParams p)
{
    extern __shared__ __align__(16) int32_t smem[];
    int32_t *tmp = smem;   // 33 ints of scan scratch
    uint32_t *err = reinterpret_cast<uint32_t *>(p.header + H_ERR);
    const int32_t L = p.L, M = p.M;
    pdl_trigger();
    pdl_wait();   // the previous launch on the stream may still read this workspace

    for (int i = threadIdx.x; i < p.sync_ints; i += kBuildThreads) p.sync[i] = 0;

    // ---------------- dense: key = adapter id, L = dropped ----------------
    auto dkey = [&](int32_t t) -> int32_t {
        const int32_t i = p.ids[t];
        if (i >= 0 && i < L) return (p.enabled == nullptr || p.enabled[i]) ? i : L;
        return L;
    };
    for (int t = threadIdx.x; t < M; t += kBuildThreads) {
        const int32_t i = p.ids[t];
        if (i < -1 || i >= L) atomicOr(err, kErrBadId);
    }
    {
        SortSmem s = carve(smem, L + 1);
        sort_count(s, M, dkey);
        for (int k = threadIdx.x; k <= L; k += kBuildThreads) s.base[k] = s.tot[k];
        __syncthreads();
        const int32_t total = block_exclusive_scan(s.base, L + 1, tmp);
        (void)total;
        sort_place(s, M, dkey, [&](int32_t t, int32_t, int32_t pos) { p.perm[pos] = t; });
        // compact the non-empty adapter buckets into the segment list
        int32_t *flag = s.hist;   // reuse
        for (int k = threadIdx.x; k < L; k += kBuildThreads) flag[k] = s.tot[k] > 0 ? 1 : 0;
        __syncthreads();
        const int32_t nseg = block_exclusive_scan(flag, L, tmp);
        for (int k = threadIdx.x; k < L; k += kBuildThreads)
            if (s.tot[k] > 0) p.segments[flag[k]] = make_int4(k, 0, s.base[k], s.tot[k]);
        if (threadIdx.x == 0) {
            p.header[H_M] = M;
            p.header[H_NUM_SEGMENTS] = nseg;
            p.header[H_NUM_VALID] = s.base[L];
        }
        __syncthreads();
    }

    // ---------------- MoE: key = adapter * E + expert ----------------
    if (p.block_m > 0 && p.topk_ids != nullptr) {
        const int32_t E = p.E, topk = p.topk, bm = p.block_m;
        const int32_t P = M * topk;
        const int32_t P_max = (int32_t)(((int64_t)P + (int64_t)E * (bm - 1) + bm - 1) / bm * bm);
        const int32_t B_max = P_max / bm;
        const int32_t dropped = L * E;
        auto mkey = [&](int32_t q) -> int32_t {
            const int32_t i = p.ids[q / topk];
            const int32_t e = p.topk_ids[q];
            if (i < 0 || i >= L) return dropped;
            if (p.enabled != nullptr && !p.enabled[i]) return dropped;
            if (e < 0 || e >= E) return dropped;
            return i * E + e;
        };
        for (int q = threadIdx.x; q < P; q += kBuildThreads) {
            const int32_t i = p.ids[q / topk];
            const int32_t e = p.topk_ids[q];
            if (i >= 0 && i < L && (e < 0 || e >= E)) atomicOr(err, kErrBadExpert);
        }
        SortSmem s = carve(smem, dropped + 1);
        sort_count(s, P, mkey);
        // padded start of every (adapter, expert) group inside the adapter's row
        for (int l = threadIdx.x; l < L; l += kBuildThreads) {
            int32_t pos = 0;
            for (int e = 0; e < E; ++e) {
                const int32_t k = l * E + e;
                s.base[k] = l * P_max + pos;
                pos += (s.tot[k] + bm - 1) / bm * bm;
            }
            p.ntpp[l] = pos;
        }
        s.base[dropped] = 0;
        for (int64_t q = threadIdx.x; q < (int64_t)L * P_max; q += kBuildThreads) p.sorted_ids[q] = P;
        for (int64_t q = threadIdx.x; q < (int64_t)L * B_max; q += kBuildThreads) p.expert_ids[q] = -1;
        __syncthreads();
        sort_place(s, P, mkey, [&](int32_t q, int32_t k, int32_t pos) {
            if (k != dropped) p.sorted_ids[pos] = q;
        });
        for (int k = threadIdx.x; k < dropped; k += kBuildThreads) {
            const int32_t c = s.tot[k];
            if (c > 0) {
                const int32_t l = k / E, e = k % E;
                const int32_t start = s.base[k] - l * P_max;
                const int32_t padded = (c + bm - 1) / bm * bm;
                for (int32_t b = start / bm; b < (start + padded) / bm; ++b) p.expert_ids[l * B_max + b] = e;
            }
        }
        int32_t *flag = s.hist;
        for (int k = threadIdx.x; k < dropped; k += kBuildThreads) flag[k] = s.tot[k] > 0 ? 1 : 0;
        __syncthreads();
        const int32_t ng = block_exclusive_scan(flag, dropped, tmp);
        for (int k = threadIdx.x; k < dropped; k += kBuildThreads)
            if (s.tot[k] > 0) p.moe_groups[flag[k]] = make_int4(k / E, k % E, s.base[k], s.tot[k]);
        if (threadIdx.x == 0) {
            p.header[H_NUM_MOE_GROUPS] = ng;
            p.header[H_TOPK] = topk;
            p.header[H_E] = E;
            p.header[H_BLOCK_M] = bm;
            p.header[H_P_MAX] = P_max;
            p.header[H_B_MAX] = B_max;
        }
    } else if (threadIdx.x == 0) {
        p.header[H_NUM_MOE_GROUPS] = 0;
        p.header[H_BLOCK_M] = 0;
    }
}

// Dense batches of at most 32 tokens: one warp, one token per lane, placed by
// warp_rank_ids (the slots of the stable counting sort above, from one ballot
// per key bit).  The first lane of each adapter writes its segment.
__global__ void __launch_bounds__(32, 1) build_warp_kernel(BuildParams p)
{
    const int lane = threadIdx.x;
    const int32_t L = p.L, M = p.M;
    uint32_t *err = reinterpret_cast<uint32_t *>(p.header + H_ERR);
    pdl_trigger();
    pdl_wait();   // the previous launch on the stream may still read this workspace
    for (int i = lane; i < p.sync_ints; i += 32) p.sync[i] = 0;
    const WarpRank r = warp_rank_ids(p.ids, p.enabled, M, L);
    if (r.bad) atomicOr(err, kErrBadId);
    if (lane < M) p.perm[r.rank] = lane;
    const bool start = r.first && r.key < L;
    if (start) p.segments[r.seg] = make_int4(r.key, 0, r.rank, r.count);
    const int num_segments = __popc(__ballot_sync(0xffffffffu, start));
    const int num_valid = __popc(__ballot_sync(0xffffffffu, lane < M && r.key < L));
    if (lane == 0) {
        p.header[H_M] = M;
        p.header[H_NUM_SEGMENTS] = num_segments;
        p.header[H_NUM_VALID] = num_valid;
        p.header[H_NUM_MOE_GROUPS] = 0;
        p.header[H_BLOCK_M] = 0;
    }
}

cudaError_t launch_build(const BuildParams &p, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (p.M <= 32 && (p.block_m <= 0 || p.topk_ids == nullptr)) {
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(32);
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, build_warp_kernel, p);
    }
    // (the block-wide build starts in plain stream order: scheduled early, it was measured to slow the
    // step down)
    cfg.numAttrs = 0;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kBuildSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kBuildThreads);
    cfg.dynamicSmemBytes = kBuildSmemBytes;
    return cudaLaunchKernelEx(&cfg, build_kernel, p);
}

}  // namespace lora
