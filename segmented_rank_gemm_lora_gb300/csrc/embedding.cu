// Embedding LoRA: y[t] += scale_i * B_i * A_i[:, vocab[t]].
//
// "[SGLang] LoRA Layers", VocabParallelEmbeddingWithLoRA: in the embedding
// layer the LoRA A matrix (rank x vocabulary) acts as an embedding lookup and
// B (embedding width x rank) as a plain matmul added to the base embedding.
// The tokens come grouped by adapter from the segment table of the last build
// ("vLLM-Ascend dynamic LoRA fused operator", section 2.3).
//
// One CTA per (up to 32 tokens of one segment, 128 output columns = one packed
// B tile).  The shrink is a gather: token t's S row is column vocab[t] of the
// packed A block ([V/8][rp][8]: the rp values sit 16 bytes apart in one
// contiguous run of rp * 16 bytes).  The B tile ([rp/8][128][8]) is staged in
// shared memory; thread (column c, token parity) accumulates S[t] . B[c] in
// fp32 on CUDA cores (rank <= 64, a few thousand multiply-adds per thread) and
// adds scale * acc to the bf16 base row, rounding once.
#include "embedding.h"

namespace lora {

namespace {

constexpr int kT = kEmbedThreads;
constexpr int kRows = kEmbedRows;

struct EmbSmem {
    float S[kRows][kMaxRank + 1];
    __align__(16) __nv_bfloat16 Bt[kMaxRank / 8][128][8];
    int32_t row[kRows];
    int32_t adapter, slot0, rows, rp;
    uint64_t b_blk, a_blk;
    float sc;
};

__global__ void __launch_bounds__(kT) embedding_kernel(const __grid_constant__ EmbedParams p)
{
    __shared__ EmbSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = blockIdx.x;    // B tile (128 output columns)
    const int rt = blockIdx.y;   // token tile
    pdl_wait();
    pdl_trigger();

    // ---- the token tile: tile rt of the segments, each cut into tiles of kRows tokens ----
    if (warp == 0) {
        const int nG = p.header[H_NUM_SEGMENTS];
        int base = 0;
        bool found = false;
        if (lane == 0) sm.rows = 0;
        for (int c = 0; c < nG && !found; c += 32) {
            const int g = c + lane;
            const int4 seg = g < nG ? p.segments[g] : make_int4(0, 0, 0, 0);
            const int tl = (seg.w + kRows - 1) / kRows;
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
                    sm.slot0 = seg.z + (rt - first) * kRows;
                    sm.rows = min(kRows, seg.w - (rt - first) * kRows);
                }
                found = true;
            }
            base += total;
        }
    }
    __syncthreads();
    const int rows = sm.rows;
    if (rows <= 0) return;
    if (tid == 0) {
        const int a = sm.adapter;
        const bool ok = a >= 0 && a < p.L;
        sm.rp = ok ? p.rpad[a] : 0;
        sm.a_blk = ok ? p.a_ptr[a] : 0;
        sm.b_blk = ok ? p.b_ptr[a] : 0;
        sm.sc = ok ? p.scale[a] : 0.f;
    }
    if (tid < rows) {
        const int r = p.perm[sm.slot0 + tid];
        const int v = p.vocab[r];
        const bool ok = v >= 0 && v < p.V;
        if (!ok && j == 0) atomicOr(p.err, kErrBadId);
        sm.row[tid] = ok ? r : -1;
    }
    __syncthreads();
    const int rp = sm.rp;
    if (rp <= 0) return;

    // ---- the lookup: S[t][k] = A[k][vocab[row t]] (k < rp), and the B tile into shared memory ----
    const __nv_bfloat16 *ablk = reinterpret_cast<const __nv_bfloat16 *>(sm.a_blk);
    for (int i = tid; i < rows * rp; i += kT) {
        const int t = i / rp, k = i - t * rp;
        const int r = sm.row[t];
        float v = 0.f;
        if (r >= 0) {
            const int voc = p.vocab[r];
            v = __bfloat162float(ablk[((int64_t)(voc >> 3) * rp + k) * 8 + (voc & 7)]);
        }
        sm.S[t][k] = v;
    }
    const uint4 *bsrc = reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(sm.b_blk) +
                                                        (int64_t)j * rp * 256);
    uint4 *bdst = reinterpret_cast<uint4 *>(&sm.Bt[0][0][0]);
    for (int i = tid; i < rp * 16; i += kT) bdst[i] = bsrc[i];
    __syncthreads();

    // ---- y rows of the tile += scale * S B_tile^T: thread (column c, token parity h) ----
    int s = 0;
    while (s + 1 < p.n_slices && j >= p.slice_tile_off[s + 1]) ++s;
    const int lt = j - p.slice_tile_off[s];
    const int col0 = p.slice_off[s] + lt * 128, width = min(128, p.slice_n[s] - lt * 128);
    const int c = tid & 127, h = tid >> 7;
    if (c >= width) return;
    float bcol[kMaxRank];
#pragma unroll
    for (int kg = 0; kg < kMaxRank / 8; ++kg) {
        if (kg * 8 >= rp) break;
        const uint4 q = *reinterpret_cast<const uint4 *>(&sm.Bt[kg][c][0]);
        bf16x8_to_f32(q, &bcol[kg * 8]);
    }
    const float sc = sm.sc;
    for (int t = h; t < rows; t += 2) {
        const int r = sm.row[t];
        if (r < 0) continue;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxRank; ++k) {
            if (k >= rp) break;
            acc += sm.S[t][k] * bcol[k];
        }
        __nv_bfloat16 *yp = p.y + (int64_t)r * p.ldy + col0 + c;
        *yp = __float2bfloat16_rn(__bfloat162float(*yp) + sc * acc);
    }
}

}  // namespace

cudaError_t launch_embedding(const EmbedParams &p, dim3 grid, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, embedding_kernel, p);
}

}  // namespace lora
