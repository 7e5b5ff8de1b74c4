// Load-time packing of one adapter's A and B into the table layout.
//
// "vLLM-Ascend dynamic LoRA fused operator", section 2.1: adapters of equal
// rank live in one contiguous run, laid out once when the adapter is loaded;
// section 2.2: keep A in the orientation the shrink reads and pre-lay B for the
// expand so no step transposes on the device; section 4.3: the rank dimension
// is zero-padded to a multiple of 16.
//
// Packed A (one (adapter, expert) block): [K/8][n_a * rpad][8] bf16.  Element
// A[s*r + j][k] sits at ((k/8) * n_a*rpad + s*rpad + j) * 8 + k%8.  A K-range
// that starts on a multiple of 8 is one contiguous run, and eight consecutive
// k of one row are one 16-byte vector.  The same bytes are a K-major operand
// in the no-swizzle canonical tcgen05 layout (core matrix = 8 rows x 16 bytes;
// rows 16 bytes apart, K core matrices n_a*rpad*16 bytes apart).
//
// Packed B (one block): for each slice s, ceil(N_s/128) tiles of
// [rpad/8][128][8]: element B[off_s + n][j] sits in tile n/128 of the slice at
// ((j/8) * 128 + n%128) * 8 + j%8.  Rows past N_s and columns past r are zero.
// Each tile is contiguous (a run of consecutive tiles is one bulk copy), the
// 16-byte vector of one row holds eight consecutive j, and a tile is a K-major
// canonical operand of the expand MMA (N = 128).
#include "common.cuh"

namespace lora {

__global__ void pack_a_kernel(const __nv_bfloat16 *__restrict__ src, __nv_bfloat16 *__restrict__ dst, int32_t K,
                              int32_t n_a, int32_t rank, int32_t rpad)
{
    const int32_t R = n_a * rpad;
    const int64_t total = (int64_t)(K / 8) * R;
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        const int32_t kg = (int32_t)(v / R);
        const int32_t row = (int32_t)(v % R);
        const int32_t s = row / rpad, j = row % rpad;
        __align__(16) __nv_bfloat16 out[8];
        if (j < rank) {
            const __nv_bfloat16 *p = src + (int64_t)(s * rank + j) * K + (int64_t)kg * 8;
#pragma unroll
            for (int u = 0; u < 8; ++u) out[u] = p[u];
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) out[u] = __float2bfloat16(0.0f);
        }
        reinterpret_cast<uint4 *>(dst)[v] = *reinterpret_cast<const uint4 *>(out);
    }
}

struct SliceInfo {
    int32_t n_slices;
    int32_t slice_n[kMaxSlices];
    int32_t col_off[kMaxSlices];
    int32_t tile_off[kMaxSlices + 1];
};

__global__ void pack_b_kernel(const __nv_bfloat16 *__restrict__ src, __nv_bfloat16 *__restrict__ dst,
                              int32_t rank, int32_t rpad, SliceInfo si)
{
    const int32_t kgroups = rpad / 8;
    const int64_t per_tile = (int64_t)kgroups * kNTile;
    const int64_t total = (int64_t)si.tile_off[si.n_slices] * per_tile;
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        const int32_t tile = (int32_t)(v / per_tile);
        const int32_t rem = (int32_t)(v % per_tile);
        const int32_t kg = rem / kNTile, row = rem % kNTile;
        int32_t s = 0;
        while (s + 1 < si.n_slices && tile >= si.tile_off[s + 1]) ++s;
        const int32_t n_local = (tile - si.tile_off[s]) * kNTile + row;
        __align__(16) __nv_bfloat16 out[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t j = kg * 8 + u;
            out[u] = (n_local < si.slice_n[s] && j < rank)
                         ? src[(int64_t)(si.col_off[s] + n_local) * rank + j]
                         : __float2bfloat16(0.0f);
        }
        reinterpret_cast<uint4 *>(dst)[v] = *reinterpret_cast<const uint4 *>(out);
    }
}

cudaError_t launch_pack_a(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int32_t K, int32_t n_a, int32_t rank,
                          int32_t rpad, cudaStream_t s)
{
    const int64_t total = (int64_t)(K / 8) * n_a * rpad;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    pack_a_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(src, dst, K, n_a, rank, rpad);
    return cudaGetLastError();
}

cudaError_t launch_pack_b(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int32_t rank, int32_t rpad,
                          int32_t n_slices, const int32_t *slice_n, cudaStream_t s)
{
    SliceInfo si{};
    si.n_slices = n_slices;
    int32_t col = 0, tiles = 0;
    for (int i = 0; i < n_slices; ++i) {
        si.slice_n[i] = slice_n[i];
        si.col_off[i] = col;
        si.tile_off[i] = tiles;
        col += slice_n[i];
        tiles += (int32_t)ceil_div(slice_n[i], kNTile);
    }
    si.tile_off[n_slices] = tiles;
    const int64_t total = (int64_t)tiles * (rpad / 8) * kNTile;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    pack_b_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(src, dst, rank, rpad, si);
    return cudaGetLastError();
}

}  // namespace lora
